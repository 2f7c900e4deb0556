// Step 3, variant S: the N residue products on the INT8 tensor path that
// sm_103a offers outside tcgen05 (it has no tcgen05 kind::i8).
//
// [Q] "誤差のないINT8行列積(手順3)": per modulus, one exact integer product of
// the residue matrices; with |r| <= 128 every product is at most 2^14 and an
// int32 sum stays exact below 2^17 terms.  Here that product runs as
// mma.sync.m16n8k32 s8 x s8 -> s32 on int8 residue planes (step 2 writes the
// planes as int8 for this variant): A planes [N][m][kp], B planes
// [N][b_plane_rows][kp], every row K-contiguous, so the rows of B's planes are
// the columns of the product.
//
// CTA tile 128 x 128, eight warps as 2 x 4, warp tile 64 x 32 (4 x 4 MMAs of
// 16 x 8 per 32-byte k step).  A 3-stage cp.async ring holds 128-byte k slices
// of the CTA's 128 rows of A and of B (16 KB each); each row's eight 16-byte
// chunks are stored XOR-swizzled by the row index, so the ldmatrix reads of
// eight rows hit eight different bank groups.  Rows past m or n and bytes
// past kp are zero-filled by the copies.
//
// Mod-p output: the accumulators are reduced mod p_l every 65536 terms (a sum
// of 65536 products plus a carried residue below 256 stays below 2^31), and
// the final value becomes the symmetric residue c_l as int8.  Raw output: the
// int32 product itself (the caller keeps k below 2^17).
#include "os2_internal.cuh"

namespace {

constexpr int BM = 128, BN = 128;
constexpr int BKB = 128;                      // k bytes (terms) per stage
constexpr int kStages = 3, kThreads = 256;
constexpr int kStageBytes = (BM + BN) * BKB;  // 32 KB
constexpr int kSmem = kStages * kStageBytes;  // 96 KB
constexpr int kSegStages = 65536 / BKB;       // stages between two reductions mod p

// Byte offset of 16-byte chunk `c` of row `row` in a 128-byte-row tile.
__device__ __forceinline__ uint32_t swz(int row, int c) {
  return (uint32_t)(row * BKB + ((c ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp16(uint32_t dst, const void *src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int PENDING>
__device__ __forceinline__ void cp_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(PENDING) : "memory");
}

__device__ __forceinline__ void ldsm4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D += A (16 x 32, row-major) B (32 x 8, column-major), s8 x s8 -> s32.
// Fragments (g = lane / 4, t = lane % 4): a0 = A[g][4t..4t+3], a1 = A[g+8][..],
// a2 = A[g][16+4t..], a3 = A[g+8][16+4t..]; b0 = B[4t..4t+3][g],
// b1 = B[16+4t..][g]; d0, d1 = D[g][2t, 2t+1], d2, d3 = D[g+8][2t, 2t+1].
__device__ __forceinline__ void mma_s8(int (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                       uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(d[0]), "+r"(d[1]), "+r"(d[2]), "+r"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int OUT>
__global__ void __launch_bounds__(kThreads, 2)
    k_gemm_s8(int m, int n, int kp, const int8_t *__restrict__ RA, const int8_t *__restrict__ RB,
              int b_plane_rows, void *__restrict__ out, int ldo, const GemmConsts gc,
              int *status) {
  extern __shared__ __align__(128) uint8_t smem[];
  const int l = blockIdx.z;
  const int tm = blockIdx.y * BM, tn = blockIdx.x * BN;
  const int8_t *A = RA + (size_t)l * m * kp;
  const int8_t *B = RB + (size_t)l * b_plane_rows * kp;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wm = warp >> 2, wn = warp & 3;  // warp tile rows wm*64.., columns wn*32..
  const uint32_t sbase = (uint32_t)__cvta_generic_to_shared(smem);
  const int nk = (kp + BKB - 1) / BKB;

  // copies of k slice kb into ring slot `slot`: 1024 chunks of A, then 1024 of B
  auto load = [&](int kb, int slot) {
    const uint32_t sa = sbase + slot * kStageBytes, sb = sa + BM * BKB;
#pragma unroll
    for (int u = 0; u < 4; u++) {
      const int q = threadIdx.x + u * kThreads;
      const int row = q >> 3, c = q & 7;
      const int kbyte = kb * BKB + c * 16;
      const bool kin = kbyte < kp;
      const bool va = kin && tm + row < m, vb = kin && tn + row < n;
      cp16(sa + swz(row, c), va ? A + (size_t)(tm + row) * kp + kbyte : A, va);
      cp16(sb + swz(row, c), vb ? B + (size_t)(tn + row) * kp + kbyte : B, vb);
    }
  };

  int acc[4][4][4];
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int j = 0; j < 4; j++)
#pragma unroll
      for (int v = 0; v < 4; v++) acc[i][j][v] = 0;

#pragma unroll
  for (int s = 0; s < kStages - 1; s++) {
    if (s < nk) load(s, s);
    cp_commit();
  }
  const int p = (int)gc.p[l];

#pragma unroll 1
  for (int kb = 0; kb < nk; kb++) {
    cp_wait<kStages - 2>();  // slice kb has landed (this thread's copies)
    __syncthreads();         // everyone's copies of it, and everyone is done with slot kb - 1
    if (kb + kStages - 1 < nk) load(kb + kStages - 1, (kb + kStages - 1) % kStages);
    cp_commit();
    const uint32_t sa = sbase + (kb % kStages) * kStageBytes, sb = sa + BM * BKB;
#pragma unroll
    for (int ks = 0; ks < BKB / 32; ks++) {
      uint32_t a[4][4], b[4][2];
#pragma unroll
      for (int i = 0; i < 4; i++) {
        const int row = wm * 64 + i * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
        ldsm4(sa + swz(row, ks * 2 + (lane >> 4)), a[i]);
      }
#pragma unroll
      for (int jp = 0; jp < 2; jp++) {
        const int row = wn * 32 + jp * 16 + (lane & 7) + (lane >> 4) * 8;
        uint32_t r[4];
        ldsm4(sb + swz(row, ks * 2 + ((lane >> 3) & 1)), r);
        b[2 * jp][0] = r[0];
        b[2 * jp][1] = r[1];
        b[2 * jp + 1][0] = r[2];
        b[2 * jp + 1][1] = r[3];
      }
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++) mma_s8(acc[i][j], a[i], b[j][0], b[j][1]);
    }
    if (OUT == OS2_OUT_MODP_INT8 && (kb + 1) % kSegStages == 0) {
#pragma unroll
      for (int i = 0; i < 4; i++)
#pragma unroll
        for (int j = 0; j < 4; j++)
#pragma unroll
          for (int v = 0; v < 4; v++) acc[i][j][v] %= p;
    }
  }
  cp_wait<0>();

  const int g = lane >> 2, t = lane & 3;
  const int hi = (int)gc.hi[l], lo = (int)gc.lo[l];
  if (!OS2_DBG_GUARD(l < gc.N && n <= ldo, status)) return;
#pragma unroll
  for (int i = 0; i < 4; i++)
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int row = tm + wm * 64 + i * 16 + g + 8 * h;
      if (row >= m) continue;
#pragma unroll
      for (int j = 0; j < 4; j++) {
        const int col = tn + wn * 32 + j * 8 + 2 * t;
        if (col >= n) continue;
        const int x0 = acc[i][j][2 * h], x1 = acc[i][j][2 * h + 1];
        const size_t o = ((size_t)l * m + row) * ldo + col;
        if (OUT == OS2_OUT_RAW_INT32) {
          int32_t *d = reinterpret_cast<int32_t *>(out) + o;
          if (col + 1 < n)
            *reinterpret_cast<int2 *>(d) = make_int2(x0, x1);
          else
            d[0] = x0;
        } else {
          int r0 = x0 % p, r1 = x1 % p;
          r0 = r0 > hi ? r0 - p : (r0 < lo ? r0 + p : r0);
          r1 = r1 > hi ? r1 - p : (r1 < lo ? r1 + p : r1);
          int8_t *d = reinterpret_cast<int8_t *>(out) + o;
          if (col + 1 < n)
            *reinterpret_cast<uint16_t *>(d) =
                (uint16_t)((uint32_t)(uint8_t)r0 | ((uint32_t)(uint8_t)r1 << 8));
          else
            d[0] = (int8_t)r0;
        }
      }
    }
}

template <int OUT>
cudaError_t launch_t(int m, int n, int kp, const int8_t *RA, const int8_t *RB, int b_plane_rows,
                     int N, void *out, int ldo, const Os2Tables *t, int *status, cudaStream_t s) {
  static cudaError_t attr = cudaFuncSetAttribute(
      k_gemm_s8<OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (attr != cudaSuccess) return attr;
  const dim3 grid((n + BN - 1) / BN, (m + BM - 1) / BM, N);
  k_gemm_s8<OUT><<<grid, kThreads, kSmem, s>>>(m, n, kp, RA, RB, b_plane_rows, out, ldo, t->gemm,
                                              status);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_s8(int m, int n, int kp, const void *RA, const void *RB, int N,
                           int out_kind, void *out, int ldo, const Os2Tables *t, int *status,
                           cudaStream_t s, int b_plane_rows) {
  if (m <= 0 || n <= 0 || N <= 0) return cudaSuccess;
  if (m > 65535 * BM || kp % 16) return cudaErrorInvalidValue;
  const int8_t *a = reinterpret_cast<const int8_t *>(RA);
  const int8_t *b = reinterpret_cast<const int8_t *>(RB);
  const int bpr = b_plane_rows > 0 ? b_plane_rows : n;
  return out_kind == OS2_OUT_RAW_INT32
             ? launch_t<OS2_OUT_RAW_INT32>(m, n, kp, a, b, bpr, N, out, ldo, t, status, s)
             : launch_t<OS2_OUT_MODP_INT8>(m, n, kp, a, b, bpr, N, out, ldo, t, status, s);
}
