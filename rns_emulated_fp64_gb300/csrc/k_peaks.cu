// Pipe-peak probes: the throughput ceiling of the tensor-core paths this
// library can use on sm_103a, measured by its own kernels (a measurement aid;
// the pages have no counterpart).  They give step 3's roofline a same-pipe
// denominator next to the cuBLAS BF16 figure.
//
//  PROBE_F16_1SM  tcgen05.mma.cta_group::1.kind::f16, M = 128, N = 256, K = 16,
//                 FP32 accumulator in TMEM, operands resident in shared memory
//                 (one 128 x 64 A tile and one 256 x 64 B tile, 128-byte
//                 swizzle, the layout step 3 uses).  One CTA per SM.
//  PROBE_F16_2SM  the same with cta_group::2 on CTA pairs, M = 256, N = 256
//                 (the instruction form of step 3's kernel).
//  PROBE_S8_SYNC  mma.sync.m16n8k32 s8 x s8 -> s32 from registers: the INT8
//                 tensor path that sm_103a offers outside tcgen05 (it has no
//                 tcgen05 kind::i8).  Eight independent accumulators per warp.
//
// Operand values are small signed integers given by a fixed formula of (row,
// k), like step 3's residues, so every product is exact.  With `check` set the
// probe compares the whole result with the same formula evaluated on the CUDA
// cores and adds the mismatches to result[0] (result[1] counts the CTAs that
// checked); timed runs pass check = 0.  Every wait is bounded: on expiry the
// CTA records OS2_ERR_TIMEOUT, waits once more (bounded) for its MMAs and
// frees its TMEM.
#include <cuda_fp16.h>

#include "os2_internal.cuh"
#include "ptx.cuh"

using namespace os2ptx;

namespace {

constexpr long long kProbeWait = 4000000000LL;  // clock cycles (about 2 s)

__host__ __device__ __forceinline__ int val_a(int r, int k) {
  return (int)((unsigned)(r * 37 + k * 11 + ((r * k) >> 3)) % 255u) - 127;
}
__host__ __device__ __forceinline__ int val_b(int n, int k) {
  return (int)((unsigned)(n * 29 + k * 13 + (n ^ k) * 7) % 251u) - 125;
}

// Byte offset of element (row, k) in a K-major tile of 64 FP16 per row with
// the 128-byte swizzle (atoms of 8 rows x 128 bytes, 1024 bytes apart).
__device__ __forceinline__ uint32_t sw128_off(int row, int k) {
  return (uint32_t)((row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 3) ^ (row & 7))) << 4) +
                    (k & 7) * 2);
}

__device__ __forceinline__ void fill_tile(uint8_t *tile, int rows, int row0, bool is_a) {
  for (int e = threadIdx.x; e < rows * 64; e += blockDim.x) {
    const int r = e >> 6, k = e & 63;
    const int v = is_a ? val_a(row0 + r, k) : val_b(row0 + r, k);
    *reinterpret_cast<__half *>(tile + sw128_off(r, k)) = __int2half_rn(v);
  }
}

// Compares this thread's TMEM lane (row `arow` of D, 256 columns) with the
// exact product of the formula operands.
__device__ __forceinline__ int check_row(uint32_t lane_addr, int arow) {
  int bad = 0;
#pragma unroll 1
  for (int g = 0; g < 8; g++) {
    uint32_t v[32];
    tmem_ld32(lane_addr + g * 32, v);
    tmem_wait_ld();
#pragma unroll 1
    for (int i = 0; i < 32; i++) {
      int s = 0;
      for (int k = 0; k < 64; k++) s += val_a(arow, k) * val_b(g * 32 + i, k);
      if (__uint_as_float(v[i]) != (float)s) bad++;
    }
  }
  return bad;
}

template <int PAIR>
__global__ void __launch_bounds__(128, 1)
    k_peak_f16(int iters, int check, int32_t *result, int *status) {
  constexpr int A_ROWS = 128, B_ROWS = PAIR ? 128 : 256;
  constexpr uint32_t A_BYTES = A_ROWS * 128, B_BYTES = B_ROWS * 128;
  constexpr uint32_t IDESC = idesc_f16_f32(PAIR ? 256 : 128, 256);
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem, *sB = smem + A_BYTES;
  uint64_t *bar = reinterpret_cast<uint64_t *>(sB + B_BYTES);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bar + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = PAIR ? cluster_ctarank() : 0;

  fill_tile(sA, A_ROWS, (int)rank * 128, true);
  fill_tile(sB, B_ROWS, (int)rank * 128, false);
  fence_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    if (PAIR) {
      tmem_alloc2(s_tmem, 256);
      tmem_relinquish2();
    } else {
      tmem_alloc(s_tmem, 256);
      tmem_relinquish();
    }
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (threadIdx.x == 0 && rank == 0) {
    const uint64_t ad = sdesc_k128(smem_u32(sA)), bd = sdesc_k128(smem_u32(sB));
#pragma unroll 1
    for (int it = 0; it < iters; it++) {
#pragma unroll
      for (int kk = 0; kk < 4; kk++) {
        if (PAIR)
          umma2_f16(tmem, ad + 2 * kk, bd + 2 * kk, IDESC, kk > 0 ? 1u : 0u);
        else
          umma_f16(tmem, ad + 2 * kk, bd + 2 * kk, IDESC, kk > 0 ? 1u : 0u);
      }
    }
    if (PAIR)
      umma2_commit_mc(bar, 0x3);
    else
      umma_commit(bar);
  }
  volatile int no_abort = 0;
  bool ok = mbar_wait_bounded(bar, 0, &no_abort, kProbeWait);
  if (!ok) {
    if (threadIdx.x == 0 && status) atomicCAS(status, 0, OS2_ERR_TIMEOUT);
    mbar_wait_bounded(bar, 0, &no_abort, kProbeWait);
  }
  tc_fence_after();
  if (check && ok) {
    const int bad = check_row(tmem + ((uint32_t)(warp * 32) << 16), (int)rank * 128 + warp * 32 + lane);
    atomicAdd(&result[0], bad);
    if (threadIdx.x == 0) atomicAdd(&result[1], 1);
  }
  tc_fence_before();
  __syncthreads();
  if (PAIR) cluster_sync();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    if (PAIR)
      tmem_dealloc2(tmem, 256);
    else
      tmem_dealloc(tmem, 256);
  }
}

// Four int8 values of the formula packed little-endian.
__device__ __forceinline__ uint32_t pack_a(int r, int k0) {
  uint32_t w = 0;
  for (int i = 0; i < 4; i++) w |= ((uint32_t)val_a(r, k0 + i) & 0xFFu) << (8 * i);
  return w;
}
__device__ __forceinline__ uint32_t pack_b(int n, int k0) {
  uint32_t w = 0;
  for (int i = 0; i < 4; i++) w |= ((uint32_t)val_b(n, k0 + i) & 0xFFu) << (8 * i);
  return w;
}

__device__ __forceinline__ void mma_s8(int (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// A 16 x 32 (rows = the warp's 16 rows, from the warp index), B 32 x 8.
// Fragments: lane = 4 g + t; a0 = A[g][4t..4t+3], a1 = A[g+8][4t..], a2 =
// A[g][16+4t..], a3 = A[g+8][16+4t..]; b0 = B[4t..4t+3][g], b1 =
// B[16+4t..][g]; c0, c1 = D[g][2t, 2t+1], c2, c3 = D[g+8][2t, 2t+1].
__global__ void __launch_bounds__(256) k_peak_s8(int iters, int check, int32_t *result) {
  const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
  const int r0 = (threadIdx.x >> 5) * 16;
  uint32_t a[4] = {pack_a(r0 + g, 4 * t), pack_a(r0 + g + 8, 4 * t), pack_a(r0 + g, 16 + 4 * t),
                   pack_a(r0 + g + 8, 16 + 4 * t)};
  uint32_t b[2] = {pack_b(g, 4 * t), pack_b(g, 16 + 4 * t)};
  int c[8][4];
#pragma unroll
  for (int j = 0; j < 8; j++)
#pragma unroll
    for (int q = 0; q < 4; q++) c[j][q] = 0;
#pragma unroll 1
  for (int it = 0; it < iters; it++) {
#pragma unroll
    for (int j = 0; j < 8; j++) mma_s8(c[j], a, b);
  }
  if (check) {
    int bad = 0;
#pragma unroll
    for (int q = 0; q < 4; q++) {
      const int row = r0 + g + (q >> 1) * 8, col = 2 * t + (q & 1);
      int s = 0;
      for (int k = 0; k < 32; k++) s += val_a(row, k) * val_b(col, k);
      const int want = s * iters;
#pragma unroll
      for (int j = 0; j < 8; j++) bad += c[j][q] != want;
    }
    atomicAdd(&result[0], bad);
    if (threadIdx.x == 0) atomicAdd(&result[1], 1);
  } else {
    int x = 0;
#pragma unroll
    for (int j = 0; j < 8; j++) x ^= c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
    if (x == 0x7FFFFFFF && result) result[2] = x;  // keeps the loop live; never true for these values
  }
}

template <int PAIR>
cudaError_t launch_f16(int iters, int check, int32_t *result, int *status, cudaStream_t s,
                       double *flop) {
  constexpr size_t smem = 1024 + 128 * 128 + (PAIR ? 128 : 256) * 128 + 64;
  cudaError_t e = cudaFuncSetAttribute(k_peak_f16<PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e) return e;
  const int sms = os2_sm_count();
  const int grid = PAIR ? (sms / 2) * 2 : sms;
  if (flop) *flop = (double)(PAIR ? grid / 2 : grid) * iters * 4.0 * 2.0 * (PAIR ? 256 : 128) * 256 * 16;
  if (PAIR) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, k_peak_f16<1>, iters, check, result, status);
    if (e) return e;
  } else {
    k_peak_f16<0><<<grid, 128, smem, s>>>(iters, check, result, status);
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_peak_probe(int kind, int iters, int check, int32_t *result, int *status,
                              cudaStream_t s, double *flop) {
  if (kind == OS2_PROBE_F16_1SM) return launch_f16<0>(iters, check, result, status, s, flop);
  if (kind == OS2_PROBE_F16_2SM) return launch_f16<1>(iters, check, result, status, s, flop);
  if (kind == OS2_PROBE_S8_SYNC) {
    const int grid = os2_sm_count() * 4;
    if (flop) *flop = (double)grid * 8 * iters * 8.0 * 2.0 * 16 * 8 * 32;
    k_peak_s8<<<grid, 256, 0, s>>>(iters, check, result);
    return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}
