// Steps 4 and 5 with the limb sums on the tensor cores.
//
// [Q] "繰り上がりのない計算" / "秦九韶の大衍求一術": the integer with residues c_l is
// X = (sum_l c_l W_l) mod P with the use numbers W_l = M_l inv_l; [Q]
// "高い精度での復元(手順4)": P passes 2^125 at 16 moduli, so this needs more than
// double precision.  Here X is computed exactly.  Write every W_l in signed
// 10-bit digits, W_l = sum_t w_{l,t} 2^(10 t) with |w_{l,t}| <= 512.  Then
//   Y = sum_l (c_l + 128) W_l = sum_t d_t 2^(10 t),  d_t = sum_l (c_l + 128) w_{l,t},
// and each digit sum d_t is an entry of the small matrix product
//   [entries x N residues] . [N x T digits],
// which runs as one FP16 tensor-core MMA per 128 entries: the A operand holds
// 1152 + c_l = 1024 + (c_l + 128) (the FP16 whose bit pattern is 0x64 followed
// by the byte c_l ^ 0x80, so an int8 plane widens with two byte permutes per
// four entries), the B operand the digits w_{l,t}.  Every product and partial
// sum is an integer below 1279 * 512 * 20 < 2^24, so the FP32 accumulator is
// exact; subtracting 1024 sum_l w_{l,t} leaves |d_t| < 255 * 512 * 20 < 2^22,
// and adding 1.5 * 2^23 in the same FP32 add puts 0x4B400000 + d_t in the bit
// pattern.  The CUDA cores then only
//   - fold the T digit patterns into 32-bit limbs (one 32 x 32 -> 64 multiply-
//     add each; the 0x4B400000 offsets and the -128 below are one constant),
//   - estimate q = round((Y - 128) / P) >= 0 from the top digits in FP32
//     (error below 0.003; the W_l sum to 1 mod P, so Y - 128 = S mod P),
//   - form X = Y - 128 - q P modulo 2^(32 LX) (X lies in [-P/2, P/2); LX is
//     the smallest limb count with 2^(32 LX) > 3P, so X +- P keeps its sign),
//     fix q by one exact comparison with P/2 when the estimate sat near a
//     half-integer, and
//   - round X 2^-(e_i + f_j) once to nearest-even ([Q] "2の累乗による整数化(手順1と5)").
// The results are bit-identical to the CUDA-core kernel (k_crt.cu).
//
// Layout: a persistent CTA of 8 warps takes rounds of 512 consecutive entries of
// one row of C.  Each warp reads moduli l = warp, warp + 8, ... as 16-byte loads
// (32 lanes x 16 entries), widens them into an MN-major, 128-byte-swizzled FP16
// tile (entries contiguous, one 8-row atom per 8 moduli), and one thread issues
// four MMAs of 128 entries into TMEM.  Rounds are double-buffered in shared
// memory and TMEM: the next round's loads and MMAs run while the warps fold the
// previous round's digit sums (tcgen05.ld: lane = entry, columns = digits; a
// warp reads its TMEM lane quarter of two of the four tiles, so each thread
// reconstructs two independent entries per round, their exponents loaded one
// round ahead).
// Every wait is bounded; on expiry the CTA records OS2_ERR_TIMEOUT, waits once
// more (bounded) for its MMAs, frees its TMEM and returns.
#include <cuda_fp16.h>

#include <algorithm>

#include "crt_round.cuh"
#include "os2_internal.cuh"
#include "ptx.cuh"

using namespace os2ptx;
using namespace os2crt;

namespace {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr int kU = 4;                 // MMA tiles of 128 entries per round
constexpr int kSeg = 128 * kU;        // entries per round
constexpr long long kWait = 4000000000LL;  // clock cycles (about 2 s)

// Signed 10-bit digits of the W_l and the top digits that fix q, per N
// (checked against the tables the host builds).
constexpr int kDigits[OS2_MAX_MODULI + 1] = {0, 1, 2, 3, 4, 5, 5, 6, 7, 8, 9,
                                             9, 10, 11, 12, 12, 13, 14, 15, 15, 16};
constexpr int kQDigits[OS2_MAX_MODULI + 1] = {0, 1, 2, 3, 4, 5, 4, 4, 4, 4, 5,
                                              4, 4, 4, 5, 4, 4, 4, 5, 4, 4};
// 32-bit limbs of X: the smallest LX with 2^(32 LX) > 3P, so that X +- P (a
// quotient one off) still has the right sign in LX limbs.
constexpr int kLimbs[OS2_MAX_MODULI + 1] = {0, 1, 1, 1, 2, 2, 2, 2, 3, 3, 3,
                                            3, 4, 4, 4, 4, 4, 5, 5, 5, 5};

template <int N>
struct Shape {
  static constexpr int KPAD = N <= 16 ? 16 : 32;        // moduli, padded to MMA K
  static constexpr int NMMA = N <= 16 ? 16 : 32;        // digit columns (>= T)
  static constexpr int T = kDigits[N], Q = kQDigits[N];
  static constexpr int LX = kLimbs[N];
  static constexpr int MPW = (N + kWarps - 1) / kWarps; // moduli each warp loads
  static constexpr uint32_t SBO = 2048;                 // 8-modulus atoms, 2 x 1024 B apart
  static constexpr uint32_t A_TILE = 128 * KPAD * 2;    // one MMA's A (bytes)
  static constexpr uint32_t A_BUF = kU * A_TILE;
  static constexpr uint32_t B_BYTES = NMMA * 128;       // K-major rows of 128 bytes
  static constexpr uint32_t TMEM_COLS = 2 * kU * NMMA;  // 128 or 256
  static constexpr int PER_SM = 512 / TMEM_COLS;        // CTAs whose TMEM fits one SM
  static constexpr size_t SMEM_USED = 1024 + 2 * (size_t)A_BUF + B_BYTES + 64;
  // TMEM is not a scheduling resource: the shared memory is padded so that no
  // more than PER_SM CTAs fit on an SM (228 KB), and none beside a product CTA,
  // so tcgen05.alloc never has to wait.
  static constexpr size_t SMEM = PER_SM == 4 ? 52 * 1024 : 104 * 1024;
  static_assert(SMEM_USED <= SMEM, "shared memory layout exceeds its padding");
};

__device__ __forceinline__ uint4 ldg16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void sts16(uint32_t saddr, uint32_t a, uint32_t b, uint32_t c,
                                      uint32_t d) {
  asm volatile("st.shared.v4.u32 [%0], {%1,%2,%3,%4};" ::"r"(saddr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// FP16 1152 + c for the four int8 residues c of a word: [c0 c1] and [c2 c3].
__device__ __forceinline__ void widen4(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t x = w ^ 0x80808080u;
  lo = __byte_perm(x, 0x64646464u, 0x4140);
  hi = __byte_perm(x, 0x64646464u, 0x4342);
}

// One entry: digit sums v[0..T) (FP32 bit patterns) -> C[i][j] (and X).
template <int N, typename OutT>
__device__ __forceinline__ void finish_entry(const uint32_t *v, const CrtTcConsts &cc, int s_exp,
                                             OutT *dst, uint32_t *xo) {
  using S = Shape<N>;
  constexpr int T = S::T, Q = S::Q, LX = S::LX;
  uint64_t acc[LX];
#pragma unroll
  for (int u = 0; u < LX; u++) acc[u] = cc.negc[u];
  float dq[Q];
#pragma unroll
  for (int t = 0; t < T; t++) {
    const float r = __uint_as_float(v[t]) + cc.rmag[t];  // exact: 1.5 * 2^23 + d_t
    const int u0 = (10 * t) >> 5;
    if (u0 < LX) acc[u0 < LX ? u0 : 0] += (uint64_t)__float_as_uint(r) * cc.pw[t];
    if (t >= T - Q) dq[T - 1 - t] = r - 12582912.0f;     // d_t, exact
  }
  // q = round((Y - 128) / P) from the top Q digits
  float tq = cc.c0;
#pragma unroll
  for (int j = Q - 1; j >= 0; j--) tq = fmaf(dq[j], cc.s[j], tq);
  // Y >= 0, so tq >= -128/P - 0.003 and the rounded q is never negative
  const float tr = tq + 12582912.0f;
  const uint32_t qi = (uint32_t)(__float_as_int(tr) - 0x4B400000);
  const float qf = tr - 12582912.0f;
#pragma unroll
  for (int u = 0; u < LX; u++) acc[u] += (uint64_t)qi * cc.np[u];
  uint32_t x[LX];
  uint64_t cy = 0;
#pragma unroll
  for (int u = 0; u < LX; u++) {
    const uint64_t sum = acc[u] + cy;
    x[u] = (uint32_t)sum;
    cy = sum >> 32;
  }
  // near a half-integer the estimate may be one off: compare X with +-P/2
  const float fr = tq - qf;
  if (fr > 0.49f || fr < -0.49f) {
    const bool up = fr > 0.49f;  // X may be >= P/2 (then X -= P); else X may be < -P/2
    long long cr = 0;
    uint32_t last = 0;
#pragma unroll
    for (int u = 0; u < LX; u++) {
      const long long dv = (long long)x[u] + (up ? -(long long)cc.H32[u] : (long long)cc.H32[u]) + cr;
      last = (uint32_t)dv;
      cr = dv >> 32;
    }
    const bool dneg = (int32_t)last < 0;  // sign of X -+ P/2 (within LX limbs)
    if (up ? !dneg : dneg) {
      long long cr2 = 0;
#pragma unroll
      for (int u = 0; u < LX; u++) {
        const long long sv =
            (long long)x[u] + (up ? -(long long)cc.P32[u] : (long long)cc.P32[u]) + cr2;
        x[u] = (uint32_t)sv;
        cr2 = sv >> 32;
      }
    }
  }
  const uint32_t sm = (uint32_t)((int32_t)x[LX - 1] >> 31);  // all ones if X < 0
  if (xo) {
#pragma unroll
    for (int u = 0; u < 8; u++) xo[u] = u < LX ? x[u < LX ? u : 0] : sm;
  }
  // |X| = (X xor sm) - sm
  uint32_t mag[LX];
  uint64_t c1 = sm & 1u;
#pragma unroll
  for (int u = 0; u < LX; u++) {
    c1 += (uint64_t)(x[u] ^ sm);
    mag[u] = (uint32_t)c1;
    c1 >>= 32;
  }
  *dst = round_scaled_top<OutT, LX>(mag, sm != 0, s_exp);
}

template <int N, typename OutT>
__global__ void __launch_bounds__(kThreads, 512 / (2 * kU * Shape<N>::NMMA))
    k_crt_tc(int m, int n, int segs, int rounds, const int8_t *__restrict__ c, int ldcres,
             const int32_t *__restrict__ e, const int32_t *__restrict__ f, OutT *__restrict__ C,
             int ldc, uint32_t *__restrict__ Xout, const __grid_constant__ CrtTcConsts cc,
             int *status) {
  using S = Shape<N>;
  constexpr int NMMA = S::NMMA, MPW = S::MPW;
  constexpr uint32_t IDESC = idesc_f16_f32(128, NMMA) | (1u << 15);  // A MN-major
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~uintptr_t(1023));
  uint8_t *sA = smem;                         // [2][kU][A_TILE]
  uint8_t *sB = smem + 2 * S::A_BUF;          // [NMMA rows][128 B]
  uint64_t *bars = reinterpret_cast<uint64_t *>(sB + S::B_BYTES);
  uint32_t *s_tmem = reinterpret_cast<uint32_t *>(bars + 2);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // zero both A buffers (the padding moduli stay 0) and build the digit tile
  for (uint32_t o = threadIdx.x * 16; o < 2 * S::A_BUF; o += kThreads * 16)
    *reinterpret_cast<uint4 *>(sA + o) = make_uint4(0, 0, 0, 0);
  for (int idx = threadIdx.x; idx < NMMA * 64; idx += kThreads) {
    const int row = idx >> 6, k = idx & 63;  // row = digit t, k = modulus l
    const int w = (row < S::T && k < N) ? cc.wd[k < N ? k : 0][row < S::T ? row : 0] : 0;
    const uint32_t off = (row >> 3) * 1024 + (row & 7) * 128 + ((((k >> 3) ^ (row & 7))) << 4) +
                         (k & 7) * 2;
    *reinterpret_cast<__half *>(sB + off) = __int2half_rn(w);
  }
  fence_async_smem();
  if (threadIdx.x == 0) {
    mbar_init(&bars[0], 1);
    mbar_init(&bars[1], 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(s_tmem, S::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *s_tmem;
  const size_t plane = (size_t)m * ldcres;

  // loads: this lane's 16 entries of a round (tile u, entries e0 .. e0+15 of
  // it) of moduli warp, warp + 8, ...
  const int eR = 16 * lane;
  const int tile = eR >> 7, e0 = eR & 127;
  // reconstruction: TMEM lane quarter `quarter`, tiles 2 half and 2 half + 1
  const int quarter = warp & 3, half = warp >> 2;
  uint4 raw[MPW];
  auto load = [&](int i, int sg) {
    const int j = sg * kSeg + eR;
    const int8_t *src = c + (size_t)i * ldcres + j;
#pragma unroll
    for (int q = 0; q < MPW; q++) {
      const int l = warp + kWarps * q;
      raw[q] = (l < N && j < ldcres && OS2_DBG_GUARD(i < m && j + 16 <= ldcres, status))
                   ? ldg16(src + (size_t)(l < N ? l : 0) * plane)
                   : make_uint4(0, 0, 0, 0);
    }
  };
  // exponent sums e_i + f_j of this thread's two entries of a round
  auto load_exp = [&](int i, int sg, int (&ef)[2]) {
    const int jr = sg * kSeg;
    const int ei = __ldg(e + i);
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int j = jr + (2 * half + h) * 128 + quarter * 32 + lane;
      ef[h] = j < n ? ei + __ldg(f + j) : 0;
    }
  };
  auto stage = [&](int buf) {
    const uint32_t tbase = smem_u32(sA) + buf * S::A_BUF + tile * S::A_TILE + (e0 >> 6) * 1024;
    const int ch = (e0 >> 3) & 7;  // even: this lane's two 16-byte chunks are ch, ch + 1
#pragma unroll
    for (int q = 0; q < MPW; q++) {
      const int l = warp + kWarps * q;
      if (l < N) {
        uint32_t h[8];
        widen4(raw[q].x, h[0], h[1]);
        widen4(raw[q].y, h[2], h[3]);
        widen4(raw[q].z, h[4], h[5]);
        widen4(raw[q].w, h[6], h[7]);
        const uint32_t rowa = tbase + (l >> 3) * S::SBO + (l & 7) * 128;
        sts16(rowa + ((ch ^ (l & 7)) << 4), h[0], h[1], h[2], h[3]);
        sts16(rowa + (((ch + 1) ^ (l & 7)) << 4), h[4], h[5], h[6], h[7]);
      }
    }
  };
  auto issue = [&](int buf) {
    const uint64_t bd = sdesc_k128(smem_u32(sB));
#pragma unroll
    for (int u = 0; u < kU; u++) {
      const uint32_t abase = smem_u32(sA) + buf * S::A_BUF + u * S::A_TILE;
      const uint32_t d = tmem_base + (uint32_t)((buf * kU + u) * NMMA);
#pragma unroll
      for (int kk = 0; kk < S::KPAD / 16; kk++)
        umma_f16(d, sdesc_mn128(abase + kk * 2 * S::SBO, 1024, S::SBO), bd + 2 * kk, IDESC,
                 kk > 0 ? 1u : 0u);
    }
    umma_commit(&bars[buf]);
  };
  // this thread's two entries of round r: both TMEM loads, one wait, then
  // the two independent reconstructions
  auto post = [&](int i, int sg, int buf, const int (&ef)[2]) {
    const int jr = sg * kSeg;
    uint32_t v[2][NMMA];
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const uint32_t taddr = tmem_base + ((uint32_t)(quarter * 32) << 16) +
                             (uint32_t)((buf * kU + 2 * half + h) * NMMA);
      if (NMMA == 16)
        tmem_ld16(taddr, *reinterpret_cast<uint32_t(*)[16]>(v[h]));
      else
        tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(v[h]));
    }
    tmem_wait_ld();
#pragma unroll
    for (int h = 0; h < 2; h++) {
      const int j = jr + (2 * half + h) * 128 + quarter * 32 + lane;
      if (j < n && OS2_DBG_GUARD(i < m && n <= ldc, status))
        finish_entry<N, OutT>(v[h], cc, ef[h], C + (size_t)i * ldc + j,
                              Xout ? Xout + ((size_t)i * n + j) * 8 : nullptr);
    }
  };

  volatile int no_abort = 0;
  bool ok = true;
  int it = 0;
  int r = blockIdx.x;
  int ef_post[2] = {0, 0}, ef_next[2] = {0, 0};
  // round r = i * segs + sg, stepped by the grid without divisions
  const int di = (int)gridDim.x / segs, ds = (int)gridDim.x - di * segs;
  int ci = r / segs, cs = r - ci * segs;  // round r
  int pi = 0, ps = 0;                     // the round before it
  if (r < rounds) load(ci, cs);
  for (; r < rounds; r += gridDim.x, it++) {
    const int buf = it & 1;
    stage(buf);  // the MMAs that last read this buffer completed (waited on in post)
    fence_async_smem();
    tc_fence_before();
    ok = __syncthreads_and(ok);
    if (!ok) break;
    tc_fence_after();
    if (threadIdx.x == 0) issue(buf);
    // next round's residues and this round's exponents: issued after the
    // proxy fence (which may wait for outstanding memory operations), in
    // flight while the previous round is reconstructed
    int ni = ci + di, ns = cs + ds;
    if (ns >= segs) {
      ns -= segs;
      ni++;
    }
    if (r + (int)gridDim.x < rounds) load(ni, ns);
    ef_post[0] = ef_next[0];
    ef_post[1] = ef_next[1];
    load_exp(ci, cs, ef_next);  // used one iteration later, by post of this round
    if (it > 0) {
      if (mbar_wait_bounded(&bars[buf ^ 1], ((it - 1) >> 1) & 1, &no_abort, kWait)) {
        tc_fence_after();
        post(pi, ps, buf ^ 1, ef_post);
      } else {
        ok = false;
      }
    }
    pi = ci;
    ps = cs;
    ci = ni;
    cs = ns;
  }
  if (ok && it > 0) {
    if (mbar_wait_bounded(&bars[(it - 1) & 1], ((it - 1) >> 1) & 1, &no_abort, kWait)) {
      tc_fence_after();
      post(pi, ps, (it - 1) & 1, ef_next);
    } else {
      ok = false;
    }
  }
  if (!ok) {
    if (status) atomicCAS(status, 0, OS2_ERR_TIMEOUT);
    // let the MMAs already issued finish before the TMEM is freed
    for (int b = 0; b < 2; b++) {
      const int uses = (it + 1 - b) / 2;  // issues on buffer b so far (upper bound)
      if (uses > 0) mbar_wait_bounded(&bars[b], (uses - 1) & 1, &no_abort, kWait);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem_base, S::TMEM_COLS);
  }
}

template <int N, typename OutT>
cudaError_t launch_n(int m, int n, const int8_t *c, int ldcres, const int32_t *e, const int32_t *f,
                     OutT *C, int ldc, uint32_t *X_out, const Os2Tables *t, int *status,
                     cudaStream_t s) {
  using S = Shape<N>;
  if (t->crt_tc.T != S::T || t->crt_tc.Q != S::Q || t->crt_tc.LX != S::LX)
    return cudaErrorInvalidValue;
  static cudaError_t attr = cudaFuncSetAttribute(
      k_crt_tc<N, OutT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
  if (attr != cudaSuccess) return attr;
  const int segs = (n + kSeg - 1) / kSeg;
  const long long rounds = (long long)m * segs;
  if (rounds > (1LL << 31) - 1) return cudaErrorInvalidValue;
  const int grid = (int)std::min<long long>(rounds, (long long)os2_sm_count() * S::PER_SM);
  k_crt_tc<N, OutT><<<grid, kThreads, S::SMEM, s>>>(m, n, segs, (int)rounds, c, ldcres, e, f, C,
                                                   ldc, X_out, t->crt_tc, status);
  return cudaGetLastError();
}

template <typename OutT>
cudaError_t crt_tc_t(int m, int n, const int8_t *c, int ldcres, const int32_t *e, const int32_t *f,
                     OutT *C, int ldc, uint32_t *X_out, const Os2Tables *t, int *status,
                     cudaStream_t s) {
  switch (t->N) {
#define OS2_CASE(NN) \
  case NN: return launch_n<NN, OutT>(m, n, c, ldcres, e, f, C, ldc, X_out, t, status, s);
    OS2_CASE(1) OS2_CASE(2) OS2_CASE(3) OS2_CASE(4) OS2_CASE(5) OS2_CASE(6) OS2_CASE(7)
    OS2_CASE(8) OS2_CASE(9) OS2_CASE(10) OS2_CASE(11) OS2_CASE(12) OS2_CASE(13) OS2_CASE(14)
    OS2_CASE(15) OS2_CASE(16) OS2_CASE(17) OS2_CASE(18) OS2_CASE(19) OS2_CASE(20)
#undef OS2_CASE
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_crt_tc(bool f32, int m, int n, const int8_t *c, int ldcres, const int32_t *e,
                          const int32_t *f, void *C, int ldc, uint32_t *X_out, const Os2Tables *t,
                          int *status, cudaStream_t s) {
  if (m <= 0 || n <= 0) return cudaSuccess;
  if (ldcres % 16 || (reinterpret_cast<uintptr_t>(c) & 15)) return cudaErrorInvalidValue;
  return f32 ? crt_tc_t<float>(m, n, c, ldcres, e, f, static_cast<float *>(C), ldc, X_out, t,
                               status, s)
             : crt_tc_t<double>(m, n, c, ldcres, e, f, static_cast<double *>(C), ldc, X_out, t,
                                status, s);
}
