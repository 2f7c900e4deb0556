// Steps 1 and 2: per-row power-of-two scaling and symmetric residue planes.
//
// [G] "Improved Scaling for Fast Mode of Ozaki Scheme II", "Methodik" 1: the
// revised fast-mode exponent mu_i = 2^floor(P' - 0.5 (log2 sum_h a_ih^2 + 4 u32)).
// Here log2 of the sum is replaced by an exact integer upper bound, so the
// result is reproducible and independent of summation order:
//   E_i = tight exponent bound, |a_ih| < 2^E_i
//   Q_i = sum_h ceil(|a_ih| 2^(23 - E_i))^2            (exact, uint64)
//   e_i = g + 23 - E_i, g the largest integer with Q_i 4^g <= H = floor((P-1)/2)
// which gives mu_i^2 sum_h a_ih^2 <= H, half of the sufficient condition
// 2 mu_i ||a_i|| ||b_j|| nu_j <= P - 1.
//
// [Q] "2の累乗による整数化(手順1と5)" / "256以下の法の選び方(手順2)": the scaled
// integers trunc(a_ih 2^e_i) are reduced to residues held around zero,
// [-floor(p/2), ceil(p/2) - 1], which always fit int8 and are stored as FP16
// (exact for |r| <= 2048) for the tensor-core products of step 3.
//
// Layout: one CTA of 256 threads per row; the row is read up to three times
// (exponent, sum of squares, residues), the re-reads hit L1/L2.  Every
// residue plane row is written with 16-byte stores, 8 values per thread.
#include <cuda_fp16.h>
#include <limits.h>

#include "os2_internal.cuh"

namespace {

constexpr int kThreads = 256;

struct Dec {
  uint64_t mant;  // |x| = mant * 2^ex2
  int ex2;
  uint32_t neg;
  bool nonfinite;
};

__device__ __forceinline__ Dec decode(double x) {
  uint64_t b = (uint64_t)__double_as_longlong(x);
  int bexp = (int)((b >> 52) & 0x7FF);
  Dec d;
  d.neg = (uint32_t)(b >> 63);
  d.nonfinite = bexp == 0x7FF;
  d.mant = b & 0xFFFFFFFFFFFFFull;
  if (bexp) d.mant |= 1ull << 52;
  else bexp = 1;
  d.ex2 = bexp - 1075;
  if (d.nonfinite) d.mant = 0;
  return d;
}

// Tight E with |x| < 2^E; INT_MIN for zero.
__device__ __forceinline__ int exp_bound(const Dec &d) {
  return d.mant ? d.ex2 + (64 - __clzll((long long)d.mant)) : INT_MIN;
}

// ceil(mant * 2^sh), sh <= 0 in every use here.
__device__ __forceinline__ uint64_t ceil_shift(uint64_t mant, int sh) {
  if (mant == 0) return 0;
  if (sh >= 0) return mant << sh;
  int r = -sh;
  if (r >= 64) return 1;
  return (mant + ((1ull << r) - 1)) >> r;
}

// Multiword compare: Q * 4^g <= H (H: OS2_H_LIMBS little-endian 32-bit limbs).
__device__ void shl8(const uint32_t *src, int nsrc, int s, uint32_t *dst) {
  int q = s >> 5, b = s & 31;
  for (int i = 0; i < 8; i++) {
    int j = i - q;
    uint32_t cur = (j >= 0 && j < nsrc) ? src[j] : 0u;
    uint32_t prev = (j - 1 >= 0 && j - 1 < nsrc) ? src[j - 1] : 0u;
    dst[i] = b ? ((cur << b) | (prev >> (32 - b))) : cur;
  }
}
__device__ bool fits(uint64_t Q, int g, const uint32_t *H) {
  uint32_t q2[2] = {(uint32_t)Q, (uint32_t)(Q >> 32)};
  uint32_t L[8], R[8];
  shl8(q2, 2, g > 0 ? 2 * g : 0, L);
  shl8(H, OS2_H_LIMBS, g < 0 ? -2 * g : 0, R);
  for (int i = 7; i >= 0; i--)
    if (L[i] != R[i]) return L[i] < R[i];
  return true;
}
// Largest integer g with Q * 4^g <= H, Q >= 1.  With b(.) the bit length,
// the answer is floor((b(H)+1-b(Q))/2) or one less.
__device__ int largest_g(uint64_t Q, const ResConsts &c) {
  int bQ = 64 - __clzll((long long)Q);
  int g = (c.bitlenH + 1 - bQ) >> 1;
  for (int it = 0; it < 3; it++, g--)
    if (fits(Q, g, c.H)) return g;
  return g;
}

__device__ __forceinline__ int block_max(int v, int *sh) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = l < (kThreads / 32) ? sh[l] : INT_MIN;
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ unsigned long long block_sum(unsigned long long v,
                                                        unsigned long long *sh) {
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = l < (kThreads / 32) ? sh[l] : 0ull;
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ void set_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

// 12-bit words of trunc(mant * 2^sh) (< 2^84), negated for negative inputs.
__device__ __forceinline__ void int_words(const Dec &d, int sh, float (&w)[7]) {
  uint64_t lo, hi;
  if (d.mant == 0) {
    lo = hi = 0;
  } else if (sh >= 0) {
    if (sh == 0) { lo = d.mant; hi = 0; }
    else if (sh < 64) { lo = d.mant << sh; hi = d.mant >> (64 - sh); }
    else { lo = 0; hi = d.mant << (sh - 64); }
  } else {
    int r = -sh;
    lo = r >= 64 ? 0 : (d.mant >> r);
    hi = 0;
  }
  uint32_t u[7];
  u[0] = (uint32_t)(lo & 0xFFF);
  u[1] = (uint32_t)((lo >> 12) & 0xFFF);
  u[2] = (uint32_t)((lo >> 24) & 0xFFF);
  u[3] = (uint32_t)((lo >> 36) & 0xFFF);
  u[4] = (uint32_t)((lo >> 48) & 0xFFF);
  u[5] = (uint32_t)(((lo >> 60) | (hi << 4)) & 0xFFF);
  u[6] = (uint32_t)((hi >> 8) & 0xFFF);
#pragma unroll
  for (int t = 0; t < 7; t++) w[t] = d.neg ? -(float)u[t] : (float)u[t];
}

// Symmetric residue of sum_t w_t 2^(12t) modulo p_l.  Every partial sum is an
// integer below 7 * 4095 * 128 < 2^24, so the FP32 chain is exact; the
// rounded quotient is off by at most one, fixed by one step each way.
__device__ __forceinline__ float residue(const float (&w)[7], const ResConsts &c, int l) {
  float x = w[0] * c.w12[l][0];
#pragma unroll
  for (int t = 1; t < 7; t++) x = fmaf(w[t], c.w12[l][t], x);
  float q = rintf(x * c.invp[l]);
  float r = fmaf(-c.p[l], q, x);
  r = r > c.hi[l] ? r - c.p[l] : r;
  r = r < c.lo[l] ? r + c.p[l] : r;
  return r;
}

template <int N, int MODE>
__global__ void __launch_bounds__(kThreads)
    k_scale_residue(const double *__restrict__ X, long ldx, int rows, int k, int kp,
                    int32_t *__restrict__ e, int32_t *__restrict__ Eout,
                    __half *__restrict__ planes, const ResConsts c, int *status) {
  __shared__ int s_int[32];
  __shared__ unsigned long long s_u64[32];
  __shared__ int s_e;
  const int row = blockIdx.x;
  const double *x = X + (size_t)row * ldx;
  int ee = 0;

  if (MODE != SM_RESIDUES) {
    int emax = INT_MIN, bad = 0;
    for (int h = threadIdx.x; h < k; h += kThreads) {
      Dec d = decode(__ldg(x + h));
      bad |= d.nonfinite;
      emax = max(emax, exp_bound(d));
    }
    emax = block_max(emax, s_int);
    bad = block_max(bad, s_int);
    if (bad && threadIdx.x == 0) set_status(status, OS2_ERR_NONFINITE);
    const bool nonzero = emax != INT_MIN;
    const int E = nonzero ? emax : 0;

    if (MODE == SM_BARS) {
      // accurate mode: E_i and Abar_ih = ceil(|a_ih| 2^(6 - E_i)) in [0, 64]
      if (threadIdx.x == 0) Eout[row] = E;
      __half *dst = planes + (size_t)row * kp;
      for (int ch = threadIdx.x; ch < kp / 8; ch += kThreads) {
        int h0 = ch * 8;
        __align__(16) __half v[8];
#pragma unroll
        for (int u = 0; u < 8; u++) {
          int h = h0 + u;
          Dec d = decode(h < k ? __ldg(x + h) : 0.0);
          v[u] = __float2half_rn((float)ceil_shift(d.mant, d.ex2 + 6 - E));
        }
        *reinterpret_cast<uint4 *>(dst + h0) = *reinterpret_cast<uint4 *>(v);
      }
      return;
    }

    unsigned long long Q = 0;
    for (int h = threadIdx.x; h < k; h += kThreads) {
      Dec d = decode(__ldg(x + h));
      unsigned long long q = ceil_shift(d.mant, d.ex2 + 23 - E);
      Q += q * q;
    }
    Q = block_sum(Q, s_u64);
    if (threadIdx.x == 0) {
      int v = (nonzero && !bad && Q) ? largest_g(Q, c) + 23 - E : 0;
      e[row] = v;
      s_e = v;
    }
    __syncthreads();
    ee = s_e;
    if (MODE == SM_FAST_SCALE) return;
  } else {
    ee = e[row];
  }

  // residue planes: plane l, row `row`, columns [h0, h0 + 8) per thread
  for (int ch = threadIdx.x; ch < kp / 8; ch += kThreads) {
    const int h0 = ch * 8;
    float w[8][7];
#pragma unroll
    for (int u = 0; u < 8; u++) {
      int h = h0 + u;
      Dec d = decode(h < k ? __ldg(x + h) : 0.0);
      int_words(d, d.ex2 + ee, w[u]);
    }
#pragma unroll
    for (int l = 0; l < N; l++) {
      __align__(16) __half2 v[4];
#pragma unroll
      for (int u = 0; u < 4; u++)
        v[u] = __floats2half2_rn(residue(w[2 * u], c, l), residue(w[2 * u + 1], c, l));
      *reinterpret_cast<uint4 *>(planes + ((size_t)l * rows + row) * kp + h0) =
          *reinterpret_cast<uint4 *>(v);
    }
  }
}

__global__ void k_accu_exponents(const int32_t *__restrict__ bound, const int32_t *__restrict__ E,
                                 int rows, int32_t *__restrict__ e, const ResConsts c) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows) return;
  int R = bound[i];
  e[i] = R > 0 ? largest_g((uint64_t)R, c) + 6 - E[i] : -E[i];
}

template <int MODE>
cudaError_t dispatch(int N, dim3 grid, cudaStream_t s, const double *X, long ldx, int rows, int k,
                     int kp, int32_t *e, int32_t *E, __half *planes, const ResConsts &c,
                     int *status) {
#define OS2_CASE(NN)                                                                          \
  case NN:                                                                                    \
    k_scale_residue<NN, MODE><<<grid, kThreads, 0, s>>>(X, ldx, rows, k, kp, e, E, planes, c, \
                                                        status);                              \
    break;
  switch (N) {
    OS2_CASE(1) OS2_CASE(2) OS2_CASE(3) OS2_CASE(4) OS2_CASE(5) OS2_CASE(6) OS2_CASE(7)
    OS2_CASE(8) OS2_CASE(9) OS2_CASE(10) OS2_CASE(11) OS2_CASE(12) OS2_CASE(13) OS2_CASE(14)
    OS2_CASE(15) OS2_CASE(16) OS2_CASE(17) OS2_CASE(18) OS2_CASE(19) OS2_CASE(20)
    default: return cudaErrorInvalidValue;
  }
#undef OS2_CASE
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_scale_residue(int mode, const double *X, long ldx, int rows, int k, int kp,
                                 int32_t *e, int32_t *E, void *planes, const Os2Tables *t,
                                 int *status, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  dim3 grid(rows);
  __half *pl = reinterpret_cast<__half *>(planes);
  switch (mode) {
    case SM_FAST_FUSED:
      return dispatch<SM_FAST_FUSED>(t->N, grid, s, X, ldx, rows, k, kp, e, E, pl, t->res, status);
    case SM_RESIDUES:
      return dispatch<SM_RESIDUES>(t->N, grid, s, X, ldx, rows, k, kp, e, E, pl, t->res, status);
    case SM_FAST_SCALE:
      k_scale_residue<1, SM_FAST_SCALE>
          <<<grid, kThreads, 0, s>>>(X, ldx, rows, k, kp, e, E, pl, t->res, status);
      return cudaGetLastError();
    case SM_BARS:
      k_scale_residue<1, SM_BARS>
          <<<grid, kThreads, 0, s>>>(X, ldx, rows, k, kp, e, E, pl, t->res, status);
      return cudaGetLastError();
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_accu_exponents(const int32_t *bound, const int32_t *E, int rows, int32_t *e,
                                  const Os2Tables *t, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_accu_exponents<<<(rows + 255) / 256, 256, 0, s>>>(bound, E, rows, e, t->res);
  return cudaGetLastError();
}
