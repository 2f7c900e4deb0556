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
// Two kernels, each launched once for both operands (A's rows, then B's
// columns):
//   k_row_scale  one CTA per row: exponent bound (pass 1), then either the
//                fast-mode sum of squares and e_i, or the accurate-mode
//                7-bit magnitude plane (pass 2 re-reads the row from L1/L2).
//   k_residues   element-parallel residue planes (k_residues.cuh; its
//                instances live in k_residues_{d,f}{1,2,3,4}.cu).  This file
//                holds the launcher that picks the instance.
#include <cuda_fp16.h>
#include <limits.h>

#include <type_traits>

#include "k_residues.cuh"

namespace {

using os2dev::Dec;
using os2dev::decode;
using os2dev::load2;
using os2dev::RowSet;
using os2dev::set_status;

// Row scale kernel: one CTA of NT threads per row, NT = 256, 512 or 1024 as k
// grows (see launch_row_scale).

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
__device__ bool fits(uint64_t Qlo, uint64_t Qhi, int g, const uint32_t *H) {
  uint32_t q4[4] = {(uint32_t)Qlo, (uint32_t)(Qlo >> 32), (uint32_t)Qhi, (uint32_t)(Qhi >> 32)};
  uint32_t L[8], R[8];
  shl8(q4, 4, g > 0 ? 2 * g : 0, L);
  shl8(H, OS2_H_LIMBS, g < 0 ? -2 * g : 0, R);
  for (int i = 7; i >= 0; i--)
    if (L[i] != R[i]) return L[i] < R[i];
  return true;
}
// Largest integer g with Q * 4^g <= H, Q = Qhi 2^64 + Qlo >= 1.  With b(.)
// the bit length and g0 = floor((b(H) + 1 - b(Q)) / 2), Q 4^g0 has b(H) + 1
// bits (then g0 - 1 is the answer) or b(H) bits; in the second case the 64
// leading bits of Q and of H decide, unless they are equal and both have set
// bits below them (then the full comparison does).
__device__ int largest_g(uint64_t Qlo, uint64_t Qhi, const ResConsts &c) {
  const int bQ = Qhi ? 128 - __clzll((long long)Qhi) : 64 - __clzll((long long)Qlo);
  const int g = (c.bitlenH + 1 - bQ) >> 1;
  if (bQ + 2 * g > c.bitlenH) return g - 1;
  uint64_t w;
  bool rest;
  if (bQ <= 64) {
    w = Qlo << (64 - bQ);
    rest = false;
  } else {
    const int s = bQ - 64;  // 1..64
    w = s == 64 ? Qhi : (Qhi << (64 - s)) | (Qlo >> s);
    rest = s == 64 ? Qlo != 0 : (Qlo & ((1ull << s) - 1)) != 0;
  }
  if (w != c.H64) return w < c.H64 ? g : g - 1;
  if (!rest) return g;
  if (!c.Hrest) return g - 1;
  return fits(Qlo, Qhi, g, c.H) ? g : g - 1;
}

template <int NT>
__device__ __forceinline__ int block_max(int v, int *sh) {
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) sh[w] = v;
  __syncthreads();
  v = l < (NT / 32) ? sh[l] : INT_MIN;
  for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
// 128-bit block sum of per-thread 64-bit partials (hi:lo).
__device__ __forceinline__ void add128(unsigned long long &lo, unsigned long long &hi,
                                       unsigned long long blo, unsigned long long bhi) {
  const unsigned long long s = lo + blo;
  hi += bhi + (s < lo ? 1ull : 0ull);
  lo = s;
}
template <int NT>
__device__ __forceinline__ void block_sum128(unsigned long long &lo, unsigned long long &hi,
                                             unsigned long long *sh) {
  for (int o = 16; o; o >>= 1)
    add128(lo, hi, __shfl_xor_sync(0xffffffffu, lo, o), __shfl_xor_sync(0xffffffffu, hi, o));
  int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    sh[2 * w] = lo;
    sh[2 * w + 1] = hi;
  }
  __syncthreads();
  lo = l < (NT / 32) ? sh[2 * l] : 0ull;
  hi = l < (NT / 32) ? sh[2 * l + 1] : 0ull;
  for (int o = 16; o; o >>= 1)
    add128(lo, hi, __shfl_xor_sync(0xffffffffu, lo, o), __shfl_xor_sync(0xffffffffu, hi, o));
}

// ------------------------------------------------------------- row scale ---
// Monotone integer keys of |x| and the ceilings of steps 1 and 1A for rows
// that hold at least one normal number and no Inf or NaN (every other row
// takes the exact decode above).  key(x) = the high word of |x|'s bits, whose
// maximum over a row gives the row's largest exponent field, so
// E = (key >> kMantHi) - kEBias is the tight bound |x| < 2^E.
template <typename T> struct FBits;
template <> struct FBits<double> {
  static constexpr uint32_t kInfKey = 0x7FF00000u, kNormKey = 0x00100000u;
  static constexpr int kMantHi = 20, kEBias = 1022;
  static __device__ __forceinline__ uint32_t key(double x) {
    return (uint32_t)__double2hiint(x) & 0x7FFFFFFFu;
  }
  // ceil(|x| 2^(S - E)) for finite x with |x| < 2^E and E >= -1021: the
  // significand m shifted right by r = E - S - ex2 >= 30 (S <= 23), taken as
  // ((m - 1) >> r) + 1.
  template <int S>
  static __device__ __forceinline__ uint32_t ceil_scaled(double x, int E) {
    const uint32_t hi = (uint32_t)__double2hiint(x), lo = (uint32_t)__double2loint(x);
    const uint32_t bexp = (hi >> 20) & 0x7FFu;
    const uint32_t mh = (hi & 0xFFFFFu) | (bexp ? 0x100000u : 0u);
    if ((mh | lo) == 0u) return 0u;
    const int r = E - S + 1075 - (int)max(bexp, 1u);
    const uint32_t mlo = lo - 1u, mhi = mh - (lo == 0u ? 1u : 0u);
    const uint32_t t = r < 32 ? __funnelshift_rc(mlo, mhi, (unsigned)r)
                              : __funnelshift_rc(mhi, 0u, (unsigned)(r - 32));
    return t + 1u;
  }
};
template <> struct FBits<float> {
  static constexpr uint32_t kInfKey = 0x7F800000u, kNormKey = 0x00800000u;
  static constexpr int kMantHi = 23, kEBias = 126;
  static __device__ __forceinline__ uint32_t key(float x) {
    return __float_as_uint(x) & 0x7FFFFFFFu;
  }
  template <int S>
  static __device__ __forceinline__ uint32_t ceil_scaled(float x, int E) {
    const uint32_t b = __float_as_uint(x);
    const uint32_t bexp = (b >> 23) & 0xFFu;
    const uint32_t m = (b & 0x7FFFFFu) | (bexp ? 0x800000u : 0u);
    if (m == 0u) return 0u;
    const int r = E - S + 150 - (int)max(bexp, 1u);  // >= 1 for S <= 23
    return __funnelshift_rc(m - 1u, 0u, (unsigned)r) + 1u;
  }
};

// Calls f on each of the thread's entries of a row (strided by the CTA),
// with U two-entry vector loads in flight before the first use.  Entries past
// k are passed as zero.
template <int NT, typename T, typename F>
__device__ __forceinline__ void for_row(const T *x, int k, bool vec, F &&f) {
  if (vec) {
    constexpr int U = 4;
    for (int h0 = 2 * threadIdx.x; h0 < k; h0 += 2 * NT * U) {
      T v[2 * U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int h = h0 + u * 2 * NT;
        if (h + 1 < k) {
          load2(x + h, v[2 * u], v[2 * u + 1]);
        } else {
          v[2 * u] = h < k ? __ldg(x + h) : T(0);
          v[2 * u + 1] = T(0);
        }
      }
#pragma unroll
      for (int i = 0; i < 2 * U; i++) f(v[i]);
    }
  } else {
    for (int h = threadIdx.x; h < k; h += NT) f(__ldg(x + h));
  }
}

template <int MODE, typename T, int NT>
__global__ void __launch_bounds__(NT, 2048 / NT)
    k_row_scale(const RowSet a, const RowSet b, int k, int kp, const ResConsts c, int *status) {
  __shared__ int s_int[32];
  __shared__ unsigned long long s_u64[2 * 32];
  const bool isA = (int)blockIdx.x < a.rows;
  const RowSet &rs = isA ? a : b;
  const int row = isA ? (int)blockIdx.x : (int)blockIdx.x - a.rows;
  const T *x = reinterpret_cast<const T *>(rs.X) + (size_t)row * rs.ldx;
  const bool vec = ((reinterpret_cast<uintptr_t>(x) & (2 * sizeof(T) - 1)) == 0);
  if (!OS2_DBG_GUARD(row < rs.rows && k <= rs.ldx && (MODE != SM_BARS || k <= kp), status))
    return;  // (uniform over the CTA)

  // pass 1: the largest key of the row.  For doubles only the high words are
  // loaded, sixteen 4-byte loads per thread in flight: the same DRAM sectors
  // as full loads, but twice the entries per register.
  uint32_t key = 0;
  if (sizeof(T) == 8) {
    constexpr int U = 16;
    const uint32_t *xh = reinterpret_cast<const uint32_t *>(x) + 1;
    for (int h0 = threadIdx.x; h0 < k; h0 += NT * U) {
      uint32_t hv[U];
#pragma unroll
      for (int u = 0; u < U; u++) {
        const int h = h0 + u * NT;
        hv[u] = h < k ? __ldg(xh + 2 * (size_t)h) : 0u;
      }
#pragma unroll
      for (int u = 0; u < U; u++) key = max(key, hv[u] & 0x7FFFFFFFu);
    }
  } else {
    for_row<NT>(x, k, vec, [&](T v) { key = max(key, FBits<T>::key(v)); });
  }
  key = (uint32_t)block_max<NT>((int)key, s_int);
  const bool general = key >= FBits<T>::kInfKey || key < FBits<T>::kNormKey;
  int E, bad = 0;
  bool nonzero = true;
  if (!general) {
    E = (int)(key >> FBits<T>::kMantHi) - FBits<T>::kEBias;
  } else {
    // Inf or NaN present, or no normal number: exponent bound and finiteness
    // entry by entry
    int emax = INT_MIN;
    for_row<NT>(x, k, vec, [&](T v) {
      const Dec d = decode(v);
      bad |= d.nonfinite;
      emax = max(emax, exp_bound(d));
    });
    emax = block_max<NT>(emax, s_int);
    bad = block_max<NT>(bad, s_int);
    if (bad && threadIdx.x == 0) set_status(status, OS2_ERR_NONFINITE);
    nonzero = emax != INT_MIN;
    E = nonzero ? emax : 0;
  }

  if (MODE == SM_BARS) {
    // accurate mode: E_i and Abar_ih = ceil(|a_ih| 2^(6 - E_i)) in [0, 64]
    if (threadIdx.x == 0) rs.E[row] = E;
    __half *dst = rs.planes + (size_t)row * kp;
    for (int ch = threadIdx.x; ch < kp / 8; ch += NT) {
      const int h0 = ch * 8;
      T xv[8];
      if (vec && h0 + 8 <= k) {
#pragma unroll
        for (int u = 0; u < 4; u++) load2(x + h0 + 2 * u, xv[2 * u], xv[2 * u + 1]);
      } else {
#pragma unroll
        for (int u = 0; u < 8; u++) xv[u] = h0 + u < k ? __ldg(x + h0 + u) : T(0);
      }
      __align__(16) __half v[8];
      if (!general) {
#pragma unroll
        for (int u = 0; u < 8; u++)
          v[u] = __float2half_rn((float)FBits<T>::template ceil_scaled<6>(xv[u], E));
      } else {
#pragma unroll
        for (int u = 0; u < 8; u++) {
          const Dec d = decode(xv[u]);
          v[u] = __float2half_rn((float)ceil_shift(d.mant, d.ex2 + 6 - E));
        }
      }
      if (OS2_DBG_GUARD(h0 + 8 <= kp, status))
        *reinterpret_cast<uint4 *>(dst + h0) = *reinterpret_cast<uint4 *>(v);
    }
    return;
  }

  // pass 2 (fast mode): exact sum of squares of the 23-bit upper roundings
  // (each q^2 <= 2^46; a thread's partial stays below 2^64 for k < 2^26;
  // the block sum is 128-bit)
  unsigned long long Q = 0, Qhi = 0;
  if (!general) {
    for_row<NT>(x, k, vec, [&](T v) {
      const uint32_t q = FBits<T>::template ceil_scaled<23>(v, E);
      Q += (unsigned long long)q * q;
    });
  } else {
    for_row<NT>(x, k, vec, [&](T v) {
      const Dec d = decode(v);
      const unsigned long long q = ceil_shift(d.mant, d.ex2 + 23 - E);
      Q += q * q;
    });
  }
  block_sum128<NT>(Q, Qhi, s_u64);
  if (threadIdx.x == 0)
    rs.e[row] = (nonzero && !bad && (Q | Qhi)) ? largest_g(Q, Qhi, c) + 23 - E : 0;
}

__global__ void k_accu_exponents(const int32_t *__restrict__ bound, const int32_t *__restrict__ E,
                                 int rows, int32_t *__restrict__ e, const ResConsts c) {
  int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= rows) return;
  int R = bound[i];
  e[i] = R > 0 ? largest_g((uint64_t)R, 0ull, c) + 6 - E[i] : -E[i];
}

}  // namespace

cudaError_t launch_row_scale(int mode, bool f32, const void *XA, long lda, int rowsA,
                             int32_t *eA, int32_t *EA, void *barsA, const void *XB, long ldb,
                             int rowsB, int32_t *eB, int32_t *EB, void *barsB, int k, int kp,
                             const Os2Tables *t, int *status, cudaStream_t s) {
  if (rowsA + rowsB <= 0) return cudaSuccess;
  RowSet a{XA, lda, rowsA, eA, EA, reinterpret_cast<__half *>(barsA), rowsA};
  RowSet b{XB, ldb, rowsB, eB, EB, reinterpret_cast<__half *>(barsB), rowsB};
  dim3 grid(rowsA + rowsB);
  // About 32 entries per thread: the rows in flight (2048 threads per SM) then
  // hold about 80 MB of doubles whatever k is, so the second pass over each
  // row still finds it in L2.
  const int nt = k > 16384 ? 1024 : (k > 8192 ? 512 : 256);
#define OS2_SCALE(M, T)                                                                    \
  (nt == 1024  ? (k_row_scale<M, T, 1024><<<grid, 1024, 0, s>>>(a, b, k, kp, t->res, status), 0) \
   : nt == 512 ? (k_row_scale<M, T, 512><<<grid, 512, 0, s>>>(a, b, k, kp, t->res, status), 0)   \
               : (k_row_scale<M, T, 256><<<grid, 256, 0, s>>>(a, b, k, kp, t->res, status), 0))
  if (mode == SM_BARS) {
    if (f32) OS2_SCALE(SM_BARS, float);
    else OS2_SCALE(SM_BARS, double);
  } else {
    if (f32) OS2_SCALE(SM_FAST_SCALE, float);
    else OS2_SCALE(SM_FAST_SCALE, double);
  }
#undef OS2_SCALE
  return cudaGetLastError();
}

cudaError_t launch_residues(bool f32, const void *XA, long lda, int rowsA, const int32_t *eA,
                            void *planesA, const void *XB, long ldb, int rowsB,
                            const int32_t *eB, void *planesB, int k, int kp, const Os2Tables *t,
                            cudaStream_t s, long prowB, bool i8) {
  if (rowsA + rowsB <= 0 || kp <= 0) return cudaSuccess;
  RowSet a{XA, lda, rowsA, const_cast<int32_t *>(eA), nullptr, reinterpret_cast<__half *>(planesA),
           rowsA};
  RowSet b{XB, ldb, rowsB, const_cast<int32_t *>(eB), nullptr, reinterpret_cast<__half *>(planesB),
           prowB > 0 ? prowB : rowsB};
  int *status = os2_status_ptr();
  const int N = t->N;
  if (N < 1 || N > OS2_MAX_MODULI) return cudaErrorInvalidValue;
  using namespace os2dev;
  const ResConsts &c = t->res;
  if (f32) {
    if (N <= 12) return residues_f1(N, a, b, k, kp, c, status, s, i8);
    if (N <= 16) return residues_f2(N, a, b, k, kp, c, status, s, i8);
    if (N <= 18) return residues_f3(N, a, b, k, kp, c, status, s, i8);
    return residues_f4(N, a, b, k, kp, c, status, s, i8);
  }
  if (N <= 12) return residues_d1(N, a, b, k, kp, c, status, s, i8);
  if (N <= 16) return residues_d2(N, a, b, k, kp, c, status, s, i8);
  if (N <= 18) return residues_d3(N, a, b, k, kp, c, status, s, i8);
  return residues_d4(N, a, b, k, kp, c, status, s, i8);
}

cudaError_t launch_accu_exponents(const int32_t *bound, const int32_t *E, int rows, int32_t *e,
                                  const Os2Tables *t, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_accu_exponents<<<(rows + 255) / 256, 256, 0, s>>>(bound, E, rows, e, t->res);
  return cudaGetLastError();
}
