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
//   k_residues   element-parallel: every thread turns 8 consecutive entries
//                into 8 residues per modulus and writes one 16-byte vector to
//                each plane.  Residues of the odd moduli use FP32 arithmetic
//                only: the integer is split into four to six 15-bit words w_t
//                (as many as its size needs) and x = K + sum_t w_t (2^(15t)
//                mod p) is exact below 2^23, so one fused multiply-add rounds
//                x / p to the nearest integer exactly.  Two entries share each
//                packed FP32 instruction.  Mod 256 is the integer's low byte.
#include <cuda_fp16.h>
#include <limits.h>

#include <type_traits>

#include "os2_internal.cuh"

namespace {

constexpr int kThreads = 256;       // residue kernel
// Row scale kernel: one CTA of NT threads per row, NT = 256, 512 or 1024 as k
// grows (see launch_row_scale).

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

__device__ __forceinline__ Dec decode(float x) {
  const uint32_t b = __float_as_uint(x);
  int bexp = (int)((b >> 23) & 0xFF);
  Dec d;
  d.neg = b >> 31;
  d.nonfinite = bexp == 0xFF;
  d.mant = b & 0x7FFFFFu;
  if (bexp) d.mant |= 1ull << 23;
  else bexp = 1;
  d.ex2 = bexp - 150;
  if (d.nonfinite) d.mant = 0;
  return d;
}

// Two consecutive entries through one vector load (aligned to 2 * sizeof(T)).
__device__ __forceinline__ void load2(const double *p, double &a, double &b) {
  const double2 v = __ldg(reinterpret_cast<const double2 *>(p));
  a = v.x;
  b = v.y;
}
__device__ __forceinline__ void load2(const float *p, float &a, float &b) {
  const float2 v = __ldg(reinterpret_cast<const float2 *>(p));
  a = v.x;
  b = v.y;
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

__device__ __forceinline__ void set_status(int *status, int code) {
  if (status) atomicCAS(status, 0, code);
}

struct RowSet {
  const void *X;    // double or float entries, row-major
  long ldx;
  int rows;
  int32_t *e;       // exponents (out for scale, in for residues)
  int32_t *E;       // accurate mode: exponent bounds (out)
  __half *planes;   // residue planes [N][prow][kp] (first `rows` rows written) or the
                    // magnitude plane [rows][kp]
  long prow;        // rows from one residue plane to the next (>= rows)
};

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

// --------------------------------------------------------------- residues --
__device__ __forceinline__ float byte_residue(uint32_t b) {
  return (float)((int)(b ^ 0x80u) - 128);  // [-128, 127]
}

// Words of the scaled integer.  trunc(mant * 2^sh), of magnitude below
// 2^(15 NW - 1), is taken in two's complement and cut into NW fields of 15 bits,
// the top one signed.  Each field is shifted down by 2^14 into [-2^14, 2^14)
// and held exactly as a float (2^23 + v from the bit pattern, minus
// 2^23 + 2^14), so the integer is
//   sum_t w_t 2^(15t) + 2^14 (1 + 2^15 + ... + 2^(15 (NW - 2))).
// lowbyte: the integer's low byte, its residue mod 256.
template <int NW>
__device__ __forceinline__ void int_words(const Dec &d, int sh, float (&w)[NW],
                                          uint32_t &lowbyte) {
  static_assert(NW >= 4 && NW <= 6, "four to six words");
  uint32_t v[NW];
  if (NW == 4) {
    uint64_t mag;
    if (sh >= 64) mag = 0;  // only for mant == 0: a nonzero entry has sh <= 58
    else if (sh >= 0) mag = d.mant << sh;
    else mag = -sh >= 64 ? 0 : d.mant >> -sh;
    const uint64_t t = d.neg ? 0ull - mag : mag;
    v[0] = (uint32_t)t & 0x7FFFu;
    v[1] = (uint32_t)(t >> 15) & 0x7FFFu;
    v[2] = (uint32_t)(t >> 30) & 0x7FFFu;
    v[3] = (uint32_t)(t >> 45) & 0x7FFFu;
    lowbyte = (uint32_t)t & 0xFFu;
  } else {
    uint64_t lo, hi;  // |integer| < 2^89: a nonzero entry has sh <= 88
    if (d.mant == 0 || sh <= -64) { lo = 0; hi = 0; }
    else if (sh >= 64) { lo = 0; hi = d.mant << (sh - 64); }
    else if (sh > 0) { lo = d.mant << sh; hi = d.mant >> (64 - sh); }
    else { lo = d.mant >> -sh; hi = 0; }
    if (d.neg) {
      hi = ~hi + (lo == 0 ? 1ull : 0ull);
      lo = 0ull - lo;
    }
    v[0] = (uint32_t)lo & 0x7FFFu;
    v[1] = (uint32_t)(lo >> 15) & 0x7FFFu;
    v[2] = (uint32_t)(lo >> 30) & 0x7FFFu;
    v[3] = (uint32_t)(lo >> 45) & 0x7FFFu;
    v[4] = (uint32_t)((lo >> 60) | (hi << 4)) & 0x7FFFu;
    if (NW == 6) v[NW - 1] = (uint32_t)(hi >> 11) & 0x7FFFu;
    lowbyte = (uint32_t)lo & 0xFFu;
  }
  v[NW - 1] ^= 0x4000u;  // signed top field + 2^14
#pragma unroll
  for (int t = 0; t < NW; t++) w[t] = __uint_as_float(0x4B000000u | v[t]) - 8404992.0f;
}

// Pairs of FP32 values in one 64-bit register: the packed FP32 instructions of
// sm_100 and later do two FMAs (or adds) per lane and issue slot.
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(unsigned long long v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long fma2(unsigned long long a, unsigned long long b,
                                                   unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ unsigned long long add2(unsigned long long a, unsigned long long b) {
  unsigned long long d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Residues of EPT entries (held as int_words gives them) for every modulus,
// one vector store of EPT FP16 values per plane.  For odd p_l, with
// c_t = 2^(15t) mod p_l and K = 2^14 (c_0 + ... + c_(NW-2)) mod p_l, both held
// around zero: x = K + sum_t w_t c_t is congruent to the integer, and for the
// twenty moduli of the set and NW <= 6, |x| <= 2^14 sum_t |c_t| + |K| <
// 6.8e6 < 2^23.  So every partial sum is exact, x * fl(1/p_l) lies within
// 1/(2 p_l) of x/p_l, which is at least 1/(2 p_l) from any half-integer, and
// adding 1.5 * 2^23 in the same FMA rounds it to round(x/p_l) exactly:
// x - p_l round(x/p_l) is the canonical residue, with no fix-up.  Two entries
// go through each packed instruction.
template <int N, int NW, int EPT>
__device__ __forceinline__ void emit(const float (&w)[EPT][NW], const uint32_t (&lb)[EPT],
                                     const ResConsts &c, __half *dst, size_t pstride) {
  static_assert(EPT == 4 || EPT == 8, "4 or 8 entries per thread");
  using Vec = typename std::conditional<EPT == 8, uint4, uint2>::type;
  {
    __align__(16) __half2 v[EPT / 2];
#pragma unroll
    for (int u = 0; u < EPT / 2; u++)
      v[u] = __floats2half2_rn(byte_residue(lb[2 * u]), byte_residue(lb[2 * u + 1]));
    *reinterpret_cast<Vec *>(dst) = *reinterpret_cast<Vec *>(v);
  }
  unsigned long long W[EPT / 2][NW];
#pragma unroll
  for (int u = 0; u < EPT / 2; u++)
#pragma unroll
    for (int t = 0; t < NW; t++) W[u][t] = pack2(w[2 * u][t], w[2 * u + 1][t]);
  constexpr unsigned long long kMagic2 = 0x4B4000004B400000ull;     // 1.5 * 2^23, twice
  constexpr unsigned long long kNegMagic2 = 0xCB400000CB400000ull;  // -1.5 * 2^23, twice
#pragma unroll
  for (int l = 1; l < N; l++) {
    __align__(16) __half2 v[EPT / 2];
#pragma unroll
    for (int u = 0; u < EPT / 2; u++) {
      unsigned long long x = fma2(W[u][0], c.w15x2[l][0], c.k15x2[l][NW - 4]);
#pragma unroll
      for (int t = 1; t < NW; t++) x = fma2(W[u][t], c.w15x2[l][t], x);
      const unsigned long long q = add2(fma2(x, c.invp2[l], kMagic2), kNegMagic2);
      float r0, r1;
      unpack2(fma2(c.negp2[l], q, x), r0, r1);
      v[u] = __floats2half2_rn(r0, r1);
    }
    *reinterpret_cast<Vec *>(dst + l * pstride) = *reinterpret_cast<Vec *>(v);
  }
}

template <int N, int NW, typename T, int EPT>
__device__ __forceinline__ void residues_of(const T (&v)[EPT], int ee, const ResConsts &c,
                                            __half *dst, size_t pstride) {
  float w[EPT][NW];
  uint32_t lb[EPT];
#pragma unroll
  for (int u = 0; u < EPT; u++) {
    const Dec d = decode(v[u]);
    int_words<NW>(d, d.ex2 + ee, w[u], lb[u]);
  }
  emit<N, NW, EPT>(w, lb, c, dst, pstride);
}

// Residue planes: EPT consecutive entries per thread, one vector store per plane.
constexpr int kEPT = 8;

template <int N, typename T>
__global__ void __launch_bounds__(kThreads, 3)
    k_residues(const RowSet a, const RowSet b, int k, int kp, const ResConsts c, int *status) {
  constexpr int EPT = kEPT;
  const int cpr = kp / EPT;  // chunks per row
  const int total_rows = a.rows + b.rows;
  for (int rr = blockIdx.y; rr < total_rows; rr += gridDim.y) {
    const bool isA = rr < a.rows;
    const RowSet &rs = isA ? a : b;
    const int row = isA ? rr : rr - a.rows;
    const T *x = reinterpret_cast<const T *>(rs.X) + (size_t)row * rs.ldx;
    const int ee = __ldg(rs.e + row);
    const size_t pstride = (size_t)rs.prow * kp;
    const bool vec = ((reinterpret_cast<uintptr_t>(x) & (2 * sizeof(T) - 1)) == 0);
    for (int ch = blockIdx.x * kThreads + threadIdx.x; ch < cpr; ch += gridDim.x * kThreads) {
      const int h0 = ch * EPT;
      T v[EPT];
      if (vec && h0 + EPT <= k) {
#pragma unroll
        for (int u = 0; u < EPT / 2; u++) load2(x + h0 + 2 * u, v[2 * u], v[2 * u + 1]);
      } else {
#pragma unroll
        for (int u = 0; u < EPT; u++) v[u] = h0 + u < k ? __ldg(x + h0 + u) : T(0);
      }
      // bit length bound of the integers (row exponent + element exponent)
      int top = INT_MIN;
#pragma unroll
      for (int u = 0; u < EPT; u++) {
        const Dec d = decode(v[u]);
        if (d.mant) top = max(top, d.ex2 + 64 - __clzll((long long)d.mant) + ee);
      }
      __half *dst = rs.planes + (size_t)row * kp + h0;
      if (top <= 59) {
        residues_of<N, 4>(v, ee, c, dst, pstride);
      } else if (top <= 74) {
        residues_of<N, 5>(v, ee, c, dst, pstride);
      } else if (top <= 89) {
        residues_of<N, 6>(v, ee, c, dst, pstride);
      } else {
        // beyond every exponent that step 1 produces (|integer| < 2^84):
        // reported, and the entries' residues are left as zero
        set_status(status, OS2_ERR_RANGE);
#pragma unroll
        for (int l = 0; l < N; l++)
#pragma unroll
          for (int u = 0; u < EPT; u++) dst[l * pstride + u] = __float2half(0.0f);
      }
    }
  }
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

template <typename T>
cudaError_t residues_t(const RowSet &a, const RowSet &b, int k, int kp, const Os2Tables *t,
                       int *status, cudaStream_t s) {
  const int cpr = kp / kEPT;
  const int bx = (cpr + kThreads - 1) / kThreads;
  const int rows = a.rows + b.rows;
  dim3 grid(bx, rows < 65535 ? rows : 65535);
#define OS2_CASE(NN)                                                         \
  case NN:                                                                   \
    k_residues<NN, T><<<grid, kThreads, 0, s>>>(a, b, k, kp, t->res, status);  \
    break;
  switch (t->N) {
    OS2_CASE(1) OS2_CASE(2) OS2_CASE(3) OS2_CASE(4) OS2_CASE(5) OS2_CASE(6) OS2_CASE(7)
    OS2_CASE(8) OS2_CASE(9) OS2_CASE(10) OS2_CASE(11) OS2_CASE(12) OS2_CASE(13) OS2_CASE(14)
    OS2_CASE(15) OS2_CASE(16) OS2_CASE(17) OS2_CASE(18) OS2_CASE(19) OS2_CASE(20)
    default: return cudaErrorInvalidValue;
  }
#undef OS2_CASE
  return cudaGetLastError();
}

cudaError_t launch_residues(bool f32, const void *XA, long lda, int rowsA, const int32_t *eA,
                            void *planesA, const void *XB, long ldb, int rowsB,
                            const int32_t *eB, void *planesB, int k, int kp, const Os2Tables *t,
                            cudaStream_t s, long prowB) {
  if (rowsA + rowsB <= 0 || kp <= 0) return cudaSuccess;
  RowSet a{XA, lda, rowsA, const_cast<int32_t *>(eA), nullptr, reinterpret_cast<__half *>(planesA),
           rowsA};
  RowSet b{XB, ldb, rowsB, const_cast<int32_t *>(eB), nullptr, reinterpret_cast<__half *>(planesB),
           prowB > 0 ? prowB : rowsB};
  int *status = os2_status_ptr();
  return f32 ? residues_t<float>(a, b, k, kp, t, status, s)
             : residues_t<double>(a, b, k, kp, t, status, s);
}

cudaError_t launch_accu_exponents(const int32_t *bound, const int32_t *E, int rows, int32_t *e,
                                  const Os2Tables *t, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  k_accu_exponents<<<(rows + 255) / 256, 256, 0, s>>>(bound, E, rows, e, t->res);
  return cudaGetLastError();
}
