// Rounding of a multi-limb integer times a power of two to binary64 or
// binary32, shared by the two CRT kernels.  [Q] "2の累乗による整数化(手順1と5)":
// C_ij = X_ij 2^-(e_i + f_j), rounded once to nearest-even from the exact
// integer (subnormals and overflow to +-Inf included).
#pragma once
#include <stdint.h>

namespace os2crt {

// Target formats: binary64 (DGEMM) and binary32 (SGEMM emulation).
template <typename OutT>
struct Fmt;
template <>
struct Fmt<double> {
  static constexpr int prec = 53, emin = -1022, emax = 1023;
  // normal number from a significand with its leading bit at bit prec - 1 (or
  // 2^prec after a rounding carry) and the exponent of that leading bit: the
  // add carries a full significand into the exponent, up to +-Inf
  static __device__ __forceinline__ double pack_normal(uint64_t sig, int ex, bool neg) {
    uint64_t b = ((uint64_t)(ex + 1022) << 52) + sig;
    if (neg) b |= 1ull << 63;
    return __longlong_as_double((long long)b);
  }
  static __device__ __forceinline__ double make(uint64_t mant, int ex, bool neg, int kind) {
    // kind 0: normal (mant has prec bits, ex unbiased); 1: subnormal bits in mant; 2: inf
    uint64_t b = kind == 2 ? 0x7FF0000000000000ull
                           : (kind == 1 ? mant : (((uint64_t)(ex + 1023) << 52) | (mant & ((1ull << 52) - 1))));
    if (neg) b |= 1ull << 63;
    return __longlong_as_double((long long)b);
  }
};
template <>
struct Fmt<float> {
  static constexpr int prec = 24, emin = -126, emax = 127;
  static __device__ __forceinline__ float pack_normal(uint64_t sig, int ex, bool neg) {
    uint32_t b = ((uint32_t)(ex + 126) << 23) + (uint32_t)sig;
    if (neg) b |= 1u << 31;
    return __uint_as_float(b);
  }
  static __device__ __forceinline__ float make(uint64_t mant, int ex, bool neg, int kind) {
    uint32_t b = kind == 2 ? 0x7F800000u
                           : (kind == 1 ? (uint32_t)mant
                                        : (((uint32_t)(ex + 127) << 23) | ((uint32_t)mant & 0x7FFFFFu)));
    if (neg) b |= 1u << 31;
    return __uint_as_float(b);
  }
};

// RN-even of |X| * 2^-s to the format of OutT, |X| in 32-bit limbs m[0..L),
// sign `neg` (general routine: zero, subnormal and overflowing results; kept
// out of line).
// The limbs are passed as scalars (at most 6): an out-of-line call taking an
// array (or a struct) made every caller spill its limbs to the stack on every
// entry, slow path or not.
template <typename OutT, int L>
__device__ __noinline__ OutT round_scaled_v(uint32_t m0, uint32_t m1, uint32_t m2, uint32_t m3,
                                            uint32_t m4, uint32_t m5, bool neg, int s) {
  static_assert(L >= 1 && L <= 6, "at most 6 limbs");
  const uint32_t all[6] = {m0, m1, m2, m3, m4, m5};
  uint32_t m[L];
#pragma unroll
  for (int u = 0; u < L; u++) m[u] = all[u];
  using F = Fmt<OutT>;
  constexpr int lsb = F::prec - 1 - F::emin;  // -log2 of the smallest subnormal
  int top = -1;
#pragma unroll
  for (int u = 0; u < L; u++)
    if (m[u]) top = u;
  if (top < 0) return OutT(0);
  uint32_t mt = 0;
#pragma unroll
  for (int u = 0; u < L; u++)
    if (u == top) mt = m[u];
  const int b = 32 * top + 32 - __clz(mt);  // bit length of |X|
  int cut = max(b - F::prec, s - lsb);
  uint64_t kept;
  if (cut <= 0) {
    kept = (uint64_t)m[0] | (L > 1 ? (uint64_t)m[L > 1 ? 1 : 0] << 32 : 0ull);
    cut = 0;
  } else if (cut > b) {
    kept = 0;
  } else {
    // bits [cut, cut + prec + 1) of |X|, round bit cut - 1, sticky below
    const int w = cut >> 5, o = cut & 31;
    uint32_t a0 = 0, a1 = 0, a2 = 0;
#pragma unroll
    for (int u = 0; u < L; u++) {
      if (u == w) a0 = m[u];
      if (u == w + 1) a1 = m[u];
      if (u == w + 2) a2 = m[u];
    }
    const uint64_t lo64 = (uint64_t)a0 | ((uint64_t)a1 << 32);
    kept = (lo64 >> o) | (o ? ((uint64_t)a2 << (64 - o)) : 0ull);
    const int rb = cut - 1;
    const int rw = rb >> 5, ro = rb & 31;
    uint32_t rwv = 0;
    bool sticky = false;
#pragma unroll
    for (int u = 0; u < L; u++) {
      if (u == rw) rwv = m[u];
      if (u < rw) sticky |= m[u] != 0;
    }
    const uint32_t round = (rwv >> ro) & 1u;
    sticky |= (rwv & ((1u << ro) - 1u)) != 0;
    if (round && (sticky || (kept & 1))) kept++;
  }
  if (kept == 0) return neg ? -OutT(0) : OutT(0);
  const int x = cut - s;  // value = kept * 2^x
  const int bk = 64 - __clzll((long long)kept);
  const int etop = x + bk - 1;
  if (etop >= F::emin) {
    if (etop > F::emax) return F::make(0, 0, neg, 2);
    const uint64_t mant = bk >= F::prec ? kept >> (bk - F::prec) : kept << (F::prec - bk);
    return F::make(mant, etop, neg, 0);
  }
  return F::make(kept << (x + lsb), 0, neg, 1);  // subnormal: x >= -lsb by construction of cut
}

template <typename OutT, int L>
__device__ __forceinline__ OutT round_scaled(const uint32_t (&m)[L], bool neg, int s) {
  auto w = [&](int u) { return u < L ? m[u < L ? u : 0] : 0u; };
  return round_scaled_v<OutT, L>(w(0), w(1), w(2), w(3), w(4), w(5), neg, s);
}

// Normal-range fast path: the top three nonzero-anchored limbs hold at least
// 65 significant bits, enough for the significand, the round bit and a sticky
// bit (OR-ed with everything below).  Falls back to the general routine for
// zero, subnormal or overflowing results.
template <typename OutT, int L>
__device__ __forceinline__ OutT round_scaled_fast(const uint32_t (&m)[L], bool neg, int s) {
  using F = Fmt<OutT>;
  int t = -1;
#pragma unroll
  for (int u = 0; u < L; u++)
    if (m[u]) t = u;
  uint32_t hi = 0, mid = 0, lo = 0;
  bool rest = false;
#pragma unroll
  for (int u = 0; u < L; u++) {
    if (u == t) hi = m[u];
    if (u == t - 1) mid = m[u];
    if (u == t - 2) lo = m[u];
    if (u < t - 2) rest |= m[u] != 0;
  }
  const int lz = __clz(hi);
  const int etop = 32 * t + 31 - lz - s;  // exponent of the leading bit of |X| 2^-s
  if (t < 0 || etop < F::emin || etop > F::emax) return round_scaled<OutT, L>(m, neg, s);
  const uint32_t t1 = __funnelshift_l(mid, hi, lz);
  const uint32_t t0 = __funnelshift_l(lo, mid, lz);
  const uint32_t tail = lo << lz;  // bits below the 64-bit window (lz < 32)
  const uint64_t T = ((uint64_t)t1 << 32) | t0;
  uint64_t kept = T >> (64 - F::prec);  // leading bit set
  const bool round = (T >> (63 - F::prec)) & 1;
  const bool sticky = (T & ((1ull << (63 - F::prec)) - 1)) != 0 || tail != 0 || rest;
  int ex = etop;
  if (round && (sticky || (kept & 1))) {
    kept++;
    if (kept >> F::prec) {
      kept >>= 1;
      ex++;
    }
  }
  return ex > F::emax ? F::make(0, 0, neg, 2) : F::make(kept, ex, neg, 0);
}

// RN-even of |X| 2^-s for |X| whose top limb m[L-1] is nonzero and whose
// result is a normal number (the common case); anything else goes to the
// general routine.  The significand is the top 64 bits below the leading one
// of the top limb; the bits below that window only feed the sticky bit.
template <typename OutT, int L>
__device__ __forceinline__ OutT round_scaled_top(const uint32_t (&m)[L], bool neg, int s) {
  using F = Fmt<OutT>;
  const uint32_t hi = m[L - 1];
  const int lz = __clz(hi);
  const int etop = 32 * (L - 1) + 31 - lz - s;  // exponent of the leading bit of |X| 2^-s
  if (hi == 0 || etop < F::emin || etop > F::emax) return round_scaled<OutT, L>(m, neg, s);
  const uint32_t mid = L >= 2 ? m[L >= 2 ? L - 2 : 0] : 0u;
  const uint32_t lo = L >= 3 ? m[L >= 3 ? L - 3 : 0] : 0u;
  uint32_t rest = 0;
#pragma unroll
  for (int u = 0; u + 3 < L; u++) rest |= m[u];
  const uint64_t T = ((uint64_t)__funnelshift_l(mid, hi, lz) << 32) | __funnelshift_l(lo, mid, lz);
  const uint64_t kept = T >> (64 - F::prec);
  const uint32_t round = (uint32_t)(T >> (63 - F::prec)) & 1u;
  const bool sticky = (T & ((1ull << (63 - F::prec)) - 1)) != 0 || (lo << lz) != 0 || rest != 0;
  const uint32_t inc = round & ((sticky ? 1u : 0u) | (uint32_t)kept);
  return F::pack_normal(kept + inc, etop, neg);
}

// Exact float of x < 2^23 from its bit pattern.
__device__ __forceinline__ float u23_to_float(uint32_t x) {
  return __uint_as_float(0x4B000000u | x) - 8388608.0f;
}
// fl(y) for y < 2^46, one rounding.
__device__ __forceinline__ float u46_to_float(uint64_t y) {
  return fmaf(u23_to_float((uint32_t)(y >> 23)), 8388608.0f, u23_to_float((uint32_t)y & 0x7FFFFFu));
}

}  // namespace os2crt
