// Step 2: the residue kernel, instantiated for N = 1..20 moduli and both
// element types in eight translation units (k_residues_{d,f}{1,2,3,4}.cu),
// which compile in parallel.
//
// [Q] "2の累乗による整数化(手順1と5)" / "256以下の法の選び方(手順2)": the scaled
// integers trunc(a_ih 2^e_i) are reduced to residues held around zero,
// [-floor(p/2), ceil(p/2) - 1], which always fit int8 and are stored as FP16
// (exact for |r| <= 2048) for the tensor-core products of step 3.
//
// Element-parallel: every thread turns 8 consecutive entries into 8 residues
// per modulus and writes one 16-byte vector to each plane.  Residues of the
// odd moduli use FP32 arithmetic only: the integer is split into four to six
// 15-bit words w_t (as many as its size needs) and x = K + sum_t w_t (2^(15t)
// mod p) is exact below 2^23, so one fused multiply-add rounds x / p to the
// nearest integer exactly.  Two entries share each packed FP32 instruction.
// Mod 256 is the integer's low byte.
#pragma once
#include <type_traits>

#include "k_rows.cuh"

namespace os2dev {

constexpr int kThreads = 256;

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

// EPT residues (exact small integers held as floats) as int8: the low byte of
// r + 1.5 * 2^23 is r in two's complement.
template <int EPT>
__device__ __forceinline__ void store_i8(const float (&r)[EPT], int8_t *dst) {
  uint32_t b[EPT];
#pragma unroll
  for (int u = 0; u < EPT; u++) b[u] = __float_as_uint(r[u] + 12582912.0f);
  uint32_t w[EPT / 4];
#pragma unroll
  for (int q = 0; q < EPT / 4; q++)
    w[q] = __byte_perm(__byte_perm(b[4 * q], b[4 * q + 1], 0x0040),
                       __byte_perm(b[4 * q + 2], b[4 * q + 3], 0x0040), 0x5410);
  if (EPT == 8)
    *reinterpret_cast<uint2 *>(dst) = make_uint2(w[0], w[EPT == 8 ? 1 : 0]);
  else
    *reinterpret_cast<uint32_t *>(dst) = w[0];
}

// Residues of EPT entries (held as int_words gives them) for every modulus,
// one vector store of EPT values per plane: FP16 (exact for |r| <= 2048), or
// int8 when `i8` (half the bytes; the step-3 variant widens them on chip).  For odd p_l, with
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
                                     const ResConsts &c, __half *dst, size_t pstride, bool i8) {
  static_assert(EPT == 4 || EPT == 8, "4 or 8 entries per thread");
  using Vec = typename std::conditional<EPT == 8, uint4, uint2>::type;
  int8_t *dst8 = reinterpret_cast<int8_t *>(dst);  // int8 planes: element offsets in bytes
  if (i8) {
    float r[EPT];
#pragma unroll
    for (int u = 0; u < EPT; u++) r[u] = byte_residue(lb[u]);
    store_i8<EPT>(r, dst8);
  } else {
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
    float r[EPT];
#pragma unroll
    for (int u = 0; u < EPT / 2; u++) {
      unsigned long long x = fma2(W[u][0], c.w15x2[l][0], c.k15x2[l][NW - 4]);
#pragma unroll
      for (int t = 1; t < NW; t++) x = fma2(W[u][t], c.w15x2[l][t], x);
      const unsigned long long q = add2(fma2(x, c.invp2[l], kMagic2), kNegMagic2);
      unpack2(fma2(c.negp2[l], q, x), r[2 * u], r[2 * u + 1]);
    }
    if (i8) {
      store_i8<EPT>(r, dst8 + l * pstride);
    } else {
      __align__(16) __half2 v[EPT / 2];
#pragma unroll
      for (int u = 0; u < EPT / 2; u++) v[u] = __floats2half2_rn(r[2 * u], r[2 * u + 1]);
      *reinterpret_cast<Vec *>(dst + l * pstride) = *reinterpret_cast<Vec *>(v);
    }
  }
}

template <int N, int NW, typename T, int EPT>
__device__ __forceinline__ void residues_of(const T (&v)[EPT], int ee, const ResConsts &c,
                                            __half *dst, size_t pstride, bool i8) {
  float w[EPT][NW];
  uint32_t lb[EPT];
#pragma unroll
  for (int u = 0; u < EPT; u++) {
    const Dec d = decode(v[u]);
    int_words<NW>(d, d.ex2 + ee, w[u], lb[u]);
  }
  emit<N, NW, EPT>(w, lb, c, dst, pstride, i8);
}

// Residue planes: EPT consecutive entries per thread, one vector store per plane.
constexpr int kEPT = 8;

template <int N, typename T>
__global__ void __launch_bounds__(kThreads, 3)
    k_residues(const RowSet a, const RowSet b, int k, int kp, const ResConsts c, int *status,
               bool i8) {
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
      if (!OS2_DBG_GUARD(row < rs.rows && rs.prow >= rs.rows && h0 + EPT <= kp && k <= kp &&
                             k <= rs.ldx,
                         status))
        continue;
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
      // element offset row * kp + h0 (FP16 or int8 elements)
      __half *dst = i8 ? reinterpret_cast<__half *>(reinterpret_cast<int8_t *>(rs.planes) +
                                                     (size_t)row * kp + h0)
                       : rs.planes + (size_t)row * kp + h0;
      if (top <= 59) {
        residues_of<N, 4>(v, ee, c, dst, pstride, i8);
      } else if (top <= 74) {
        residues_of<N, 5>(v, ee, c, dst, pstride, i8);
      } else if (top <= 89) {
        residues_of<N, 6>(v, ee, c, dst, pstride, i8);
      } else {
        // beyond every exponent that step 1 produces (|integer| < 2^84):
        // reported, and the entries' residues are left as zero
        set_status(status, OS2_ERR_RANGE);
#pragma unroll
        for (int l = 0; l < N; l++)
#pragma unroll
          for (int u = 0; u < EPT; u++) {
            if (i8)
              reinterpret_cast<int8_t *>(dst)[l * pstride + u] = 0;
            else
              dst[l * pstride + u] = __float2half(0.0f);
          }
      }
    }
  }
}

template <int N, typename T>
cudaError_t residues_launch(const RowSet &a, const RowSet &b, int k, int kp, const ResConsts &c,
                            int *status, cudaStream_t s, bool i8) {
  const int cpr = kp / kEPT;
  const int bx = (cpr + kThreads - 1) / kThreads;
  const int rows = a.rows + b.rows;
  dim3 grid(bx, rows < 65535 ? rows : 65535);
  k_residues<N, T><<<grid, kThreads, 0, s>>>(a, b, k, kp, c, status, i8);
  return cudaGetLastError();
}

// One translation unit each: N in [1, 12], [13, 16], [17, 18], [19, 20], double
// and float (the larger N unroll more code).
#define OS2_RESIDUES_PART(name)                                                               \
  cudaError_t name(int N, const RowSet &a, const RowSet &b, int k, int kp, const ResConsts &c, \
                   int *status, cudaStream_t s, bool i8)
OS2_RESIDUES_PART(residues_d1);
OS2_RESIDUES_PART(residues_d2);
OS2_RESIDUES_PART(residues_d3);
OS2_RESIDUES_PART(residues_d4);
OS2_RESIDUES_PART(residues_f1);
OS2_RESIDUES_PART(residues_f2);
OS2_RESIDUES_PART(residues_f3);
OS2_RESIDUES_PART(residues_f4);
#define OS2_RESIDUES_CASE(NN, T) \
  case NN:                       \
    return residues_launch<NN, T>(a, b, k, kp, c, status, s, i8);

}  // namespace os2dev
