// Steps 4 and 5: Chinese-remainder reconstruction and unscaling.
//
// [Q] "繰り上がりのない計算" / "秦九韶の大衍求一術": the integer with residues c_l is
// X = (sum_l c_l W_l) mod P, W_l = M_l inv_l (the "use numbers"), M_l = P/p_l,
// inv_l = M_l^-1 mod p_l.  [Q] "高い精度での復元(手順4)": P reaches 2^125 at 16
// moduli, beyond double and int64, so this step needs more precision.  GB300's
// FP64 rate is low, so instead of the double-double arithmetic the article
// describes, X is computed exactly in integer limbs:
//   S_u = sum_l c_l W_l,u  (16-bit limbs of W_l; |S_u| < 2^31, no carries yet)
//   q   = rint(sum_l c_l fl(inv_l / p_l))   (FP32; the exact S/P = sum c_l inv_l/p_l)
//   X   = S - q P, carries propagated once; a one-step correction if the FP32
//         estimate was within 0.01 of a half-integer.
// X lies in [-P/2, P/2).  [Q] "2の累乗による整数化(手順1と5)": C_ij = X_ij 2^-(e_i+f_j),
// rounded once to nearest-even from the exact integer (subnormals, overflow).
//
// One thread per 4 consecutive entries of a row: each residue plane is read
// with one 4-byte load per thread (coalesced), C with 8-byte stores.
#include "os2_internal.cuh"

namespace {

constexpr int kThreads = 128;

// RN-even of (w2:w1:w0) * 2^-s, sign `neg`; mirrors IEEE-754 binary64.
__device__ __forceinline__ double round_scaled(uint64_t w0, uint64_t w1, uint64_t w2, bool neg,
                                               int s) {
  if ((w0 | w1 | w2) == 0) return 0.0;
  const uint64_t w[4] = {w0, w1, w2, 0};
  int b = w2 ? 128 + 64 - __clzll((long long)w2)
             : (w1 ? 64 + 64 - __clzll((long long)w1) : 64 - __clzll((long long)w0));
  int cut = max(b - 53, s - 1074);
  uint64_t kept;
  if (cut <= 0) {
    kept = w0;
    cut = 0;
  } else if (cut > b) {
    kept = 0;
  } else {
    const int idx = cut >> 6, off = cut & 63;
    kept = w[idx] >> off;
    if (off && idx + 1 < 4) kept |= w[idx + 1] << (64 - off);
    const int rb = cut - 1;  // round bit position
    const uint64_t round = (w[rb >> 6] >> (rb & 63)) & 1;
    bool sticky = false;
    const int sw = rb >> 6, sb = rb & 63;  // bits [0, rb)
    for (int i = 0; i < sw; i++) sticky |= w[i] != 0;
    if (sb) sticky |= (w[sw] & ((1ull << sb) - 1)) != 0;
    if (round && (sticky || (kept & 1))) kept++;
  }
  if (kept == 0) return neg ? -0.0 : 0.0;
  const int x = cut - s;  // value = kept * 2^x
  const int bk = 64 - __clzll((long long)kept);
  const int etop = x + bk - 1;
  uint64_t bits;
  if (etop >= -1022) {
    if (etop > 1023) {
      bits = 0x7FF0000000000000ull;
    } else {
      const uint64_t mant = bk >= 53 ? kept >> (bk - 53) : kept << (53 - bk);
      bits = ((uint64_t)(etop + 1023) << 52) | (mant & ((1ull << 52) - 1));
    }
  } else {
    bits = kept << (x + 1074);  // subnormal: x >= -1074 by construction of cut
  }
  if (neg) bits |= 1ull << 63;
  return __longlong_as_double((long long)bits);
}

template <int N>
__global__ void __launch_bounds__(kThreads)
    k_crt(int m, int n, int groups, const int8_t *__restrict__ c, int ldcres,
          const int32_t *__restrict__ e, const int32_t *__restrict__ f, double *__restrict__ C,
          int ldc, uint32_t *__restrict__ Xout, const CrtConsts cc) {
  const long long gid = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (gid >= (long long)m * groups) return;
  const int i = (int)(gid / groups);
  const int j0 = (int)(gid - (long long)i * groups) * 4;

  int32_t r4[N];
  const size_t plane = (size_t)m * ldcres;
  const int8_t *src = c + (size_t)i * ldcres + j0;
  if (j0 + 4 <= n) {
#pragma unroll
    for (int l = 0; l < N; l++) r4[l] = __ldg(reinterpret_cast<const int32_t *>(src + l * plane));
  } else {
#pragma unroll
    for (int l = 0; l < N; l++) {
      uint32_t v = 0;
      for (int u = 0; u < 4 && j0 + u < n; u++) v |= (uint32_t)(uint8_t)src[l * plane + u] << (8 * u);
      r4[l] = (int32_t)v;
    }
  }
  const int ei = e[i];

#pragma unroll 1
  for (int u = 0; u < 4; u++) {
    const int j = j0 + u;
    if (j >= n) break;
    float t = 0.f;
    int acc[OS2_CRT_LIMBS];
#pragma unroll
    for (int v = 0; v < OS2_CRT_LIMBS; v++) acc[v] = 0;
#pragma unroll
    for (int l = 0; l < N; l++) {
      const int cl = (int)(int8_t)((uint32_t)r4[l] >> (8 * u));
      t = fmaf((float)cl, cc.phi[l], t);
#pragma unroll
      for (int v = 0; v < OS2_CRT_LIMBS; v++) acc[v] += cl * cc.W16[l][v];
    }
    const float qf = rintf(t);
    const int q = (int)qf;
#pragma unroll
    for (int v = 0; v < OS2_CRT_LIMBS; v++) acc[v] -= q * cc.P16[v];
    uint32_t x16[OS2_CRT_LIMBS];
    int carry = 0;
#pragma unroll
    for (int v = 0; v < OS2_CRT_LIMBS; v++) {
      const int sv = acc[v] + carry;
      x16[v] = (uint32_t)sv & 0xFFFFu;
      carry = sv >> 16;
    }
    // |t - S/P| < 0.003, so X is already in [-P/2, P/2) unless the estimate
    // was near a half-integer; then compare with P/2 exactly.
    const float fr = t - qf;
    if (fr > 0.49f) {
      int cr = 0;
      for (int v = 0; v < OS2_CRT_LIMBS; v++) cr = ((int)x16[v] - cc.half16[v] + cr) >> 16;
      if (carry + cr >= 0) {  // X >= P/2: X -= P
        cr = 0;
        for (int v = 0; v < OS2_CRT_LIMBS; v++) {
          const int sv = (int)x16[v] - cc.P16[v] + cr;
          x16[v] = (uint32_t)sv & 0xFFFFu;
          cr = sv >> 16;
        }
        carry += cr;
      }
    } else if (fr < -0.49f) {
      int cr = 0;
      for (int v = 0; v < OS2_CRT_LIMBS; v++) cr = ((int)x16[v] + cc.half16[v] + cr) >> 16;
      if (carry + cr < 0) {  // X < -P/2: X += P
        cr = 0;
        for (int v = 0; v < OS2_CRT_LIMBS; v++) {
          const int sv = (int)x16[v] + cc.P16[v] + cr;
          x16[v] = (uint32_t)sv & 0xFFFFu;
          cr = sv >> 16;
        }
        carry += cr;
      }
    }
    const bool neg = carry < 0;
    uint64_t w0 = (uint64_t)x16[0] | ((uint64_t)x16[1] << 16) | ((uint64_t)x16[2] << 32) |
                  ((uint64_t)x16[3] << 48);
    uint64_t w1 = (uint64_t)x16[4] | ((uint64_t)x16[5] << 16) | ((uint64_t)x16[6] << 32) |
                  ((uint64_t)x16[7] << 48);
    uint64_t w2 = (uint64_t)x16[8] | ((uint64_t)x16[9] << 16);
    if (neg) w2 |= 0xFFFFFFFF00000000ull;  // sign-extend the 160-bit value to 192 bits
    if (Xout) {
      uint32_t *xo = Xout + ((size_t)i * n + j) * 8;
      xo[0] = (uint32_t)w0; xo[1] = (uint32_t)(w0 >> 32);
      xo[2] = (uint32_t)w1; xo[3] = (uint32_t)(w1 >> 32);
      xo[4] = (uint32_t)w2; xo[5] = (uint32_t)(w2 >> 32);
      xo[6] = neg ? 0xFFFFFFFFu : 0u; xo[7] = neg ? 0xFFFFFFFFu : 0u;
    }
    if (neg) {  // magnitude = two's complement
      w0 = ~w0; w1 = ~w1; w2 = ~w2;
      w0 += 1;
      const uint64_t c0 = w0 == 0;
      w1 += c0;
      const uint64_t c1 = c0 & (w1 == 0);
      w2 += c1;
    }
    C[(size_t)i * ldc + j] = round_scaled(w0, w1, w2, neg, ei + f[j]);
  }
}

}  // namespace

cudaError_t launch_crt(int m, int n, const int8_t *c, int ldcres, const int32_t *e,
                       const int32_t *f, double *C, int ldc, uint32_t *X_out, const Os2Tables *t,
                       cudaStream_t s) {
  if (m <= 0 || n <= 0) return cudaSuccess;
  const int groups = (n + 3) / 4;
  const long long total = (long long)m * groups;
  const unsigned blocks = (unsigned)((total + kThreads - 1) / kThreads);
#define OS2_CASE(NN)                                                                         \
  case NN:                                                                                   \
    k_crt<NN><<<blocks, kThreads, 0, s>>>(m, n, groups, c, ldcres, e, f, C, ldc, X_out, t->crt); \
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
