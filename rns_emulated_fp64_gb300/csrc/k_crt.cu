// Steps 4 and 5: Chinese-remainder reconstruction and unscaling.
//
// [Q] "繰り上がりのない計算" / "秦九韶の大衍求一術": the integer with residues c_l is
// X = (sum_l c_l W_l) mod P, W_l = M_l inv_l (the "use numbers"), M_l = P/p_l,
// inv_l = M_l^-1 mod p_l.  [Q] "高い精度での復元(手順4)": P reaches 2^125 at 16
// moduli, beyond double and int64, so this step needs more precision.  GB300's
// FP64 rate is low, so instead of the double-double arithmetic the article
// describes, X is computed exactly in 32-bit integer limbs:
//   Y_u = sum_l (c_l + 128) W_l,u      unsigned 64-bit sums, no carries yet
//   Y   = sum_u Y_u 2^(32u) = S + 128 sum_l W_l,   S = sum_l c_l W_l
// The W_l sum to 1 mod P (each is 1 mod its own p_l and 0 mod the others), so
// Y - 128 = S mod P, and
//   q   = nearest integer to (Y - 128) / P >= 0, estimated in FP32 from the
//         two highest limb sums (error below 0.003)
//   X   = Y - 128 - q P, carries propagated once; if the estimate was within
//         0.01 of a half-integer, one exact comparison with P/2 fixes q.
// Only full-rate FP32 and 32-bit integer units are used: the limb sums reach
// FP32 through 23-bit pieces laid into float bit patterns, and the estimate is
// rounded by adding 1.5 * 2^23 (64-bit-integer conversions and rounding
// instructions run on GB300's narrow FP64 and conversion units).
// X lies in [-P/2, P/2).  [Q] "2の累乗による整数化(手順1と5)": C_ij = X_ij 2^-(e_i+f_j),
// rounded once to nearest-even from the exact integer (subnormals, overflow).
//
// One thread per 4 consecutive entries of a row: each residue plane is read
// with one 4-byte load per thread (coalesced).
#include "crt_round.cuh"
#include "os2_internal.cuh"

namespace {

using namespace os2crt;

constexpr int kThreads = 128;

// 32-bit limbs of P (and of every W_l < P): each group of four moduli of the
// table adds just under 32 bits (bit lengths 32, 64, 95, 126, 156 at N = 4,
// 8, 12, 16, 20), so (N + 3) / 4 limbs hold P; one more holds Y < 256 N P.
template <int N>
struct Limbs {
  static constexpr int LW = (N + 3) / 4;
  static constexpr int LX = LW + 1;
};

template <int N, typename OutT>
__global__ void __launch_bounds__(kThreads)
    k_crt(int m, int n, int groups, const int8_t *__restrict__ c, int ldcres,
          const int32_t *__restrict__ e, const int32_t *__restrict__ f, OutT *__restrict__ C,
          int ldc, uint32_t *__restrict__ Xout, const CrtConsts cc, int *status) {
  constexpr int LW = Limbs<N>::LW, LX = Limbs<N>::LX;
  const int g = blockIdx.x * kThreads + threadIdx.x;
  if (g >= groups) return;
  const int j0 = g * 4;
  for (int i = blockIdx.y; i < m; i += gridDim.y) {

  // residues + 128 of 4 entries per modulus, one byte each
  uint32_t r4[N];
  const size_t plane = (size_t)m * ldcres;
  const int8_t *src = c + (size_t)i * ldcres + j0;
  if (j0 + 4 <= n) {
#pragma unroll
    for (int l = 0; l < N; l++)
      r4[l] = OS2_DBG_GUARD(i < m && j0 + 4 <= ldcres, status)
                  ? __ldg(reinterpret_cast<const uint32_t *>(src + l * plane)) ^ 0x80808080u
                  : 0x80808080u;
  } else {
#pragma unroll
    for (int l = 0; l < N; l++) {
      uint32_t v = 0;
      for (int u = 0; u < 4 && j0 + u < n; u++) v |= (uint32_t)(uint8_t)src[l * plane + u] << (8 * u);
      r4[l] = v ^ 0x80808080u;
    }
  }
  const int ei = e[i];

#pragma unroll 1
  for (int u = 0; u < 4; u++) {
    const int j = j0 + u;
    if (j >= n) break;
    const uint32_t sel = 0x4440u | (uint32_t)u;  // byte u, zero-extended
    // Y_v = sum_l (c_l + 128) W_l,v
    uint64_t Y[LW];
#pragma unroll
    for (int v = 0; v < LW; v++) Y[v] = 0;
#pragma unroll
    for (int l = 0; l < N; l++) {
      const uint32_t cl = __byte_perm(r4[l], 0u, sel);
#pragma unroll
      for (int v = 0; v < LW; v++) Y[v] += (uint64_t)cl * cc.W32[l][v];
    }
    // q = round((Y - 128) / P) from the two top limb sums (each < 2^46)
    float t = fmaf(u46_to_float(Y[LW - 1]), cc.s_top, -cc.s128);
    if (LW > 1) t = fmaf(u46_to_float(Y[LW > 1 ? LW - 2 : 0]), cc.s_next, t);
    const float tq = t + 12582912.0f;  // 1.5 * 2^23: rounds t (-0.5 <= t < 2^13) to an integer
    int qi = __float_as_int(tq) - 0x4B400000;
    float qf = tq - 12582912.0f;
    if (qi < 0) {  // only when Y - 128 is within rounding of -P/2 (then q = 0 is right)
      qi = 0;
      qf = 0.0f;
    }
    const uint32_t q = (uint32_t)qi;
    // X = Y - 128 - q P in signed 64-bit limb sums (|each| < 2^46), one carry pass
    uint32_t x[LX];
    long long carry = 0;
#pragma unroll
    for (int v = 0; v < LX; v++) {
      const long long yv = v < LW ? (long long)Y[v < LW ? v : 0] : 0ll;
      const long long qp = (long long)((uint64_t)q * cc.P32[v]);
      const long long sv = yv - qp - (v == 0 ? 128 : 0) + carry;
      x[v] = (uint32_t)sv;
      carry = sv >> 32;
    }
    // X is far inside the 32*LX-bit window, so its sign is the top bit of
    // x[LX-1].  The quotient can be off by one only when the estimate sat
    // within 0.01 of a half-integer; then compare X with +-P/2 exactly.
    const float fr = t - qf;
    if (fr > 0.49f || fr < -0.49f) {
      const bool up = fr > 0.49f;  // X may be >= P/2 (then X -= P); else X may be < -P/2
      long long cr = 0;
      uint32_t last = 0;
#pragma unroll
      for (int v = 0; v < LX; v++) {
        const long long dv =
            (long long)x[v] + (up ? -(long long)cc.H32[v] : (long long)cc.H32[v]) + cr;
        last = (uint32_t)dv;
        cr = dv >> 32;
      }
      const bool dneg = (int32_t)last < 0;  // sign of X -+ P/2
      if (up ? !dneg : dneg) {
        long long cr2 = 0;
#pragma unroll
        for (int v = 0; v < LX; v++) {
          const long long sv =
              (long long)x[v] + (up ? -(long long)cc.P32[v] : (long long)cc.P32[v]) + cr2;
          x[v] = (uint32_t)sv;
          cr2 = sv >> 32;
        }
      }
    }
    const bool neg = (int32_t)x[LX - 1] < 0;
    if (Xout && OS2_DBG_GUARD(i < m && j < n, status)) {
      uint32_t *xo = Xout + ((size_t)i * n + j) * 8;
#pragma unroll
      for (int v = 0; v < 8; v++) xo[v] = v < LX ? x[v < LX ? v : 0] : (neg ? 0xFFFFFFFFu : 0u);
    }
    uint32_t mag[LX];
    if (neg) {
      uint64_t cy = 1;
#pragma unroll
      for (int v = 0; v < LX; v++) {
        cy += (uint64_t)(~x[v]);
        mag[v] = (uint32_t)cy;
        cy >>= 32;
      }
    } else {
#pragma unroll
      for (int v = 0; v < LX; v++) mag[v] = x[v];
    }
    // |X| <= P/2 < 2^(32 LW): the top limb of the window is zero, and the
    // normal-range fast path reads the LW limbs below it
    uint32_t magw[LW];
#pragma unroll
    for (int v = 0; v < LW; v++) magw[v] = mag[v];
    if (OS2_DBG_GUARD(i < m && j < n && n <= ldc, status))
      C[(size_t)i * ldc + j] = round_scaled_top<OutT, LW>(magw, neg, ei + f[j]);
  }
  }
}

template <typename OutT>
cudaError_t crt_t(int m, int n, const int8_t *c, int ldcres, const int32_t *e, const int32_t *f,
                  OutT *C, int ldc, uint32_t *X_out, const Os2Tables *t, cudaStream_t s,
                  int *status) {
  const int groups = (n + 3) / 4;
  const dim3 grid((groups + kThreads - 1) / kThreads, m < 65535 ? m : 65535);
#define OS2_CASE(NN)                                                                              \
  case NN:                                                                                        \
    k_crt<NN, OutT><<<grid, kThreads, 0, s>>>(m, n, groups, c, ldcres, e, f, C, ldc, X_out, t->crt, \
                                              status);                                        \
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

}  // namespace

cudaError_t launch_crt(bool f32, int m, int n, const int8_t *c, int ldcres, const int32_t *e,
                       const int32_t *f, void *C, int ldc, uint32_t *X_out, const Os2Tables *t,
                       cudaStream_t s, int *status) {
  if (m <= 0 || n <= 0) return cudaSuccess;
  return f32 ? crt_t<float>(m, n, c, ldcres, e, f, static_cast<float *>(C), ldc, X_out, t, s,
                            status)
             : crt_t<double>(m, n, c, ldcres, e, f, static_cast<double *>(C), ldc, X_out, t, s,
                             status);
}
