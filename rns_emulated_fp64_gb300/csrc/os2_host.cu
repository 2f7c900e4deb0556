// libos2 host side: the C ABI declared in include/os2.h, argument checking,
// workspace layout, constant tables and the launch sequence of the five steps.
#include <cuda_runtime.h>
#include <math.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "os2_internal.cuh"

// ---------------------------------------------------------------------------
// Device status word (one per device); kernels receive its address.
// ---------------------------------------------------------------------------
__device__ int g_os2_status;

int os2_sm_count() {
  int dev = 0, v = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
  return v > 0 ? v : 1;
}

int *os2_status_ptr() {
  static std::mutex mu;
  static int *ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_os2_status) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<int *>(p);
  }
  return ptrs[dev];
}

// ---------------------------------------------------------------------------
// Constant tables.  [Q] "256以下の法の選び方(手順2)" (moduli, footnote 6 order),
// "秦九韶の大衍求一術" (M_l, inverses by the extended Euclidean algorithm,
// use numbers W_l = M_l inv_l).
// ---------------------------------------------------------------------------
namespace {

const int kModuli[OS2_MAX_MODULI] = {256, 255, 253, 251, 247, 241, 239, 233, 229, 227,
                                     223, 217, 211, 199, 197, 193, 191, 181, 179, 173};

struct U256 {
  uint32_t w[8];
};
U256 u_from(uint32_t v) {
  U256 r = {};
  r.w[0] = v;
  return r;
}
U256 u_mul(const U256 &a, uint32_t s) {
  U256 r;
  uint64_t c = 0;
  for (int i = 0; i < 8; i++) {
    c += (uint64_t)a.w[i] * s;
    r.w[i] = (uint32_t)c;
    c >>= 32;
  }
  return r;
}
U256 u_div(const U256 &a, uint32_t d, uint32_t *rem) {
  U256 q;
  uint64_t r = 0;
  for (int i = 7; i >= 0; i--) {
    uint64_t cur = (r << 32) | a.w[i];
    q.w[i] = (uint32_t)(cur / d);
    r = cur % d;
  }
  if (rem) *rem = (uint32_t)r;
  return q;
}
U256 u_sub_small(const U256 &a, uint32_t v) {
  U256 r = a;
  uint64_t b = v;
  for (int i = 0; i < 8 && b; i++) {
    const uint64_t cur = r.w[i];
    r.w[i] = (uint32_t)(cur - b);
    b = cur < b ? 1 : 0;
  }
  return r;
}
U256 u_sub1(const U256 &a) {
  U256 r = a;
  for (int i = 0; i < 8; i++) {
    if (r.w[i]--) break;
  }
  return r;
}
U256 u_shr1(const U256 &a) {
  U256 r;
  for (int i = 0; i < 8; i++) r.w[i] = (a.w[i] >> 1) | (i + 1 < 8 ? a.w[i + 1] << 31 : 0u);
  return r;
}
U256 u_add(const U256 &a, const U256 &b) {
  U256 r;
  uint64_t c = 0;
  for (int i = 0; i < 8; i++) {
    c += (uint64_t)a.w[i] + b.w[i];
    r.w[i] = (uint32_t)c;
    c >>= 32;
  }
  return r;
}
U256 u_neg(const U256 &a) {  // two's complement modulo 2^256
  U256 r;
  uint64_t c = 1;
  for (int i = 0; i < 8; i++) {
    c += (uint64_t)(~a.w[i]);
    r.w[i] = (uint32_t)c;
    c >>= 32;
  }
  return r;
}
U256 u_shl(const U256 &a, int s) {
  U256 r = {};
  for (int i = 7; i >= 0; i--) {
    const int src = i - s / 32, o = s % 32;
    uint32_t v = src >= 0 ? a.w[src] << o : 0u;
    if (o && src - 1 >= 0) v |= a.w[src - 1] >> (32 - o);
    r.w[i] = v;
  }
  return r;
}
U256 u_shr(const U256 &a, int s) {
  U256 r = {};
  for (int i = 0; i < 8; i++) {
    const int src = i + s / 32, o = s % 32;
    uint32_t v = src < 8 ? a.w[src] >> o : 0u;
    if (o && src + 1 < 8) v |= a.w[src + 1] << (32 - o);
    r.w[i] = v;
  }
  return r;
}
bool u_zero(const U256 &a) {
  for (int i = 0; i < 8; i++)
    if (a.w[i]) return false;
  return true;
}
int u_bitlen(const U256 &a) {
  for (int i = 7; i >= 0; i--)
    if (a.w[i]) return 32 * i + 32 - __builtin_clz(a.w[i]);
  return 0;
}
double u_to_double(const U256 &a) {
  double r = 0;
  for (int i = 7; i >= 0; i--) r = r * 4294967296.0 + (double)a.w[i];
  return r;
}

// a^-1 mod p by the extended Euclidean algorithm (a, p coprime)
int inv_mod(int a, int p) {
  int r0 = p, r1 = ((a % p) + p) % p, t0 = 0, t1 = 1;
  while (r1) {
    int q = r0 / r1, tmp = r0 - q * r1;
    r0 = r1;
    r1 = tmp;
    tmp = t0 - q * t1;
    t0 = t1;
    t1 = tmp;
  }
  return ((t0 % p) + p) % p;
}

int sym(int x, int p) {
  int r = ((x % p) + p) % p;
  return r >= (p + 1) / 2 ? r - p : r;
}

void build_tables(int N, Os2Tables *t) {
  memset(t, 0, sizeof(*t));
  t->N = N;
  U256 P = u_from(1);
  for (int l = 0; l < N; l++) P = u_mul(P, (uint32_t)kModuli[l]);
  const U256 H = u_shr1(u_sub1(P));  // floor((P-1)/2)
  const U256 half = u_shr1(P);       // P/2 (P is even: 256 is a modulus)
  t->res.N = t->crt.N = t->gemm.N = N;
  for (int l = 0; l < N; l++) {
    const int p = kModuli[l];
    t->p[l] = p;
    uint32_t rem = 0;
    const U256 M = u_div(P, (uint32_t)p, nullptr);
    u_div(M, (uint32_t)p, &rem);
    t->inv[l] = inv_mod((int)rem, p);
    const U256 W = u_mul(M, (uint32_t)t->inv[l]);
    const float fp = (float)p, hi = (float)((p + 1) / 2 - 1), lo = (float)(-(p / 2));
    t->res.p[l] = t->gemm.p[l] = fp;
    t->res.invp[l] = t->gemm.invp[l] = 1.0f / fp;
    t->res.hi[l] = t->gemm.hi[l] = hi;
    t->res.lo[l] = t->gemm.lo[l] = lo;
    auto twice = [](float f) {
      uint32_t u;
      memcpy(&u, &f, 4);
      return ((unsigned long long)u << 32) | u;
    };
    int c15[6], pw = 1;
    for (int u = 0; u < 6; u++) {
      c15[u] = sym(pw, p);
      t->res.w15x2[l][u] = twice((float)c15[u]);
      pw = (int)(((long long)pw * 32768) % p);
    }
    for (int nw = 4; nw <= 6; nw++) {
      int ks = 0;
      for (int u = 0; u < nw - 1; u++) ks = (ks + 16384 * c15[u]) % p;
      t->res.k15x2[l][nw - 4] = twice((float)sym(ks, p));
    }
    t->res.invp2[l] = twice(1.0f / fp);
    t->res.negp2[l] = twice(-fp);
    for (int v = 0; v < 5; v++) t->crt.W32[l][v] = W.w[v];
  }
  for (int v = 0; v < 6; v++) {
    t->crt.P32[v] = P.w[v];
    t->crt.H32[v] = half.w[v];
  }
  // Tensor-core CRT: signed 10-bit digits of the W_l, W_l = sum_t w_{l,t} 2^(10 t)
  {
    CrtTcConsts &k = t->crt_tc;
    k.N = N;
    k.LX = 1;  // smallest limb count with 2^(32 LX) > 3P
    {
      const U256 P3 = u_mul(P, 3);
      while (k.LX < 8 && u_bitlen(P3) > 32 * k.LX) k.LX++;
    }
    int T = 0;
    for (int l = 0; l < N; l++) {
      const U256 M = u_div(P, (uint32_t)kModuli[l], nullptr);
      U256 W = u_mul(M, (uint32_t)t->inv[l]);
      int d = 0;
      while (!u_zero(W)) {
        int r = (int)(W.w[0] & 1023u);
        if (r >= 512) r -= 1024;
        if (d < OS2_CRT_DIGITS) k.wd[l][d] = (int16_t)r;
        // (W - r) / 2^10: exact, W - r >= 0
        W = r >= 0 ? u_shr(u_sub_small(W, (uint32_t)r), 10) : u_shr(u_add(W, u_from((uint32_t)-r)), 10);
        d++;
      }
      T = std::max(T, d);
    }
    k.T = std::min(T, OS2_CRT_DIGITS + 1);  // > OS2_CRT_DIGITS is rejected at launch
    const int LX = k.LX;
    const double Pd = u_to_double(P);
    for (int q = 1; q <= T; q++) {  // top digits that fix q to within 2^-11
      k.Q = q;
      if (255.0 * 512.0 * N * ldexp(1.0, 10 * (T - q)) * 1.001 / Pd <= ldexp(1.0, -11)) break;
    }
    U256 C0 = {};
    for (int tt = 0; tt < T && tt < OS2_CRT_DIGITS; tt++) {
      long long sumw = 0;
      for (int l = 0; l < N; l++) sumw += k.wd[l][tt];
      k.rmag[tt] = 12582912.0f - 1024.0f * (float)sumw;  // exact: a multiple of 1024 below 2^25
      k.pw[tt] = 1u << ((10 * tt) & 31);
      if (10 * tt < 32 * LX) C0 = u_add(C0, u_shl(u_from(0x4B400000u), 10 * tt));
    }
    const U256 negc = u_neg(u_add(C0, u_from(128)));
    const U256 np = u_neg(P);
    for (int v = 0; v < 5; v++) {
      k.negc[v] = v < LX ? negc.w[v] : 0;
      k.np[v] = v < LX ? np.w[v] : 0;
      k.P32[v] = P.w[v];
      k.H32[v] = half.w[v];
    }
    for (int j = 0; j < k.Q && j < OS2_CRT_DIGITS; j++)
      k.s[j] = (float)(ldexp(1.0, 10 * (T - 1 - j)) / Pd);
    k.c0 = (float)(-128.0 / Pd);
  }
  const int LW = (N + 3) / 4;
  const double Pd = u_to_double(P);
  t->crt.s_top = (float)(ldexp(1.0, 32 * (LW - 1)) / Pd);
  t->crt.s_next = (float)(LW > 1 ? ldexp(1.0, 32 * (LW - 2)) / Pd : 0.0);
  t->crt.s128 = (float)(128.0 / Pd);
  for (int i = 0; i < OS2_H_LIMBS; i++) t->res.H[i] = H.w[i];
  t->res.bitlenH = u_bitlen(H);
  {
    const int bH = t->res.bitlenH;
    auto bit = [&](int i) { return i >= 0 ? (H.w[i >> 5] >> (i & 31)) & 1u : 0u; };
    unsigned long long w = 0;
    for (int i = 0; i < 64; i++) w = (w << 1) | bit(bH - 1 - i);
    int rest = 0;
    for (int i = 0; i < bH - 64; i++) rest |= (int)bit(i);
    t->res.H64 = w;
    t->res.Hrest = rest;
  }
}

std::atomic<int> g_variant{OS2_GEMM_TC};
std::atomic<int> g_crt_variant{OS2_CRT_AUTO};

// The int8-plane step-3 kernels read int8 residue planes (step 2 writes them so).
bool planes_i8() {
  const int v = g_variant.load();
  return v == OS2_GEMM_TC_I8 || v == OS2_GEMM_S8_SYNC;
}

// Optional per-kernel timing: CUDA events recorded on the launching stream
// around every kernel that os2_gemm enqueues (no synchronisation added).
struct ProfRec {
  const char *name;
  cudaEvent_t a, b;
};
std::mutex g_prof_mu;
std::vector<ProfRec> g_prof;
std::atomic<bool> g_prof_on{false};

struct ProfScope {
  const char *name;
  cudaStream_t s;
  cudaEvent_t a = nullptr;
  ProfScope(const char *n, cudaStream_t st) : name(n), s(st) {
    if (g_prof_on.load() && cudaEventCreate(&a) == cudaSuccess) cudaEventRecord(a, s);
  }
  ~ProfScope() {
    cudaEvent_t b = nullptr;
    if (a && cudaEventCreate(&b) == cudaSuccess) {
      cudaEventRecord(b, s);
      std::lock_guard<std::mutex> g(g_prof_mu);
      g_prof.push_back({name, a, b});
    }
  }
};

}  // namespace

const Os2Tables *os2_tables(int N) {
  static Os2Tables tabs[OS2_MAX_MODULI + 1];
  static std::once_flag once;
  if (N < 1 || N > OS2_MAX_MODULI) return nullptr;
  std::call_once(once, [] {
    for (int n = 1; n <= OS2_MAX_MODULI; n++) build_tables(n, &tabs[n]);
  });
  return &tabs[N];
}

// ---------------------------------------------------------------------------
// Workspace layout
// ---------------------------------------------------------------------------
namespace {

// Inner-dimension limits.  Step 3 reduces every 960-term block mod p inside
// tensor memory, so the mod-p path has no INT32 limit; the remaining limits
// are the fast-mode sums (exact for k < 2^26 per thread partial, kept well
// inside), the accurate-mode bound product (int32 sums of 64*64*k < 2^31) and
// raw int32 products (128*128*k < 2^31).
constexpr int kMaxK = 1 << 24;
constexpr int kMaxKAccurate = 1 << 19;
constexpr int kMaxKRaw = 1 << 17;

struct Layout {
  size_t e, f, EA, EB, R, K, planesA, planesB, cres, total;
  int kp, ldcres;
};

bool make_layout(int m, int n, int k, int N, int mode, Layout *L) {
  if (m < 0 || n < 0 || k < 0 || N < 1 || N > OS2_MAX_MODULI) return false;
  if (mode != OS2_MODE_FAST && mode != OS2_MODE_ACCURATE) return false;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += os2_round_up(bytes, 256);
    return o;
  };
  L->kp = (int)os2_round_up((size_t)std::max(k, 1), OS2_KP_ALIGN);
  L->ldcres = (int)os2_round_up((size_t)std::max(n, 1), OS2_CRES_ALIGN);
  L->e = take(4 * (size_t)m);
  L->f = take(4 * (size_t)n);
  if (mode == OS2_MODE_ACCURATE) {
    L->EA = take(4 * (size_t)m);
    L->EB = take(4 * (size_t)n);
    L->R = take(4 * (size_t)m);
    L->K = take(4 * (size_t)n);
  } else {
    L->EA = L->EB = L->R = L->K = 0;
  }
  L->planesA = take((size_t)N * m * L->kp * 2);
  L->planesB = take((size_t)N * n * L->kp * 2);
  L->cres = take((size_t)N * m * L->ldcres);
  L->total = off;
  return true;
}

os2_status cuda_status(cudaError_t e) { return e == cudaSuccess ? OS2_OK : OS2_ERR_CUDA; }

// Steps 4 + 5 on the selected kernel: the tensor-core one needs 16-byte rows
// of the product residues (always so inside the library).  AUTO takes it for
// a reconstruction that runs alone; `beside` marks one that runs beside a
// product (row panels, host-path blocks), which takes the CUDA-core kernel.
bool crt_on_tc(int ldcres, const void *c, bool beside = false) {
  const int v = g_crt_variant.load();
  return (v == OS2_CRT_TC || (v == OS2_CRT_AUTO && !beside)) && ldcres % 16 == 0 &&
         (reinterpret_cast<uintptr_t>(c) & 15) == 0;
}
cudaError_t crt_launch(bool f32, int m, int n, const int8_t *c, int ldcres, const int32_t *e,
                       const int32_t *f, void *C, int ldc, uint32_t *X_out, const Os2Tables *t,
                       int *status, cudaStream_t s, bool beside = false) {
  if (crt_on_tc(ldcres, c, beside))
    return launch_crt_tc(f32, m, n, c, ldcres, e, f, C, ldc, X_out, t, status, s);
  return launch_crt(f32, m, n, c, ldcres, e, f, C, ldc, X_out, t, s, status);
}

template <typename T>
T *at(void *ws, size_t off) {
  return reinterpret_cast<T *>(static_cast<char *>(ws) + off);
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

os2_status check_gemm_args(int m, int n, int k, const void *A, int lda, const void *B, int ldb,
                           const void *C, int ldc, int N, int mode, size_t esize = 8) {
  if (m < 0 || n < 0 || k < 0) return OS2_ERR_INVALID_ARG;
  if (N < 1 || N > OS2_MAX_MODULI) return OS2_ERR_INVALID_ARG;
  if (mode != OS2_MODE_FAST && mode != OS2_MODE_ACCURATE) return OS2_ERR_INVALID_ARG;
  if (lda < std::max(k, 1) || ldb < std::max(k, 1) || ldc < std::max(n, 1))
    return OS2_ERR_INVALID_ARG;
  if (k >= kMaxK || (mode == OS2_MODE_ACCURATE && k >= kMaxKAccurate)) return OS2_ERR_UNSUPPORTED;
  if (m > 0 && n > 0 && !C) return OS2_ERR_INVALID_ARG;
  if (m > 0 && k > 0 && !A) return OS2_ERR_INVALID_ARG;
  if (n > 0 && k > 0 && !B) return OS2_ERR_INVALID_ARG;
  if ((A && !aligned(A, esize)) || (B && !aligned(B, esize)) || (C && !aligned(C, esize)))
    return OS2_ERR_INVALID_ARG;
  return OS2_OK;
}

// The exact bound product of accurate mode with fused row/column maxima into
// R, K (zeroed): on the 2-SM kernel when it is the selected step-3 kernel and
// either k fits one 4096-term segment or the product-residue region of the
// workspace (unused during step 1) can hold the int32 partial sums; else on
// the single-SM kernel, which sums its segments in registers.
bool bound_on_2sm(int m, const Layout &L) {
  const int segs = (L.kp + 4095) / 4096;
  const bool room = L.total - L.cres >= 4 * (size_t)m * (size_t)L.ldcres;
  const int v = g_variant.load();
  return (v == OS2_GEMM_TC || v == OS2_GEMM_TC_I8 || v == OS2_GEMM_S8_SYNC) &&
         (segs == 1 || room);
}

// Kernel launches of bound_product.
int bound_launches(int m, int, const Layout &L) {
  return bound_on_2sm(m, L) ? (L.kp + 4095) / 4096 : 1;
}

cudaError_t bound_product(int m, int n, const Layout &L, void *ws, const void *pa, const void *pb,
                          int32_t *R, int32_t *K, const Os2Tables *t, int *status,
                          cudaStream_t s) {
  if (bound_on_2sm(m, L))
    return launch_gemm_bound2(m, n, L.kp, pa, pb, at<int32_t>(ws, L.cres), L.ldcres, R, K, status,
                              s);
  return launch_gemm_tc(1, m, n, L.kp, pa, pb, 1, nullptr, 0, R, K, 12, t, status, s);
}

// Step 1 in accurate mode: magnitude planes (aliasing the residue planes), one
// exact bound product with fused row/column maxima, then the exponents e, f.
os2_status accurate_exponents(bool f32, int m, int n, int k, const void *A, int lda, const void *B,
                              int ldb, void *ws, const Layout &L, const Os2Tables *t, int *status,
                              cudaStream_t s) {
  int32_t *e = at<int32_t>(ws, L.e), *f = at<int32_t>(ws, L.f);
  void *pa = at<void>(ws, L.planesA), *pb = at<void>(ws, L.planesB);
  int32_t *EA = at<int32_t>(ws, L.EA), *EB = at<int32_t>(ws, L.EB);
  int32_t *R = at<int32_t>(ws, L.R), *K = at<int32_t>(ws, L.K);
  cudaError_t err;
  {
    ProfScope ps("scale_bars", s);
    if ((err = launch_row_scale(SM_BARS, f32, A, lda, m, nullptr, EA, pa, B, ldb, n, nullptr, EB,
                                pb, k, L.kp, t, status, s)))
      return cuda_status(err);
  }
  if ((err = cudaMemsetAsync(R, 0, 4 * (size_t)m, s))) return cuda_status(err);
  if ((err = cudaMemsetAsync(K, 0, 4 * (size_t)n, s))) return cuda_status(err);
  {
    ProfScope ps("gemm_bound", s);
    if ((err = bound_product(m, n, L, ws, pa, pb, R, K, t, status, s))) return cuda_status(err);
  }
  if ((err = launch_accu_exponents(R, EA, m, e, t, s))) return cuda_status(err);
  return cuda_status(launch_accu_exponents(K, EB, n, f, t, s));
}

// Step 3 for an m x n block: A planes [N][m][kp] and B planes [N][n][kp] give
// the mod-p products [N][m][ldcres].
os2_status residue_products(int m, int n, const Layout &L, const void *pa, const void *pb, int N,
                            int8_t *cres, const Os2Tables *t, int *status, cudaStream_t s) {
  ProfScope ps("gemm_modp", s);
  const int variant = g_variant.load();
  cudaError_t err;
  if (variant == OS2_GEMM_SIMT)
    err = launch_gemm_simt(m, n, L.kp, pa, pb, N, OS2_OUT_MODP_INT8, cres, L.ldcres, t, s);
  else if (variant == OS2_GEMM_S8_SYNC)
    err = launch_gemm_s8(m, n, L.kp, pa, pb, N, OS2_OUT_MODP_INT8, cres, L.ldcres, t, status, s);
  else
    err = launch_gemm_tc(variant == OS2_GEMM_TC_1SM ? 0 : (variant == OS2_GEMM_TC_I8 ? 3 : 2), m, n, L.kp, pa, pb, N, cres,
                         L.ldcres, nullptr, nullptr, 14, t, status, s);
  return cuda_status(err);
}

// Panels of rows (of A) or columns (of B) for the pipelined paths.
constexpr int kMaxPanels = 8;
constexpr int kPanelMinRows = 2048;

// Panel size along one dimension: at least kPanelMinRows, a multiple of the
// 256-row tile of step 3, at most kMaxPanels panels.
int panel_size(int rows) {
  const int P = std::min(kMaxPanels, std::max(1, rows / kPanelMinRows));
  return (int)os2_round_up((size_t)((rows + P - 1) / P), 256);
}

// The five steps on device operands; arguments already checked.  f32: float
// operands and result (SGEMM emulation), else double.
// Step 1 from exponents the caller already has (e_in for A's m rows, f_in for
// B's n columns): copied into the workspace.
cudaError_t given_exponents(int m, int n, const int32_t *e_in, const int32_t *f_in, void *ws,
                            const Layout &L, cudaStream_t s) {
  cudaError_t err = cudaMemcpyAsync(at<int32_t>(ws, L.e), e_in, 4 * (size_t)m,
                                    cudaMemcpyDeviceToDevice, s);
  if (err) return err;
  return cudaMemcpyAsync(at<int32_t>(ws, L.f), f_in, 4 * (size_t)n, cudaMemcpyDeviceToDevice, s);
}

os2_status run_gemm(bool f32, int m, int n, int k, const void *A, int lda, const void *B, int ldb,
                    void *C, int ldc, int N, int mode, void *ws, const Layout &L, cudaStream_t s,
                    const int32_t *e_in = nullptr, const int32_t *f_in = nullptr) {
  const size_t es = f32 ? 4 : 8;
  if (m == 0 || n == 0) return OS2_OK;
  if (k == 0) return cuda_status(cudaMemset2DAsync(C, (size_t)ldc * es, 0, (size_t)n * es, m, s));
  const Os2Tables *t = os2_tables(N);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  int32_t *e = at<int32_t>(ws, L.e), *f = at<int32_t>(ws, L.f);
  void *pa = at<void>(ws, L.planesA), *pb = at<void>(ws, L.planesB);
  int8_t *cres = at<int8_t>(ws, L.cres);
  cudaError_t err;
  if (e_in) {
    if ((err = given_exponents(m, n, e_in, f_in, ws, L, s))) return cuda_status(err);
  } else if (mode == OS2_MODE_FAST) {
    // step 1: exponents from the revised bound (A's rows and B's columns)
    ProfScope ps("scale", s);
    if ((err = launch_row_scale(SM_FAST_SCALE, f32, A, lda, m, e, nullptr, nullptr, B, ldb, n, f,
                                nullptr, nullptr, k, L.kp, t, status, s)))
      return cuda_status(err);
  } else {
    os2_status st = accurate_exponents(f32, m, n, k, A, lda, B, ldb, ws, L, t, status, s);
    if (st) return st;
  }
  // step 2: residue planes of A and B
  {
    ProfScope ps("residues", s);
    if ((err = launch_residues(f32, A, lda, m, e, pa, B, ldb, n, f, pb, k, L.kp, t, s, 0,
                               planes_i8())))
      return cuda_status(err);
  }
  // step 3
  os2_status st = residue_products(m, n, L, pa, pb, N, cres, t, status, s);
  if (st) return st;
  // steps 4 + 5
  ProfScope ps("crt_unscale", s);
  return cuda_status(crt_launch(f32, m, n, cres, L.ldcres, e, f, C, ldc, nullptr, t, status, s));
}

// Device-path pipeline.  Step 3 fills every SM with one persistent CTA that
// holds most of the shared memory but few threads and registers, so the CUDA
// cores are nearly idle while it runs; a CRT CTA needs no shared memory and
// fits beside it.  With A cut into row panels, the CRT and unscaling of panel
// i-1 run on a side stream, on those idle units, while panel i is multiplied
// on the caller's stream.  (Running the residues of the next panel beside the
// product as well was measured no faster: they contend with it for memory.)
struct DevPipe {
  cudaStream_t crt = nullptr;
  cudaEvent_t done = nullptr;
  cudaEvent_t g_done[kMaxPanels] = {};
  bool ready = false;
};

std::mutex g_dev_mu;  // held while a call enqueues (its events are shared)

DevPipe *dev_pipe() {
  static DevPipe pipes[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  DevPipe &p = pipes[dev];
  if (p.ready) return &p;
  bool ok = cudaStreamCreateWithFlags(&p.crt, cudaStreamNonBlocking) == cudaSuccess;
  auto ev = [&](cudaEvent_t *x) {
    ok = ok && cudaEventCreateWithFlags(x, cudaEventDisableTiming) == cudaSuccess;
  };
  ev(&p.done);
  for (int i = 0; i < kMaxPanels; i++) ev(&p.g_done[i]);
  p.ready = ok;
  return ok ? &p : nullptr;
}

// The five steps with A in row panels (m, n, k > 0; arguments checked).  The
// results are those of run_gemm: every entry goes through the same steps.
os2_status run_gemm_panels(bool f32, int m, int n, int k, const void *A, int lda, const void *B,
                           int ldb, void *C, int ldc, int N, int mode, void *ws, const Layout &L,
                           cudaStream_t s, const int32_t *e_in = nullptr,
                           const int32_t *f_in = nullptr) {
  const size_t es = f32 ? 4 : 8;
  const Os2Tables *t = os2_tables(N);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_dev_mu);
  DevPipe *p = dev_pipe();
  if (!p) return OS2_ERR_CUDA;
  const int mp = panel_size(m), P = (m + mp - 1) / mp;
  int32_t *e = at<int32_t>(ws, L.e), *f = at<int32_t>(ws, L.f);
  char *pa = at<char>(ws, L.planesA);
  void *pb = at<void>(ws, L.planesB);
  int8_t *cres = at<int8_t>(ws, L.cres);
  const size_t plane_row = (size_t)L.kp * (planes_i8() ? 1 : 2);  // bytes of one plane row
  const char *Ab = static_cast<const char *>(A);
  char *Cb = static_cast<char *>(C);
  cudaError_t err;
#define OS2_TRY(x)                                           \
  do {                                                       \
    if ((err = (x)) != cudaSuccess) return cuda_status(err); \
  } while (0)
  // step 1 on `stream`
  if (e_in) {
    OS2_TRY(given_exponents(m, n, e_in, f_in, ws, L, s));
  } else if (mode == OS2_MODE_FAST) {
    ProfScope ps("scale", s);
    OS2_TRY(launch_row_scale(SM_FAST_SCALE, f32, A, lda, m, e, nullptr, nullptr, B, ldb, n, f,
                             nullptr, nullptr, k, L.kp, t, status, s));
  } else {
    os2_status st = accurate_exponents(f32, m, n, k, A, lda, B, ldb, ws, L, t, status, s);
    if (st) return st;
  }
  // step 2, row panel by row panel (each panel's planes laid out as an mi-row
  // problem), B's with the first
  {
    ProfScope ps("residues", s);
    for (int i = 0; i < P; i++) {
      const int r0 = i * mp, mi = std::min(mp, m - r0);
      OS2_TRY(launch_residues(f32, Ab + (size_t)r0 * lda * es, lda, mi, e + r0,
                              pa + (size_t)r0 * N * plane_row, B, ldb, i == 0 ? n : 0, f, pb, k,
                              L.kp, t, s, 0, planes_i8()));
    }
  }
  // step 3 per panel on `stream`; steps 4 + 5 per panel on side stream 2
  for (int i = 0; i < P; i++) {
    const int r0 = i * mp, mi = std::min(mp, m - r0);
    int8_t *ci = cres + (size_t)r0 * N * L.ldcres;
    os2_status st =
        residue_products(mi, n, L, pa + (size_t)r0 * N * plane_row, pb, N, ci, t, status, s);
    if (st) return st;
    OS2_TRY(cudaEventRecord(p->g_done[i], s));
    OS2_TRY(cudaStreamWaitEvent(p->crt, p->g_done[i], 0));
    ProfScope ps("crt_unscale", p->crt);
    // the last panel's reconstruction has no product left beside it
    OS2_TRY(crt_launch(f32, mi, n, ci, L.ldcres, e + r0, f, Cb + (size_t)r0 * ldc * es, ldc,
                       nullptr, t, status, p->crt, i + 1 < P));
  }
  // `stream` covers everything: it waits for the last reconstruction
  OS2_TRY(cudaEventRecord(p->done, p->crt));
  OS2_TRY(cudaStreamWaitEvent(s, p->done, 0));
#undef OS2_TRY
  return OS2_OK;
}

// Row panels pay only with the CUDA-core CRT, which runs on the units the
// product leaves idle.  The tensor-core CRT needs TMEM and more shared memory
// than a product CTA leaves free, so it cannot run beside a product: with it
// the five steps run in one pass (one product launch, no panel tails).
// Measured at 8192^3 the two plans tie at 16 moduli, and the panels win at 18
// (the tensor-core CRT then takes 1.0 ms in series), so AUTO takes panels.
bool use_panels(int m) { return panel_size(m) < m && g_crt_variant.load() != OS2_CRT_TC; }

// run_gemm_panels when A has more than one row panel, else run_gemm.
os2_status run_gemm_auto(bool f32, int m, int n, int k, const void *A, int lda, const void *B,
                         int ldb, void *C, int ldc, int N, int mode, void *ws, const Layout &L,
                         cudaStream_t s, const int32_t *e_in = nullptr,
                         const int32_t *f_in = nullptr) {
  if (m > 0 && n > 0 && k > 0 && use_panels(m))
    return run_gemm_panels(f32, m, n, k, A, lda, B, ldb, C, ldc, N, mode, ws, L, s, e_in, f_in);
  return run_gemm(f32, m, n, k, A, lda, B, ldb, C, ldc, N, mode, ws, L, s, e_in, f_in);
}

}  // namespace

// ---------------------------------------------------------------------------
// C ABI
// ---------------------------------------------------------------------------
extern "C" {

size_t os2_workspace_size(int m, int n, int k, int num_moduli, int mode) {
  Layout L;
  return make_layout(m, n, k, num_moduli, mode, &L) ? L.total : 0;
}

os2_status os2_gemm(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                    double *C, int ldc, int num_moduli, int mode, void *workspace,
                    size_t workspace_bytes, void *stream) {
  os2_status st = check_gemm_args(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode);
  if (st) return st;
  Layout L;
  make_layout(m, n, k, num_moduli, mode, &L);
  if (m > 0 && n > 0 && k > 0) {
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256))
      return OS2_ERR_WORKSPACE;
  }
  return run_gemm_auto(false, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, workspace, L,
                       static_cast<cudaStream_t>(stream));
}

os2_status os2_sgemm(int m, int n, int k, const float *A, int lda, const float *B, int ldb,
                     float *C, int ldc, int num_moduli, int mode, void *workspace,
                     size_t workspace_bytes, void *stream) {
  os2_status st = check_gemm_args(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, 4);
  if (st) return st;
  Layout L;
  make_layout(m, n, k, num_moduli, mode, &L);
  if (m > 0 && n > 0 && k > 0) {
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256))
      return OS2_ERR_WORKSPACE;
  }
  return run_gemm_auto(true, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, workspace, L,
                  static_cast<cudaStream_t>(stream));
}

// Complex products: the real workspace of the stacked m x 2n x 2k product,
// then A2 (m x 2k), Bt2 (2n x 2k) and C2 (m x 2n) in the element type.
static bool complex_layout(int m, int n, int k, int N, int mode, size_t es, Layout *L,
                           size_t *offA2, size_t *offB2, size_t *offC2, size_t *total) {
  if (m < 0 || n < 0 || k < 0 || n > (1 << 30) || k > (1 << 30)) return false;
  if (!make_layout(m, 2 * n, 2 * k, N, mode, L)) return false;
  *offA2 = L->total;
  *offB2 = *offA2 + os2_round_up(es * (size_t)m * 2 * k, 256);
  *offC2 = *offB2 + os2_round_up(es * (size_t)2 * n * 2 * k, 256);
  *total = *offC2 + os2_round_up(es * (size_t)m * 2 * n, 256);
  return true;
}

static os2_status complex_gemm(bool f32, int m, int n, int k, const void *A, int lda,
                               const void *B, int ldb, void *C, int ldc, int N, int mode,
                               void *ws, size_t wsb, cudaStream_t s) {
  const size_t es = f32 ? 4 : 8;
  if (m < 0 || n < 0 || k < 0 || lda < std::max(k, 1) || ldb < std::max(k, 1) ||
      ldc < std::max(n, 1))
    return OS2_ERR_INVALID_ARG;
  // the stacked product has inner dimension 2k
  os2_status st = check_gemm_args(m, 2 * n, 2 * k, A, 2 * lda, B, 2 * ldb, C, 2 * ldc, N, mode, es);
  if (st) return st;
  Layout L;
  size_t oA, oB, oC, total;
  if (!complex_layout(m, n, k, N, mode, es, &L, &oA, &oB, &oC, &total)) return OS2_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OS2_OK;
  if (!ws || wsb < total || !aligned(ws, 256)) return OS2_ERR_WORKSPACE;
  void *A2 = at<char>(ws, oA), *B2 = at<char>(ws, oB), *C2 = at<char>(ws, oC);
  cudaError_t err;
  {
    ProfScope ps("complex_stack", s);
    if ((err = launch_complex_stack(f32, m, n, k, A, lda, B, ldb, A2, B2, s))) return cuda_status(err);
  }
  st = run_gemm_auto(f32, m, 2 * n, 2 * k, A2, std::max(2 * k, 1), B2, std::max(2 * k, 1), C2,
                2 * n, N, mode, ws, L, s);
  if (st) return st;
  ProfScope ps("complex_unstack", s);
  return cuda_status(launch_complex_unstack(f32, m, n, C2, C, ldc, s));
}

size_t os2_complex_workspace_size(int m, int n, int k, int num_moduli, int mode, int single) {
  Layout L;
  size_t a, b, c, total;
  return complex_layout(m, n, k, num_moduli, mode, single ? 4 : 8, &L, &a, &b, &c, &total) ? total
                                                                                          : 0;
}

os2_status os2_zgemm(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                     double *C, int ldc, int num_moduli, int mode, void *workspace,
                     size_t workspace_bytes, void *stream) {
  return complex_gemm(false, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

os2_status os2_cgemm(int m, int n, int k, const float *A, int lda, const float *B, int ldb,
                     float *C, int ldc, int num_moduli, int mode, void *workspace,
                     size_t workspace_bytes, void *stream) {
  return complex_gemm(true, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, workspace,
                      workspace_bytes, static_cast<cudaStream_t>(stream));
}

size_t os2_host_workspace_size(int m, int n, int k, int num_moduli, int mode) {
  Layout L;
  if (!make_layout(m, n, k, num_moduli, mode, &L)) return 0;
  return L.total + os2_round_up(8 * (size_t)m * k, 256) + os2_round_up(8 * (size_t)n * k, 256) +
         os2_round_up(8 * (size_t)m * n, 256);
}

// Copy of a rows x cols block of doubles (one 1-D copy when both are contiguous).
static cudaError_t copy_rows(double *dst, size_t dpitch, const double *src, size_t spitch,
                             size_t cols, size_t rows, cudaMemcpyKind kind, cudaStream_t s) {
  if (rows == 0 || cols == 0) return cudaSuccess;
  if (dpitch == cols && spitch == cols)
    return cudaMemcpyAsync(dst, src, 8 * cols * rows, kind, s);
  return cudaMemcpy2DAsync(dst, 8 * dpitch, src, 8 * spitch, 8 * cols, rows, kind, s);
}

}  // extern "C"

namespace {

// Host entry point pipeline.  Row panel i of C needs A's row panel i and all
// of B; a block (row panel, column panel) needs only the two panels.  The
// operands travel on a copy-in stream in the order A_0, B_0 .. B_{Q-1}, A_1 ..
// A_{P-1}; the caller's stream scales, splits and multiplies each block as
// soon as its panels have arrived, while later panels are still in transit; a
// CRT stream reconstructs each block beside the next block's product (see the
// device-path pipeline), and each finished block of C leaves on a copy-out
// stream.  The first and last row panels go block by block
// (a short head before the first product, a short tail after the last); the
// middle row panels go whole.  Accurate mode's exponents need all of A and all
// of B, so there the compute waits for every panel; C still leaves by blocks.

struct HostPipe {
  cudaStream_t in = nullptr, out = nullptr, crt = nullptr, res = nullptr;
  cudaEvent_t start = nullptr, out_done = nullptr;
  cudaEvent_t a_in[kMaxPanels] = {}, b_in[kMaxPanels] = {};
  cudaEvent_t a_split[kMaxPanels] = {}, b_split[kMaxPanels] = {};
  cudaEvent_t g_done[3 * kMaxPanels] = {}, c_done[3 * kMaxPanels] = {};
  bool ready = false;
};

std::mutex g_host_mu;  // held while a call enqueues (its events are shared)

// Streams and events of the pipeline on the current device, created once.
HostPipe *host_pipe() {
  static HostPipe pipes[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  HostPipe &p = pipes[dev];
  if (p.ready) return &p;
  bool ok = cudaStreamCreateWithFlags(&p.in, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.out, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.crt, cudaStreamNonBlocking) == cudaSuccess &&
            cudaStreamCreateWithFlags(&p.res, cudaStreamNonBlocking) == cudaSuccess;
  auto ev = [&](cudaEvent_t *x) {
    ok = ok && cudaEventCreateWithFlags(x, cudaEventDisableTiming) == cudaSuccess;
  };
  ev(&p.start);
  ev(&p.out_done);
  for (int i = 0; i < kMaxPanels; i++) {
    ev(&p.a_in[i]);
    ev(&p.b_in[i]);
    ev(&p.a_split[i]);
    ev(&p.b_split[i]);
  }
  for (int i = 0; i < 3 * kMaxPanels; i++) {
    ev(&p.g_done[i]);
    ev(&p.c_done[i]);
  }
  p.ready = ok;
  return ok ? &p : nullptr;
}

}  // namespace

extern "C" {

os2_status os2_gemm_host(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                         double *C, int ldc, int num_moduli, int mode, void *workspace,
                         size_t workspace_bytes, void *stream) {
  os2_status st = check_gemm_args(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode);
  if (st) return st;
  Layout L;
  make_layout(m, n, k, num_moduli, mode, &L);
  const size_t need = os2_host_workspace_size(m, n, k, num_moduli, mode);
  if (m == 0 || n == 0) return OS2_OK;
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return OS2_ERR_WORKSPACE;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  double *dA = at<double>(workspace, L.total);
  double *dB = at<double>(workspace, L.total + os2_round_up(8 * (size_t)m * k, 256));
  double *dC = at<double>(workspace, L.total + os2_round_up(8 * (size_t)m * k, 256) +
                                          os2_round_up(8 * (size_t)n * k, 256));
  cudaError_t err;
  if (k == 0) {
    if ((err = cudaMemsetAsync(dC, 0, 8 * (size_t)m * n, s))) return cuda_status(err);
    return cuda_status(copy_rows(C, ldc, dC, n, n, m, cudaMemcpyDeviceToHost, s));
  }
  const int N = num_moduli;
  const Os2Tables *t = os2_tables(N);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  std::lock_guard<std::mutex> g(g_host_mu);
  HostPipe *p = host_pipe();
  if (!p) return OS2_ERR_CUDA;
  const int mp = panel_size(m), P = (m + mp - 1) / mp;
  // column panels of B (the tensor-core step 3 reads a panel of B's planes in
  // place; the CUDA-core reference variant takes B whole)
  const int nq = g_variant.load() == OS2_GEMM_SIMT ? n : panel_size(n), Q = (n + nq - 1) / nq;
  int32_t *e = at<int32_t>(workspace, L.e), *f = at<int32_t>(workspace, L.f);
  char *pa = at<char>(workspace, L.planesA), *pb = at<char>(workspace, L.planesB);
  int8_t *cres = at<int8_t>(workspace, L.cres);
  const size_t plane_row = (size_t)L.kp * (planes_i8() ? 1 : 2);  // bytes of one plane row
#define OS2_TRY(x)                                           \
  do {                                                       \
    if ((err = (x)) != cudaSuccess) return cuda_status(err); \
  } while (0)
  // both copy streams start after the work already enqueued on `stream`
  OS2_TRY(cudaEventRecord(p->start, s));
  OS2_TRY(cudaStreamWaitEvent(p->in, p->start, 0));
  OS2_TRY(cudaStreamWaitEvent(p->out, p->start, 0));
  auto send_a = [&](int i) {
    const int r0 = i * mp, mi = std::min(mp, m - r0);
    cudaError_t r = copy_rows(dA + (size_t)r0 * k, k, A + (size_t)r0 * lda, lda, k, mi,
                              cudaMemcpyHostToDevice, p->in);
    return r ? r : cudaEventRecord(p->a_in[i], p->in);
  };
  OS2_TRY(send_a(0));
  for (int j = 0; j < Q; j++) {
    const int c0 = j * nq, nj = std::min(nq, n - c0);
    OS2_TRY(copy_rows(dB + (size_t)c0 * k, k, B + (size_t)c0 * ldb, ldb, k, nj,
                      cudaMemcpyHostToDevice, p->in));
    OS2_TRY(cudaEventRecord(p->b_in[j], p->in));
  }
  for (int i = 1; i < P; i++) OS2_TRY(send_a(i));

  // Steps 1 + 2 of each panel ("splits").  Fast mode: on a split stream, each
  // as soon as its panel has arrived, so that a panel is scaled and split
  // while the previous block is multiplied.  Accurate mode: on `stream`, after
  // the exponents (which need all of A and B).
  const bool side = mode == OS2_MODE_FAST;
  cudaStream_t sp = side ? p->res : s;
  // row panel i of A (the panel's planes are laid out as an mi-row problem)
  auto split_a = [&](int i) {
    const int r0 = i * mp, mi = std::min(mp, m - r0);
    const double *Ai = dA + (size_t)r0 * k;
    cudaError_t r = cudaSuccess;
    if (side) {
      if ((r = cudaStreamWaitEvent(sp, p->a_in[i], 0))) return r;
      ProfScope ps("scale", sp);
      r = launch_row_scale(SM_FAST_SCALE, false, Ai, k, mi, e + r0, nullptr, nullptr, nullptr, 0,
                           0, nullptr, nullptr, nullptr, k, L.kp, t, status, sp);
      if (r) return r;
    }
    {
      ProfScope ps("residues", sp);
      r = launch_residues(false, Ai, k, mi, e + r0, pa + (size_t)r0 * N * plane_row, nullptr, 0,
                          0, nullptr, nullptr, k, L.kp, t, sp, 0, planes_i8());
    }
    return r ? r : (side ? cudaEventRecord(p->a_split[i], sp) : cudaSuccess);
  };
  // column panel j of B, in place in B's [N][n][kp] planes
  auto split_b = [&](int j) {
    const int c0 = j * nq, nj = std::min(nq, n - c0);
    const double *Bj = dB + (size_t)c0 * k;
    cudaError_t r = cudaSuccess;
    if (side) {
      if ((r = cudaStreamWaitEvent(sp, p->b_in[j], 0))) return r;
      ProfScope ps("scale", sp);
      r = launch_row_scale(SM_FAST_SCALE, false, nullptr, 0, 0, nullptr, nullptr, nullptr, Bj, k,
                           nj, f + c0, nullptr, nullptr, k, L.kp, t, status, sp);
      if (r) return r;
    }
    {
      ProfScope ps("residues", sp);
      r = launch_residues(false, nullptr, 0, 0, nullptr, nullptr, Bj, k, nj, f + c0,
                          pb + (size_t)c0 * plane_row, k, L.kp, t, sp, n, planes_i8());
    }
    return r ? r : (side ? cudaEventRecord(p->b_split[j], sp) : cudaSuccess);
  };
  // steps 3-5 for the block (row panel i, columns c0 .. c0+nj of column
  // panel j, or all columns when j < 0), then its copy out
  int blocks = 0;
  auto block = [&](int i, int j, int c0, int nj, bool last) -> os2_status {
    const int r0 = i * mp, mi = std::min(mp, m - r0);
    if (side) {
      // the split stream runs in arrival order: A_0, B_0 .. B_{Q-1}, A_1 ..
      if ((err = cudaStreamWaitEvent(s, p->a_split[i], 0))) return cuda_status(err);
      if (i == 0 && j >= 0 && (err = cudaStreamWaitEvent(s, p->b_split[j], 0)))
        return cuda_status(err);
    }
    const void *pai = pa + (size_t)r0 * N * plane_row;
    int8_t *ci = cres + (size_t)r0 * N * L.ldcres + c0;
    const char *pbj = pb + (size_t)c0 * plane_row;
    {
      ProfScope ps("gemm_modp", s);
      const int variant = g_variant.load();
      if (variant == OS2_GEMM_SIMT)
        err = launch_gemm_simt(mi, nj, L.kp, pai, pbj, N, OS2_OUT_MODP_INT8, ci, L.ldcres, t, s);
      else if (variant == OS2_GEMM_S8_SYNC)
        err = launch_gemm_s8(mi, nj, L.kp, pai, pbj, N, OS2_OUT_MODP_INT8, ci, L.ldcres, t,
                             status, s, n);
      else
        err = launch_gemm_tc(variant == OS2_GEMM_TC_1SM ? 0 : (variant == OS2_GEMM_TC_I8 ? 3 : 2), mi, nj, L.kp, pai, pbj, N, ci,
                             L.ldcres, nullptr, nullptr, 14, t, status, s, n);
      if (err) return cuda_status(err);
    }
    // the block's CRT: the CUDA-core kernel runs on the CRT stream beside the
    // next block's product; the tensor-core one follows the product on `stream`
    // (the last block has no product left beside it)
    cudaEvent_t gd = p->g_done[blocks], done = p->c_done[blocks];
    blocks++;
    const bool tc = crt_on_tc(L.ldcres, ci, !last);
    cudaStream_t cs = tc ? s : p->crt;
    if (!tc) {
      if ((err = cudaEventRecord(gd, s))) return cuda_status(err);
      if ((err = cudaStreamWaitEvent(p->crt, gd, 0))) return cuda_status(err);
    }
    {
      ProfScope ps("crt_unscale", cs);
      if ((err = crt_launch(false, mi, nj, ci, L.ldcres, e + r0, f + c0, dC + (size_t)r0 * n + c0,
                            n, nullptr, t, status, cs)))
        return cuda_status(err);
    }
    if ((err = cudaEventRecord(done, cs))) return cuda_status(err);
    if ((err = cudaStreamWaitEvent(p->out, done, 0))) return cuda_status(err);
    return cuda_status(copy_rows(C + (size_t)r0 * ldc + c0, ldc, dC + (size_t)r0 * n + c0, n, nj,
                                 mi, cudaMemcpyDeviceToHost, p->out));
  };
  auto row_panel = [&](int i, bool by_blocks) -> os2_status {
    if (!by_blocks) return block(i, -1, 0, n, i == P - 1);
    for (int j = 0; j < Q; j++) {
      const int c0 = j * nq;
      if ((st = block(i, j, c0, std::min(nq, n - c0), i == P - 1 && j == Q - 1))) return st;
    }
    return OS2_OK;
  };

  if (mode == OS2_MODE_ACCURATE) {
    OS2_TRY(cudaStreamWaitEvent(s, p->b_in[Q - 1], 0));
    OS2_TRY(cudaStreamWaitEvent(s, p->a_in[P - 1], 0));
    if ((st = accurate_exponents(false, m, n, k, dA, k, dB, k, workspace, L, t, status, s)))
      return st;
  }
  OS2_TRY(split_a(0));
  for (int j = 0; j < Q; j++) OS2_TRY(split_b(j));
  for (int i = 1; i < P; i++) OS2_TRY(split_a(i));
  for (int i = 0; i < P; i++)
    if ((st = row_panel(i, i == 0 || i == P - 1))) return st;
  // `stream` covers everything: it waits for the last copy out
  OS2_TRY(cudaEventRecord(p->out_done, p->out));
  OS2_TRY(cudaStreamWaitEvent(s, p->out_done, 0));
#undef OS2_TRY
  return OS2_OK;
}

os2_status os2_scale(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                     int num_moduli, int mode, int32_t *e, int32_t *f, void *workspace,
                     size_t workspace_bytes, void *stream) {
  if (m < 0 || n < 0 || k < 0) return OS2_ERR_INVALID_ARG;
  if (lda < std::max(k, 1) || ldb < std::max(k, 1)) return OS2_ERR_INVALID_ARG;
  if (num_moduli < 1 || num_moduli > OS2_MAX_MODULI) return OS2_ERR_INVALID_ARG;
  if (mode != OS2_MODE_FAST && mode != OS2_MODE_ACCURATE) return OS2_ERR_INVALID_ARG;
  if (k >= kMaxK) return OS2_ERR_UNSUPPORTED;
  if (mode == OS2_MODE_ACCURATE && k >= kMaxKAccurate) return OS2_ERR_UNSUPPORTED;
  if ((m && (!e || (k && !A))) || (n && (!f || (k && !B)))) return OS2_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Os2Tables *t = os2_tables(num_moduli);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  cudaError_t err;
  if (k == 0) {
    if (m && (err = cudaMemsetAsync(e, 0, 4 * (size_t)m, s))) return cuda_status(err);
    if (n && (err = cudaMemsetAsync(f, 0, 4 * (size_t)n, s))) return cuda_status(err);
    return OS2_OK;
  }
  if (mode == OS2_MODE_FAST)
    return cuda_status(launch_row_scale(SM_FAST_SCALE, false, A, lda, m, e, nullptr, nullptr, B,
                                        ldb, n, f, nullptr, nullptr, k, 0, t, status, s));
  Layout L;
  make_layout(m, n, k, 1, mode, &L);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256)) return OS2_ERR_WORKSPACE;
  int32_t *EA = at<int32_t>(workspace, L.EA), *EB = at<int32_t>(workspace, L.EB);
  int32_t *R = at<int32_t>(workspace, L.R), *K = at<int32_t>(workspace, L.K);
  void *pa = at<void>(workspace, L.planesA), *pb = at<void>(workspace, L.planesB);
  if ((err = launch_row_scale(SM_BARS, false, A, lda, m, nullptr, EA, pa, B, ldb, n, nullptr, EB,
                              pb, k, L.kp, t, status, s)))
    return cuda_status(err);
  if ((err = cudaMemsetAsync(R, 0, 4 * (size_t)std::max(m, 1), s))) return cuda_status(err);
  if ((err = cudaMemsetAsync(K, 0, 4 * (size_t)std::max(n, 1), s))) return cuda_status(err);
  if (m > 0 && n > 0 && (err = bound_product(m, n, L, workspace, pa, pb, R, K, t, status, s)))
    return cuda_status(err);
  if ((err = launch_accu_exponents(R, EA, m, e, t, s))) return cuda_status(err);
  return cuda_status(launch_accu_exponents(K, EB, n, f, t, s));
}

os2_status os2_scale_bounds(int m, int n, int k, const double *A, int lda, const double *B,
                            int ldb, int32_t *R, int32_t *K, int32_t *EA, int32_t *EB,
                            void *workspace, size_t workspace_bytes, void *stream) {
  if (m < 0 || n < 0 || k < 0) return OS2_ERR_INVALID_ARG;
  if (lda < std::max(k, 1) || ldb < std::max(k, 1)) return OS2_ERR_INVALID_ARG;
  if (k >= kMaxKAccurate) return OS2_ERR_UNSUPPORTED;
  if ((m && (!R || !EA || (k && !A))) || (n && (!K || !EB || (k && !B)))) return OS2_ERR_INVALID_ARG;
  if ((A && !aligned(A, 8)) || (B && !aligned(B, 8))) return OS2_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const Os2Tables *t = os2_tables(1);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  cudaError_t err;
  if (m && (err = cudaMemsetAsync(R, 0, 4 * (size_t)m, s))) return cuda_status(err);
  if (n && (err = cudaMemsetAsync(K, 0, 4 * (size_t)n, s))) return cuda_status(err);
  if (k == 0) {  // every row is zero: E = 0, bound 0
    if (m && (err = cudaMemsetAsync(EA, 0, 4 * (size_t)m, s))) return cuda_status(err);
    if (n && (err = cudaMemsetAsync(EB, 0, 4 * (size_t)n, s))) return cuda_status(err);
    return OS2_OK;
  }
  Layout L;
  make_layout(m, n, k, 1, OS2_MODE_ACCURATE, &L);
  if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256)) return OS2_ERR_WORKSPACE;
  void *pa = at<void>(workspace, L.planesA), *pb = at<void>(workspace, L.planesB);
  if ((err = launch_row_scale(SM_BARS, false, A, lda, m, nullptr, EA, pa, B, ldb, n, nullptr, EB,
                              pb, k, L.kp, t, status, s)))
    return cuda_status(err);
  if (m > 0 && n > 0 && (err = bound_product(m, n, L, workspace, pa, pb, R, K, t, status, s)))
    return cuda_status(err);
  return OS2_OK;
}

os2_status os2_exponents_from_bounds(int count, const int32_t *bound, const int32_t *E,
                                     int num_moduli, int32_t *e, void *stream) {
  if (count < 0 || num_moduli < 1 || num_moduli > OS2_MAX_MODULI) return OS2_ERR_INVALID_ARG;
  if (count == 0) return OS2_OK;
  if (!bound || !E || !e) return OS2_ERR_INVALID_ARG;
  const Os2Tables *t = os2_tables(num_moduli);
  if (!t) return OS2_ERR_CUDA;
  return cuda_status(launch_accu_exponents(bound, E, count, e, t, static_cast<cudaStream_t>(stream)));
}

os2_status os2_gemm_exponents(int m, int n, int k, const double *A, int lda, const double *B,
                              int ldb, double *C, int ldc, int num_moduli, const int32_t *e,
                              const int32_t *f, void *workspace, size_t workspace_bytes,
                              void *stream) {
  os2_status st = check_gemm_args(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, OS2_MODE_FAST);
  if (st) return st;
  if ((m > 0 && !e) || (n > 0 && !f)) return OS2_ERR_INVALID_ARG;
  Layout L;
  make_layout(m, n, k, num_moduli, OS2_MODE_FAST, &L);
  if (m > 0 && n > 0 && k > 0) {
    if (!workspace || workspace_bytes < L.total || !aligned(workspace, 256))
      return OS2_ERR_WORKSPACE;
  }
  return run_gemm_auto(false, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, OS2_MODE_FAST,
                       workspace, L, static_cast<cudaStream_t>(stream), e, f);
}

os2_status os2_residues(int rows, int k, const double *X, int ldx, const int32_t *exps,
                        int num_moduli, void *planes, int ldp, void *stream) {
  if (rows < 0 || k < 0 || ldx < std::max(k, 1)) return OS2_ERR_INVALID_ARG;
  if (num_moduli < 1 || num_moduli > OS2_MAX_MODULI) return OS2_ERR_INVALID_ARG;
  if (ldp < k || ldp % OS2_KP_ALIGN) return OS2_ERR_INVALID_ARG;
  if (k >= kMaxK) return OS2_ERR_UNSUPPORTED;
  if (rows == 0 || ldp == 0) return OS2_OK;
  if ((k && !X) || !exps || !planes || !aligned(planes, 16)) return OS2_ERR_INVALID_ARG;
  const Os2Tables *t = os2_tables(num_moduli);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  return cuda_status(launch_residues(false, X, ldx, rows, exps, planes, nullptr, 0, 0, nullptr,
                                     nullptr, k, ldp, t, static_cast<cudaStream_t>(stream)));
}

os2_status os2_gemm_residues(int m, int n, int k, const void *RA, const void *RB, int ldp,
                             int num_moduli, int out_kind, void *out, int ldo, int variant,
                             void *stream) {
  if (m < 0 || n < 0 || k < 0 || k > ldp || ldp % OS2_KP_ALIGN) return OS2_ERR_INVALID_ARG;
  if (num_moduli < 1 || num_moduli > OS2_MAX_MODULI) return OS2_ERR_INVALID_ARG;
  if (out_kind != OS2_OUT_MODP_INT8 && out_kind != OS2_OUT_RAW_INT32) return OS2_ERR_INVALID_ARG;
  if (variant != OS2_GEMM_TC && variant != OS2_GEMM_SIMT && variant != OS2_GEMM_TC_1SM &&
      variant != OS2_GEMM_S8_SYNC)
    return OS2_ERR_INVALID_ARG;  // (OS2_GEMM_TC_I8 widens int8 planes inside os2_gemm only)
  if (ldo < std::max(n, 1)) return OS2_ERR_INVALID_ARG;
  if (out_kind == OS2_OUT_MODP_INT8 && ldo % OS2_CRES_ALIGN) return OS2_ERR_INVALID_ARG;
  if (out_kind == OS2_OUT_RAW_INT32 && ldo % 4) return OS2_ERR_INVALID_ARG;
  if (ldp >= kMaxK || (out_kind == OS2_OUT_RAW_INT32 && k >= kMaxKRaw)) return OS2_ERR_UNSUPPORTED;
  if (m == 0 || n == 0) return OS2_OK;
  if (!out || !aligned(out, 16)) return OS2_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (ldp == 0) {
    const size_t es = out_kind == OS2_OUT_RAW_INT32 ? 4 : 1;
    return cuda_status(
        cudaMemsetAsync(out, 0, es * (size_t)num_moduli * m * ldo, s));
  }
  if (!RA || !RB || !aligned(RA, 16) || !aligned(RB, 16)) return OS2_ERR_INVALID_ARG;
  const Os2Tables *t = os2_tables(num_moduli);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  if (variant == OS2_GEMM_SIMT)
    return cuda_status(launch_gemm_simt(m, n, ldp, RA, RB, num_moduli, out_kind, out, ldo, t, s));
  if (variant == OS2_GEMM_S8_SYNC)  // int8 planes
    return cuda_status(
        launch_gemm_s8(m, n, ldp, RA, RB, num_moduli, out_kind, out, ldo, t, status, s));
  const int kind = out_kind == OS2_OUT_RAW_INT32 ? 1 : (variant == OS2_GEMM_TC_1SM ? 0 : 2);
  return cuda_status(launch_gemm_tc(kind, m, n, ldp, RA, RB, num_moduli, out, ldo, nullptr, nullptr,
                                    14, t, status, s));
}

os2_status os2_crt(int m, int n, const int8_t *c, int ldcres, int num_moduli, const int32_t *e,
                   const int32_t *f, double *C, int ldc, uint32_t *X_out, void *stream) {
  if (m < 0 || n < 0 || ldcres < std::max(n, 1) || ldcres % 4 || ldc < std::max(n, 1))
    return OS2_ERR_INVALID_ARG;
  if (num_moduli < 1 || num_moduli > OS2_MAX_MODULI) return OS2_ERR_INVALID_ARG;
  if (m == 0 || n == 0) return OS2_OK;
  if (!c || !e || !f || !C || !aligned(c, 4) || !aligned(C, 8)) return OS2_ERR_INVALID_ARG;
  const Os2Tables *t = os2_tables(num_moduli);
  int *status = os2_status_ptr();
  if (!t || !status) return OS2_ERR_CUDA;
  return cuda_status(crt_launch(false, m, n, c, ldcres, e, f, C, ldc, X_out, t, status,
                                static_cast<cudaStream_t>(stream)));
}

int os2_moduli(int num_moduli, int32_t *out) {
  if (num_moduli < 1 || num_moduli > OS2_MAX_MODULI || !out) return 0;
  for (int l = 0; l < num_moduli; l++) out[l] = kModuli[l];
  return num_moduli;
}

os2_status os2_wait_selftest(long long limit_cycles, int32_t *result, void *stream) {
  if (limit_cycles < 1 || limit_cycles > (1LL << 34)) return OS2_ERR_INVALID_ARG;
  int *status = os2_status_ptr();
  if (!status) return OS2_ERR_CUDA;
  return cuda_status(
      launch_wait_selftest(limit_cycles, status, result, static_cast<cudaStream_t>(stream)));
}

os2_status os2_get_status(void *stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return OS2_ERR_CUDA;
  int *p = os2_status_ptr();
  if (!p) return OS2_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, p, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return OS2_ERR_CUDA;
  if (v && cudaMemset(p, 0, sizeof(int)) != cudaSuccess) return OS2_ERR_CUDA;
  return static_cast<os2_status>(v);
}

os2_status os2_peak_probe(int kind, int iters, int check, int32_t *result, double *flop,
                          void *stream) {
  if (kind != OS2_PROBE_F16_1SM && kind != OS2_PROBE_F16_2SM && kind != OS2_PROBE_S8_SYNC)
    return OS2_ERR_INVALID_ARG;
  if (iters < 1 || iters > (1 << 24)) return OS2_ERR_INVALID_ARG;
  if (check && (!result || !aligned(result, 4))) return OS2_ERR_INVALID_ARG;
  if (check && kind == OS2_PROBE_S8_SYNC && iters > 4096) return OS2_ERR_INVALID_ARG;
  int *status = os2_status_ptr();
  if (!status) return OS2_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (check && (err = cudaMemsetAsync(result, 0, 4 * sizeof(int32_t), s))) return cuda_status(err);
  double fl = 0;
  err = launch_peak_probe(kind, iters, check ? 1 : 0, result, status, s, &fl);
  if (flop) *flop = fl;
  return cuda_status(err);
}

os2_status os2_set_crt_variant(int variant) {
  if (variant != OS2_CRT_TC && variant != OS2_CRT_SIMT && variant != OS2_CRT_AUTO)
    return OS2_ERR_INVALID_ARG;
  g_crt_variant.store(variant);
  return OS2_OK;
}

os2_status os2_set_gemm_variant(int variant) {
  if (variant != OS2_GEMM_TC && variant != OS2_GEMM_SIMT && variant != OS2_GEMM_TC_1SM &&
      variant != OS2_GEMM_TC_I8 && variant != OS2_GEMM_S8_SYNC)
    return OS2_ERR_INVALID_ARG;
  g_variant.store(variant);
  return OS2_OK;
}

const char *os2_status_string(int status) {
  switch (status) {
    case OS2_OK: return "ok";
    case OS2_ERR_INVALID_ARG: return "invalid argument";
    case OS2_ERR_UNSUPPORTED: return "unsupported size or configuration";
    case OS2_ERR_WORKSPACE: return "workspace missing, misaligned or too small";
    case OS2_ERR_NONFINITE: return "non-finite input entry";
    case OS2_ERR_RANGE: return "scaled integer out of range (|trunc(x 2^e)| >= 2^89)";
    case OS2_ERR_TIMEOUT: return "device-side wait timed out";
    case OS2_ERR_CUDA: return "CUDA error";
    case OS2_ERR_BOUNDS: return "index check failed (debug build)";
  }
  return "unknown status";
}

os2_status os2_profile_start(void) {
  std::lock_guard<std::mutex> g(g_prof_mu);
  for (auto &r : g_prof) {
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
  g_prof_on.store(true);
  return OS2_OK;
}

int os2_profile_stop(int max_kernels, char *names, double *total_ms, int *launches) {
  g_prof_on.store(false);
  std::lock_guard<std::mutex> g(g_prof_mu);
  std::vector<std::string> keys;
  std::vector<double> tot;
  std::vector<int> cnt;
  int bad = 0;
  for (auto &r : g_prof) {
    float ms = 0.f;
    if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&ms, r.a, r.b) != cudaSuccess)
      bad = 1;
    size_t i = 0;
    while (i < keys.size() && keys[i] != r.name) i++;
    if (i == keys.size()) {
      keys.push_back(r.name);
      tot.push_back(0.0);
      cnt.push_back(0);
    }
    tot[i] += ms;
    cnt[i] += 1;
    cudaEventDestroy(r.a);
    cudaEventDestroy(r.b);
  }
  g_prof.clear();
  if (bad) return -1;
  int n = 0;
  for (size_t i = 0; i < keys.size() && n < max_kernels; i++, n++) {
    if (names) {
      strncpy(names + 32 * n, keys[i].c_str(), 31);
      names[32 * n + 31] = 0;
    }
    if (total_ms) total_ms[n] = tot[i];
    if (launches) launches[n] = cnt[i];
  }
  return n;
}

int os2_gemm_launch_count(int m, int n, int k, int num_moduli, int mode) {
  if (m <= 0 || n <= 0 || k < 0 || num_moduli < 1 || num_moduli > OS2_MAX_MODULI) return 0;
  if (k == 0) return 0;
  // os2_gemm: step 1 (fast: 1 kernel; accurate: bars, the bound product,
  // two exponent kernels), then residues, product and CRT once per row panel
  const int P = use_panels(m) ? (m + panel_size(m) - 1) / panel_size(m) : 1;
  if (mode != OS2_MODE_ACCURATE) return 1 + 3 * P;
  Layout L;
  if (!make_layout(m, n, k, num_moduli, mode, &L)) return 0;
  return 3 + bound_launches(m, n, L) + 3 * P;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// os2_gemm_noalloc: os2_gemm for callers that cannot allocate device memory.
// Its scratch lives in one file-scope device array of fixed size; every GPU
// that loads this library holds that array until the process exits.
// ---------------------------------------------------------------------------
static __device__ __align__(256) unsigned char g_os2_noalloc_scratch[OS2_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array on the current device, looked up once
// per device with that device current.  In host code the array's name is
// only a host-side stand-in, so kernels must be given this address.
void *noalloc_scratch() {
  static std::mutex mu;
  static void *ptrs[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> g(mu);
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_os2_noalloc_scratch) != cudaSuccess || !p) return nullptr;
    ptrs[dev] = p;
  }
  return ptrs[dev];
}

}  // namespace

extern "C" os2_status os2_gemm_noalloc(int m, int n, int k, const double *A, int lda,
                                       const double *B, int ldb, double *C, int ldc,
                                       int num_moduli, int mode, void *stream) {
  os2_status st = check_gemm_args(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode);
  if (st) return st;
  Layout L;
  make_layout(m, n, k, num_moduli, mode, &L);
  if (m == 0 || n == 0) return OS2_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // k == 0: C = 0 and no scratch is touched, whatever the sizes (as os2_gemm)
  if (k == 0) return run_gemm(false, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, nullptr, L, s);
  if (L.total > (size_t)OS2_NOALLOC_SCRATCH_BYTES) return OS2_ERR_WORKSPACE;
  void *ws = noalloc_scratch();
  if (!ws) return OS2_ERR_CUDA;
  // one pass on the caller's stream: the row-panel pipeline of os2_gemm would
  // create library streams and events on first use
  return run_gemm(false, m, n, k, A, lda, B, ldb, C, ldc, num_moduli, mode, ws, L, s);
}
