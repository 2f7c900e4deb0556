/*
 * os2_oracle.c -- CPU oracle for Ozaki Scheme II (CRT-emulated FP64 GEMM).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant generator with the CUDA library: every constant it
 * needs (moduli, P, H, CRT multipliers) is derived here from first principles.
 *
 * Sources (the method is stated on two web pages; titles and sections named):
 *  [Q]  "8ビットの整数で53ビットの倍精度を組み立てる。中国剰余定理をGPUに載せた
 *       Ozaki Scheme II" (Qiita article on Ozaki Scheme II).
 *  [G]  "Improved Scaling for Fast Mode of Ozaki Scheme II" (gist.science
 *       summary, section "Methodik").
 *
 * Everything is exact integer arithmetic except the final, single, correctly
 * rounded conversion to binary64.  Slow on purpose: no blocking, no fusion.
 *
 * Data conventions (same as the library boundary):
 *   A  : m x k, row-major, leading dimension lda >= k   (row i = a_i,:)
 *   Bt : n x k, row-major, leading dimension ldb >= k   (row j = b_:,j)
 *   so B = Bt^T is k x n with its columns contiguous.
 */
#include <limits.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef unsigned __int128 u128;
typedef __int128 i128;

enum { ORC_OK = 0, ORC_ERR_ARG = 1, ORC_ERR_NONFINITE = 4, ORC_ERR_RANGE = 5 };
enum { ORC_FAST = 0, ORC_ACCURATE = 1 };

/* ------------------------------------------------------------------------- */
/* 256-bit two's-complement integers, 8 little-endian 32-bit limbs.          */
/* ------------------------------------------------------------------------- */
#define NL 8
typedef struct { uint32_t w[NL]; } big_t;

static big_t big_zero(void) { big_t r; memset(&r, 0, sizeof r); return r; }

static big_t big_from_u128(u128 v) {
  big_t r = big_zero();
  for (int i = 0; i < 4; i++) { r.w[i] = (uint32_t)v; v >>= 32; }
  return r;
}

static int big_is_neg(const big_t *a) { return (int)(a->w[NL - 1] >> 31); }

static int big_is_zero(const big_t *a) {
  for (int i = 0; i < NL; i++) if (a->w[i]) return 0;
  return 1;
}

static big_t big_add(big_t a, big_t b) {
  big_t r; uint64_t c = 0;
  for (int i = 0; i < NL; i++) { c += (uint64_t)a.w[i] + b.w[i]; r.w[i] = (uint32_t)c; c >>= 32; }
  return r;
}

static big_t big_neg(big_t a) {
  big_t r; uint64_t c = 1;
  for (int i = 0; i < NL; i++) { c += (uint64_t)(uint32_t)~a.w[i]; r.w[i] = (uint32_t)c; c >>= 32; }
  return r;
}

static big_t big_sub(big_t a, big_t b) { return big_add(a, big_neg(b)); }

/* signed comparison; operands stay far below 2^254 so a-b cannot wrap */
static int big_cmp(big_t a, big_t b) {
  big_t d = big_sub(a, b);
  if (big_is_zero(&d)) return 0;
  return big_is_neg(&d) ? -1 : 1;
}

/* non-negative a times unsigned s */
static big_t big_mul_u32(big_t a, uint32_t s) {
  big_t r; uint64_t c = 0;
  for (int i = 0; i < NL; i++) { c += (uint64_t)a.w[i] * s; r.w[i] = (uint32_t)c; c >>= 32; }
  return r;
}

/* signed a times a small signed integer */
static big_t big_mul_small(big_t a, int s) {
  int neg = (s < 0) ^ big_is_neg(&a);
  big_t m = big_is_neg(&a) ? big_neg(a) : a;
  big_t r = big_mul_u32(m, (uint32_t)(s < 0 ? -s : s));
  return neg ? big_neg(r) : r;
}

static big_t big_shl(big_t a, int s) {
  big_t r = big_zero();
  int q = s / 32, b = s % 32;
  for (int i = NL - 1; i >= q; i--) {
    uint64_t v = (uint64_t)a.w[i - q] << b;
    if (b && i - q - 1 >= 0) v |= (uint64_t)a.w[i - q - 1] >> (32 - b);
    r.w[i] = (uint32_t)v;
  }
  return r;
}

static big_t big_shr(big_t a, int s) { /* logical, for non-negative a */
  big_t r = big_zero();
  int q = s / 32, b = s % 32;
  for (int i = 0; i + q < NL; i++) {
    uint64_t v = a.w[i + q] >> b;
    if (b && i + q + 1 < NL) v |= ((uint64_t)a.w[i + q + 1] << (32 - b)) & 0xffffffffu;
    r.w[i] = (uint32_t)v;
  }
  return r;
}

static int big_bitlen(big_t a) { /* non-negative a */
  for (int i = NL - 1; i >= 0; i--)
    if (a.w[i]) { int b = 0; uint32_t v = a.w[i]; while (v) { b++; v >>= 1; } return 32 * i + b; }
  return 0;
}

static uint32_t big_mod_u32(big_t a, uint32_t d) { /* non-negative a */
  uint64_t r = 0;
  for (int i = NL - 1; i >= 0; i--) r = ((r << 32) | a.w[i]) % d;
  return (uint32_t)r;
}

static big_t big_div_u32(big_t a, uint32_t d) { /* non-negative a */
  big_t q; uint64_t r = 0;
  for (int i = NL - 1; i >= 0; i--) { uint64_t cur = (r << 32) | a.w[i]; q.w[i] = (uint32_t)(cur / d); r = cur % d; }
  return q;
}

/* product of two unsigned magnitudes below 2^128 (fits 256 bits) */
static big_t big_mul_u128(u128 x, u128 y) {
  uint32_t a[4], b[4]; uint64_t acc[NL + 1];
  for (int i = 0; i < 4; i++) { a[i] = (uint32_t)(x >> (32 * i)); b[i] = (uint32_t)(y >> (32 * i)); }
  big_t r = big_zero();
  for (int i = 0; i < NL + 1; i++) acc[i] = 0;
  for (int i = 0; i < 4; i++) {
    uint64_t c = 0;
    for (int j = 0; j < 4; j++) {
      uint64_t t = (uint64_t)a[i] * b[j] + acc[i + j] + c;
      acc[i + j] = (uint32_t)t; c = t >> 32;
    }
    acc[i + 4] += c;
  }
  for (int i = 0; i < NL; i++) r.w[i] = (uint32_t)acc[i];
  return r;
}

/* a mod P in [0, P), by binary long division on |a| */
static big_t big_mod_floor(big_t a, big_t P) {
  int neg = big_is_neg(&a);
  big_t r = neg ? big_neg(a) : a;
  for (int s = big_bitlen(r) - big_bitlen(P); s >= 0; s--) {
    big_t t = big_shl(P, s);
    if (big_cmp(r, t) >= 0) r = big_sub(r, t);
  }
  if (neg && !big_is_zero(&r)) r = big_sub(P, r);
  return r;
}

/* ------------------------------------------------------------------------- */
/* Moduli and CRT constants                                                  */
/* ------------------------------------------------------------------------- */

/* [Q] section "256以下の法の選び方(手順2)" and its footnote 6: pairwise-coprime
 * moduli <= 256, as large as possible; the INT8 table order is
 * 256,255,253,251,247,241,239,233,229,227,223,217,211,199,197,193 followed by
 * 191,181,179,173.  The tests check that this is the greedy descending choice. */
static const int orc_moduli_list[20] = {256, 255, 253, 251, 247, 241, 239, 233, 229, 227,
                                        223, 217, 211, 199, 197, 193, 191, 181, 179, 173};

int orc_max_moduli(void) { return 20; }

int orc_moduli(int N, int32_t *out) {
  if (N < 1 || N > 20) return 0;
  for (int l = 0; l < N; l++) out[l] = orc_moduli_list[l];
  return N;
}

/* Multiplicative inverse by exhaustive search: the smallest t in [1, p) with
 * a*t = 1 (mod p).  ([Q] section "秦九韶の大衍求一術": the 乗率.)  Returns 0 if
 * none exists. */
int64_t orc_inverse_bruteforce(int64_t a, int64_t p) {
  int64_t r = ((a % p) + p) % p;
  for (int64_t t = 1; t < p; t++) if ((r * t) % p == 1) return t;
  return 0;
}

/* Qin Jiushao's Dayan qiuyi, as the article walks it through on a 2x2 grid:
 * top-right holds the 奇数 (a mod p), bottom-right the 定母 p, top-left 1,
 * bottom-left 0.  Repeatedly divide the larger right entry by the smaller,
 * keep the remainder, and add quotient * (the other left entry) to the left
 * entry on the divided side.  Stop when top-right is 1; the final quotient is
 * chosen to leave remainder 1.  Top-left is then the 乗率 (inverse). */
int64_t orc_dayan_qiuyi(int64_t a, int64_t p) {
  int64_t tr = ((a % p) + p) % p, br = p, tl = 1, bl = 0;
  if (p == 1 || tr == 0) return 0;
  while (tr != 1) {
    if (br == tr) return 0;        /* common factor: no inverse */
    if (br > tr) {                 /* divide bottom by top */
      int64_t q = br / tr; br -= q * tr; bl += q * tl;
      if (br == 0) return 0;       /* not coprime */
    } else {                       /* divide top by bottom, leaving 1 on top */
      int64_t q = (tr - 1) / br; tr -= q * br; tl += q * bl;
    }
  }
  return tl % p;
}

typedef struct {
  int N;
  int32_t p[20];
  big_t P, H, half;     /* P = prod p_l, H = floor((P-1)/2), half = P/2 rounded up */
  big_t W[20];          /* W_l = M_l * inv_l  (the article's 用数) */
  int32_t inv[20];
} orc_tables_t;

static int make_tables(int N, orc_tables_t *t) {
  if (N < 1 || N > 20) return ORC_ERR_ARG;
  t->N = N;
  orc_moduli(N, t->p);
  t->P = big_from_u128(1);
  for (int l = 0; l < N; l++) t->P = big_mul_u32(t->P, (uint32_t)t->p[l]);
  t->H = big_shr(big_sub(t->P, big_from_u128(1)), 1);
  t->half = big_sub(t->P, t->H); /* = ceil(P/2) */
  for (int l = 0; l < N; l++) {
    big_t M = big_div_u32(t->P, (uint32_t)t->p[l]);            /* 衍数 */
    int64_t r = big_mod_u32(M, (uint32_t)t->p[l]);             /* 奇数 */
    t->inv[l] = (int32_t)orc_inverse_bruteforce(r, t->p[l]);   /* 乗率 */
    t->W[l] = big_mul_u32(M, (uint32_t)t->inv[l]);             /* 用数 */
  }
  return ORC_OK;
}

static void big_out(big_t a, uint32_t *out) { for (int i = 0; i < NL; i++) out[i] = a.w[i]; }
static big_t big_in(const uint32_t *in) { big_t a; for (int i = 0; i < NL; i++) a.w[i] = in[i]; return a; }

/* Exported tables for the pins: P, H, W_l (each 8 x u32 limbs), inv_l. */
int orc_tables(int N, uint32_t *P, uint32_t *H, uint32_t *W, int32_t *inv) {
  orc_tables_t t;
  int st = make_tables(N, &t);
  if (st) return st;
  big_out(t.P, P); big_out(t.H, H);
  for (int l = 0; l < N; l++) { big_out(t.W[l], W + NL * l); inv[l] = t.inv[l]; }
  return ORC_OK;
}

/* Textbook CRT for arbitrary small pairwise-coprime moduli ([Q] section
 * "繰り上がりのない計算": add each 用数 as many times as the residue says, then
 * remove whole turns of the product).  Result in [0, prod). */
int orc_crt_small(int n, const int64_t *res, const int64_t *mod, int64_t *out) {
  i128 prod = 1, sum = 0;
  for (int l = 0; l < n; l++) prod *= mod[l];
  for (int l = 0; l < n; l++) {
    i128 M = prod / mod[l];
    int64_t inv = orc_inverse_bruteforce((int64_t)(M % mod[l]), mod[l]);
    if (inv == 0 && mod[l] != 1) return ORC_ERR_ARG;
    sum += M * inv * (((res[l] % mod[l]) + mod[l]) % mod[l]);
  }
  *out = (int64_t)(sum % prod);
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 1 -- scaling by powers of two                                        */
/* ------------------------------------------------------------------------- */

/* |v| = mant * 2^ex2 with mant an integer < 2^53 (v finite, nonzero). */
static void decompose(double v, uint64_t *mant, int *ex2) {
  int ex;
  double f = frexp(fabs(v), &ex); /* |v| = f * 2^ex, f in [0.5, 1) */
  *mant = (uint64_t)ldexp(f, 53);
  *ex2 = ex - 53;
}

/* ceil(|v| * 2^s) for s such that the result is below 2^53. */
static uint64_t ceil_scaled(double v, int s) {
  if (v == 0.0) return 0;
  uint64_t mant; int ex2;
  decompose(v, &mant, &ex2);
  int sh = ex2 + s;
  if (sh >= 0) return mant << sh;
  if (-sh >= 64) return 1;
  uint64_t d = (uint64_t)1 << (-sh);
  return mant / d + (mant % d != 0);
}

/* trunc(v * 2^e) toward zero, exactly, as a 128-bit integer. */
static i128 trunc_scaled(double v, int e) {
  if (v == 0.0) return 0;
  uint64_t mant; int ex2;
  decompose(v, &mant, &ex2);
  int sh = ex2 + e;
  u128 mag;
  if (sh >= 0) mag = (sh >= 74) ? ((u128)1 << 126) : ((u128)mant << sh);
  else mag = (-sh >= 64) ? 0 : (mant >> (-sh));
  return v < 0 ? -(i128)mag : (i128)mag;
}

/* Q * 4^g <= H, exactly (g may be negative: then Q <= H * 4^-g). */
static int fits(big_t Q, int g, big_t H) {
  if (g >= 0) return big_cmp(big_shl(Q, 2 * g), H) <= 0;
  return big_cmp(Q, big_shl(H, -2 * g)) <= 0;
}

/* largest integer g with Q * 4^g <= H, for Q >= 1 */
static int largest_g(big_t Q, big_t H) {
  int g = 0;
  if (fits(Q, 0, H)) { while (fits(Q, g + 1, H)) g++; }
  else { do g--; while (!fits(Q, g, H)); }
  return g;
}

/* E = 1 + max exponent over the row's nonzero entries, so |x| < 2^E
 * (frexp returns exactly that exponent).  Returns 0 for an all-zero row and
 * ORC_ERR_NONFINITE if any entry is Inf/NaN. */
static int row_max_exp(const double *x, int k, int *E, int *nonzero) {
  int best = INT_MIN;
  for (int h = 0; h < k; h++) {
    double v = x[h];
    if (!isfinite(v)) return ORC_ERR_NONFINITE;
    if (v != 0.0) { int ex; frexp(v, &ex); if (ex > best) best = ex; }
  }
  *nonzero = best != INT_MIN;
  *E = *nonzero ? best : 0;
  return ORC_OK;
}

/* [G] "Methodik", 1: revised fast-mode scaling.  The sufficient condition
 * 2 mu_i ||a_i|| ||b_j|| nu_j <= P - 1 is met by splitting it symmetrically:
 * mu_i^2 * S_i <= H and nu_j^2 * T_j <= H, where S_i is an upper bound of
 * sum_h a_ih^2.  The page takes S_i from log2f plus a 4*u32 margin; here it is
 * the exact integer upper bound S_i = Q_i * 4^(E_i - 23) with
 * Q_i = sum_h ceil(|a_ih| 2^(23 - E_i))^2.  mu_i = 2^e_i is the largest power of
 * two with mu_i^2 S_i <= H, i.e. e_i = g + 23 - E_i with g the largest integer
 * with Q_i 4^g <= H.  An all-zero row gets e_i = 0. */
static int scale_fast_row(const double *x, int k, const orc_tables_t *t, int32_t *e, uint64_t *Qout) {
  int E, nz;
  int st = row_max_exp(x, k, &E, &nz);
  if (st) return st;
  if (!nz) { *e = 0; if (Qout) *Qout = 0; return ORC_OK; }
  u128 Q = 0;
  for (int h = 0; h < k; h++) {
    uint64_t q = ceil_scaled(x[h], 23 - E);
    Q += (u128)q * q;
  }
  if (Qout) *Qout = (uint64_t)Q;
  *e = largest_g(big_from_u128(Q), t->H) + 23 - E;
  return ORC_OK;
}

int orc_scale_fast(int rows, int k, const double *X, long ldx, int N, int32_t *e, uint64_t *Q) {
  orc_tables_t t;
  if (make_tables(N, &t)) return ORC_ERR_ARG;
  int err = ORC_OK;
#pragma omp parallel for schedule(dynamic, 16)
  for (int i = 0; i < rows; i++) {
    int st = scale_fast_row(X + (long)i * ldx, k, &t, &e[i], Q ? &Q[i] : NULL);
    if (st) {
#pragma omp critical
      err = st;
    }
  }
  return err;
}

/* Accurate mode.  The article says only that an extra INT8 GEMM gives a tighter
 * bound ([Q] section "2の累乗による整数化(手順1と5)"; [G] "Problemstellung", 1).
 * Reading: Abar_ih = ceil(|a_ih| 2^(6-E_i)) in [0,64], Bbar likewise, Cbar =
 * Abar*Bbar bounds 2^(12-E_i-F_j) (|A||B|)_ij from above; with R_i = max_j Cbar_ij
 * and K_j = max_i Cbar_ij, e_i = g(R_i) + 6 - E_i and f_j = g(K_j) + 6 - F_j
 * give mu_i nu_j (|A||B|)_ij <= sqrt(4^g R_i 4^g' K_j) <= H.  A row whose
 * bound is 0 contributes nothing; it gets e_i = -E_i (its integers are 0). */
static int exp_from_bound(int64_t R, int E, const orc_tables_t *t) {
  if (R == 0) return -E;
  return largest_g(big_from_u128((u128)R), t->H) + 6 - E;
}

/* Abar for one row; returns E and nonzero flag via row_max_exp */
static int bar_row(const double *x, int k, uint8_t *out, int *E) {
  int nz;
  int st = row_max_exp(x, k, E, &nz);
  if (st) return st;
  for (int h = 0; h < k; h++) out[h] = (uint8_t)ceil_scaled(x[h], 6 - *E);
  return ORC_OK;
}

/* Exponents in accurate mode for selected rows of A and selected columns of B.
 * Cost O((nr*n + nc*m) * k). */
int orc_scale_accu(int m, int n, int k, const double *A, long lda, const double *Bt, long ldb, int N,
                   int nr, const int32_t *rows, int32_t *e_rows, int nc, const int32_t *cols,
                   int32_t *f_cols, int64_t *R_rows, int64_t *K_cols) {
  orc_tables_t t;
  if (make_tables(N, &t)) return ORC_ERR_ARG;
  uint8_t *Ab = (uint8_t *)malloc((size_t)m * (k ? k : 1));
  uint8_t *Bb = (uint8_t *)malloc((size_t)n * (k ? k : 1));
  int *EA = (int *)malloc(sizeof(int) * (m ? m : 1));
  int *EB = (int *)malloc(sizeof(int) * (n ? n : 1));
  int err = ORC_OK;
  for (int i = 0; i < m && !err; i++) err = bar_row(A + (long)i * lda, k, Ab + (size_t)i * k, &EA[i]);
  for (int j = 0; j < n && !err; j++) err = bar_row(Bt + (long)j * ldb, k, Bb + (size_t)j * k, &EB[j]);
  if (!err) {
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < nr; s++) {
      int i = rows[s]; int64_t R = 0;
      for (int j = 0; j < n; j++) {
        int64_t c = 0;
        for (int h = 0; h < k; h++) c += (int64_t)Ab[(size_t)i * k + h] * Bb[(size_t)j * k + h];
        if (c > R) R = c;
      }
      e_rows[s] = exp_from_bound(R, EA[i], &t);
      if (R_rows) R_rows[s] = R;
    }
#pragma omp parallel for schedule(dynamic, 1)
    for (int s = 0; s < nc; s++) {
      int j = cols[s]; int64_t K = 0;
      for (int i = 0; i < m; i++) {
        int64_t c = 0;
        for (int h = 0; h < k; h++) c += (int64_t)Ab[(size_t)i * k + h] * Bb[(size_t)j * k + h];
        if (c > K) K = c;
      }
      f_cols[s] = exp_from_bound(K, EB[j], &t);
      if (K_cols) K_cols[s] = K;
    }
  }
  free(Ab); free(Bb); free(EA); free(EB);
  return err;
}

/* The two ends of orc_scale_accu as separate calls, for bounds gathered
 * elsewhere -- for example the maxima R_i, K_j of a product split into output
 * blocks, each block's maxima taken over its own columns (rows) and then
 * reduced with MAX over the blocks that share its rows (columns).
 * orc_row_exponents: the exponent bases E_i (|x_ih| < 2^E_i; 0 for a row of
 * zeros).  orc_exps_from_bounds: e = g(R) + 6 - E (e = -E for R = 0). */
int orc_row_exponents(int rows, int k, const double *X, long ldx, int32_t *E) {
  int err = ORC_OK;
  for (int i = 0; i < rows && !err; i++) {
    int Ei, nz;
    err = row_max_exp(X + (long)i * ldx, k, &Ei, &nz);
    E[i] = Ei;
  }
  return err;
}

int orc_exps_from_bounds(int cnt, const int64_t *R, const int32_t *E, int N, int32_t *e) {
  orc_tables_t t;
  if (make_tables(N, &t)) return ORC_ERR_ARG;
  for (int i = 0; i < cnt; i++) {
    if (R[i] < 0) return ORC_ERR_ARG;
    e[i] = exp_from_bound(R[i], E[i], &t);
  }
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 2 -- truncation to integers and symmetric residues                    */
/* ------------------------------------------------------------------------- */

/* [Q] section "256以下の法の選び方(手順2)": residues held around zero, in
 * [-floor(p/2), ceil(p/2) - 1]; for p = 256 that is [-128, 127]. */
static int sym_mod(i128 a, int p) {
  int r = (int)(a % p);
  if (r < 0) r += p;
  if (r >= (p + 1) / 2) r -= p;
  return r;
}

/* The scaled integers of selected rows, A'_ih = trunc(a_ih 2^e_i), written
 * as (lo, hi) int64 pairs (two's complement 128-bit). */
int orc_integers(int rows, int k, const double *X, long ldx, const int32_t *e, int64_t *out) {
  for (int i = 0; i < rows; i++)
    for (int h = 0; h < k; h++) {
      i128 v = trunc_scaled(X[(long)i * ldx + h], e[i]);
      out[2 * ((size_t)i * k + h)] = (int64_t)(uint64_t)v;
      out[2 * ((size_t)i * k + h) + 1] = (int64_t)(v >> 64);
    }
  return ORC_OK;
}

/* Residue planes res[l][i][h] = sym_mod(trunc(x_ih 2^e_i), p_l). */
int orc_residues(int rows, int k, const double *X, long ldx, const int32_t *e, int N, int8_t *res) {
  int32_t p[20];
  if (orc_moduli(N, p) != N) return ORC_ERR_ARG;
#pragma omp parallel for schedule(static)
  for (int i = 0; i < rows; i++)
    for (int h = 0; h < k; h++) {
      i128 v = trunc_scaled(X[(long)i * ldx + h], e[i]);
      for (int l = 0; l < N; l++) res[((size_t)l * rows + i) * k + h] = (int8_t)sym_mod(v, p[l]);
    }
  return ORC_OK;
}

/* ------------------------------------------------------------------------- */
/* Step 5 -- one correctly rounded conversion of X * 2^-s to binary64         */
/* ------------------------------------------------------------------------- */

/* Round-to-nearest-even of X * 2^(-s) to a binary format with a prec-bit
 * significand and minimum normal exponent emin (binary64: 53, -1022;
 * binary32: 24, -126), subnormals and overflow included.  Keeps the bits of
 * |X| at positions >= cut, where cut is the larger of bitlen - prec and
 * s - (prec - 1 - emin) (the weight of the smallest subnormal).  The result is
 * returned as a double holding the value of that format (+-Inf on overflow). */
static double round_scaled_fmt(big_t X, int s, int prec, int emin, int emax) {
  const int lsb = prec - 1 - emin;
  int neg = big_is_neg(&X);
  big_t M = neg ? big_neg(X) : X;
  if (big_is_zero(&M)) return 0.0;
  int b = big_bitlen(M);
  int cut = b - prec;
  if (s - lsb > cut) cut = s - lsb;
  uint64_t kept;
  if (cut <= 0) {
    kept = (uint64_t)M.w[0] | ((uint64_t)M.w[1] << 32);   /* exact: M < 2^53 */
  } else if (cut > b) {
    kept = 0;                                             /* below half of 2^-1074 */
  } else {
    big_t K = big_shr(M, cut);
    kept = (uint64_t)K.w[0] | ((uint64_t)K.w[1] << 32);
    big_t rem = big_sub(M, big_shl(K, cut));
    big_t half = big_shl(big_from_u128(1), cut - 1);
    int c = big_cmp(rem, half);
    if (c > 0 || (c == 0 && (kept & 1))) kept += 1;
  }
  if (cut < 0) cut = 0;
  double r = ldexp((double)kept, cut - s);
  if (r >= ldexp(1.0, emax + 1)) r = INFINITY;  /* rounded value beyond the format */
  return neg ? -r : r;
}

static double round_scaled(big_t X, int s) { return round_scaled_fmt(X, s, 53, -1022, 1023); }

/* exported for the rounding pins: X given as 8 u32 limbs (two's complement) */
double orc_round_scaled(const uint32_t *X, int s) { return round_scaled(big_in(X), s); }
double orc_round_scaled_f32(const uint32_t *X, int s) {
  return round_scaled_fmt(big_in(X), s, 24, -126, 127);
}

/* Output format of orc_gemm_entries: binary64 (DGEMM) or binary32 (SGEMM;
 * [G] "Ergebnisse": the revised scaling is evaluated for SGEMM too). */
static int orc_out_f32 = 0;
void orc_set_output_f32(int on) { orc_out_f32 = on ? 1 : 0; }

/* ------------------------------------------------------------------------- */
/* Steps 3-5 for selected output entries                                      */
/* ------------------------------------------------------------------------- */

/*
 * For every (rows[a], cols[b]) pair: the scaled integers A', B' of those rows
 * and columns; X_direct = sum_h A'_ih B'_hj exactly; per modulus the integer
 * product G_l of the residue vectors and c_l = sym_mod(G_l, p_l) ([Q] section
 * "誤差のないINT8行列積(手順3)"); the CRT value X = (sum_l c_l W_l) mod P lifted to
 * [-P/2, P/2) ([Q] section "繰り上がりのない計算", [G] "Problemstellung"); the check
 * X == X_direct (the scaling guarantees |X_direct| <= H); and the unscaled
 * result C = RN(X 2^-(e_i + f_j)) ([Q] section "2の累乗による整数化(手順1と5)").
 *
 * e_rows / f_cols: the exponents of the selected rows / columns; computed here
 * (from the selected rows/cols alone) in fast mode when compute_exp != 0,
 * otherwise taken as given (accurate mode: use orc_scale_accu first).
 *
 * Outputs (any but C may be NULL), entry index a*nc + b:
 *   C[a*nc+b], X[(a*nc+b)*8 + limb], c[(a*nc+b)*N + l], G[(a*nc+b)*N + l]
 *   nmismatch: count of entries whose CRT value differs from X_direct.
 */
int orc_gemm_entries(int m, int n, int k, const double *A, long lda, const double *Bt, long ldb,
                     int N, int nr, const int32_t *rows, int nc, const int32_t *cols,
                     int compute_exp, int32_t *e_rows, int32_t *f_cols,
                     double *C, uint32_t *X, int8_t *c, int64_t *G, int64_t *nmismatch) {
  (void)m; (void)n;
  orc_tables_t t;
  if (make_tables(N, &t)) return ORC_ERR_ARG;
  int err = ORC_OK;
  if (compute_exp) {
    for (int a = 0; a < nr && !err; a++) err = scale_fast_row(A + (long)rows[a] * lda, k, &t, &e_rows[a], NULL);
    for (int b = 0; b < nc && !err; b++) err = scale_fast_row(Bt + (long)cols[b] * ldb, k, &t, &f_cols[b], NULL);
  } else {
    for (int a = 0; a < nr && !err; a++) { int E, nz; err = row_max_exp(A + (long)rows[a] * lda, k, &E, &nz); }
    for (int b = 0; b < nc && !err; b++) { int E, nz; err = row_max_exp(Bt + (long)cols[b] * ldb, k, &E, &nz); }
  }
  if (err) return err;

  size_t kk = k ? (size_t)k : 1;
  i128 *Ai = (i128 *)malloc(sizeof(i128) * nr * kk);
  i128 *Bi = (i128 *)malloc(sizeof(i128) * nc * kk);
  int16_t *rA = (int16_t *)malloc(sizeof(int16_t) * nr * kk * N);
  int16_t *rB = (int16_t *)malloc(sizeof(int16_t) * nc * kk * N);
  for (int a = 0; a < nr; a++)
    for (int h = 0; h < k; h++) {
      i128 v = trunc_scaled(A[(long)rows[a] * lda + h], e_rows[a]);
      Ai[a * kk + h] = v;
      for (int l = 0; l < N; l++) rA[((size_t)l * nr + a) * kk + h] = (int16_t)sym_mod(v, t.p[l]);
    }
  for (int b = 0; b < nc; b++)
    for (int h = 0; h < k; h++) {
      i128 v = trunc_scaled(Bt[(long)cols[b] * ldb + h], f_cols[b]);
      Bi[b * kk + h] = v;
      for (int l = 0; l < N; l++) rB[((size_t)l * nc + b) * kk + h] = (int16_t)sym_mod(v, t.p[l]);
    }

  int64_t bad = 0;
#pragma omp parallel for schedule(dynamic, 4) reduction(+ : bad)
  for (int a = 0; a < nr; a++) {
    for (int b = 0; b < nc; b++) {
      size_t idx = (size_t)a * nc + b;
      /* direct exact product */
      big_t Xd = big_zero();
      for (int h = 0; h < k; h++) {
        i128 x = Ai[a * kk + h], y = Bi[b * kk + h];
        if (x == 0 || y == 0) continue;
        int neg = (x < 0) != (y < 0);
        big_t pr = big_mul_u128((u128)(x < 0 ? -x : x), (u128)(y < 0 ? -y : y));
        Xd = neg ? big_sub(Xd, pr) : big_add(Xd, pr);
      }
      /* per-modulus products and CRT */
      big_t S = big_zero();
      for (int l = 0; l < N; l++) {
        int64_t g = 0;
        const int16_t *ra = rA + ((size_t)l * nr + a) * kk, *rb = rB + ((size_t)l * nc + b) * kk;
        for (int h = 0; h < k; h++) g += (int64_t)ra[h] * rb[h];
        int cl = sym_mod((i128)g, t.p[l]);
        if (G) G[idx * N + l] = g;
        if (c) c[idx * N + l] = (int8_t)cl;
        S = big_add(S, big_mul_small(t.W[l], cl));
      }
      big_t Xc = big_mod_floor(S, t.P);
      if (big_cmp(Xc, t.half) >= 0) Xc = big_sub(Xc, t.P); /* lift [P/2, P) to [-P/2, 0) */
      if (big_cmp(Xc, Xd) != 0) bad++;
      if (X) big_out(Xc, X + idx * NL);
      if (C) C[idx] = orc_out_f32 ? round_scaled_fmt(Xc, e_rows[a] + f_cols[b], 24, -126, 127)
                                  : round_scaled(Xc, e_rows[a] + f_cols[b]);
    }
  }
  free(Ai); free(Bi); free(rA); free(rB);
  if (nmismatch) *nmismatch = bad;
  return ORC_OK;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}
