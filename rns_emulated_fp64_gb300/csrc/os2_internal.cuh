// Internal declarations shared by the translation units of libos2.
#pragma once
#include <cuda_runtime.h>
#include <cuda.h>
#include <stddef.h>
#include <stdint.h>

#include "os2.h"

// Debug build (compiled with -DOS2_DEBUG): the kernels check the index of each
// hand-computed global access against the extent of the array it addresses;
// a failed check records OS2_ERR_BOUNDS in the status word and skips the
// access.  In the release build the checks compile to nothing.
#ifdef OS2_DEBUG
#define OS2_DBG_GUARD(cond, status) \
  ((cond) ? true : (((status) ? atomicCAS((status), 0, (int)OS2_ERR_BOUNDS) : 0), false))
#else
#define OS2_DBG_GUARD(cond, status) true
#endif

#define OS2_MAX_MODULI 20
#define OS2_KP_ALIGN 64          // residue-plane row pitch granularity (one 128-byte k-block)
#define OS2_CRES_ALIGN 16        // int8 product-residue row pitch granularity
#define OS2_H_LIMBS 7            // 32-bit limbs for H (P < 2^156 for N <= 20)

// Step-2 constants (kernel parameter, lives in the constant bank).
struct ResConsts {
  int N;
  float p[OS2_MAX_MODULI];       // p_l
  float invp[OS2_MAX_MODULI];    // fl(1/p_l)
  float hi[OS2_MAX_MODULI];      // ceil(p_l/2) - 1   (top of the symmetric range)
  float lo[OS2_MAX_MODULI];      // -floor(p_l/2)     (bottom)
  // Step 2 word constants, each float twice in 64 bits (packed FP32 pairs):
  // w15x2: symmetric residue of 2^(15 t) mod p_l, t = 0..5; k15x2[l][NW - 4]:
  // symmetric residue of 2^14 (1 + 2^15 + ... + 2^(15 (NW - 2))) mod p_l.
  unsigned long long w15x2[OS2_MAX_MODULI][6];
  unsigned long long k15x2[OS2_MAX_MODULI][3];
  unsigned long long invp2[OS2_MAX_MODULI];  // fl(1/p_l)
  unsigned long long negp2[OS2_MAX_MODULI];  // -p_l
  uint32_t H[OS2_H_LIMBS];       // H = floor((P-1)/2), little-endian 32-bit limbs
  int bitlenH;
  unsigned long long H64;        // the 64 leading bits of H (leading bit at bit 63)
  int Hrest;                     // nonzero if H has set bits below those 64
};

// Steps 4-5 constants (32-bit little-endian limbs).
struct CrtConsts {
  int N;
  uint32_t W32[OS2_MAX_MODULI][5];   // W_l = M_l inv_l
  uint32_t P32[6];                   // P
  uint32_t H32[6];                   // P / 2
  float s_top, s_next;               // fl(2^(32(LW-1)) / P), fl(2^(32(LW-2)) / P), LW = (N+3)/4
  float s128;                        // fl(128 / P)
};

// Steps 4-5 on the tensor cores (k_crt_tc): W_l in signed 10-bit digits,
// W_l = sum_t w_{l,t} 2^(10 t), |w| <= 512; the digit sums of Y = sum_l (c_l +
// 128) W_l come out of one FP16 MMA per 128 entries.
#define OS2_CRT_DIGITS 16
struct CrtTcConsts {
  int N, T, LX, Q;                                // moduli, digits, 32-bit limbs of X, digits for q
  int16_t wd[OS2_MAX_MODULI][OS2_CRT_DIGITS];     // w_{l,t}
  float rmag[OS2_CRT_DIGITS];                     // 1.5 * 2^23 - 1024 sum_l w_{l,t}
  uint32_t pw[OS2_CRT_DIGITS];                    // 2^(10 t mod 32)
  uint32_t negc[5];                               // -(C0 + 128) mod 2^(32 LX)
  uint32_t np[5];                                 // 2^(32 LX) - P
  uint32_t P32[5];                                // P
  uint32_t H32[5];                                // P / 2
  float s[OS2_CRT_DIGITS];                        // 2^(10 (T - 1 - j)) / P, j < Q
  float c0;                                       // -128 / P
};

// Step-3 constants.
struct GemmConsts {
  int N;
  float p[OS2_MAX_MODULI];
  float invp[OS2_MAX_MODULI];
  float hi[OS2_MAX_MODULI];
  float lo[OS2_MAX_MODULI];
};

struct Os2Tables {
  int N;
  int32_t p[OS2_MAX_MODULI];
  int32_t inv[OS2_MAX_MODULI];
  ResConsts res;
  CrtConsts crt;
  CrtTcConsts crt_tc;
  GemmConsts gemm;
};

// Host: tables for N moduli (cached; thread-safe).  NULL on bad N.
const Os2Tables *os2_tables(int N);

// Per-device status word (device address), set up on first use.
int *os2_status_ptr();

// Number of SMs of the current device (at least 1).
int os2_sm_count();

// One CTA whose bounded mbarrier waits run out (failure-detection self-test).
cudaError_t launch_wait_selftest(long long limit, int *status, int32_t *result, cudaStream_t s);

// Pipe-peak probes (os2_peak_probe).  Writes the flop one launch does to *flop.
cudaError_t launch_peak_probe(int kind, int iters, int check, int32_t *result, int *status,
                              cudaStream_t s, double *flop);

// Row-scale kernel modes.
enum ScaleMode {
  SM_FAST_SCALE = 0,   // fast mode: e_i from the revised bound
  SM_BARS = 1,         // accurate mode: E_i and the 7-bit magnitude plane
};

// Launchers (return cudaError_t of the launch).  Each handles A's rows and
// B's columns (rows of Bt) in one launch; pass rowsB = 0 for one operand.
// f32: the operands are float (SGEMM emulation) instead of double.
cudaError_t launch_row_scale(int mode, bool f32, const void *XA, long lda, int rowsA,
                             int32_t *eA, int32_t *EA, void *barsA, const void *XB, long ldb,
                             int rowsB, int32_t *eB, int32_t *EB, void *barsB, int k, int kp,
                             const Os2Tables *t, int *status, cudaStream_t s);
cudaError_t launch_residues(bool f32, const void *XA, long lda, int rowsA, const int32_t *eA,
                            void *planesA, const void *XB, long ldb, int rowsB,
                            const int32_t *eB, void *planesB, int k, int kp, const Os2Tables *t,
                            cudaStream_t s, long prowB = 0, bool i8 = false);
cudaError_t launch_accu_exponents(const int32_t *bound, const int32_t *E, int rows, int32_t *e,
                                  const Os2Tables *t, cudaStream_t s);
// f32: C is float (correctly rounded to binary32) instead of double.
cudaError_t launch_crt(bool f32, int m, int n, const int8_t *c, int ldcres, const int32_t *e,
                       const int32_t *f, void *C, int ldc, uint32_t *X_out, const Os2Tables *t,
                       cudaStream_t s, int *status = nullptr);
// Steps 4 + 5 on the tensor cores; needs ldcres % 16 == 0 and a 16-byte
// aligned c (else cudaErrorInvalidValue).
cudaError_t launch_crt_tc(bool f32, int m, int n, const int8_t *c, int ldcres, const int32_t *e,
                          const int32_t *f, void *C, int ldc, uint32_t *X_out, const Os2Tables *t,
                          int *status, cudaStream_t s);
cudaError_t launch_gemm_simt(int m, int n, int kp, const void *RA, const void *RB, int N,
                             int out_kind, void *out, int ldo, const Os2Tables *t, cudaStream_t s);

// mma.sync s8 GEMM (the INT8 tensor path outside tcgen05) on int8 planes RA
// [N][m][kp] and RB [N][b_plane_rows][kp] (b_plane_rows 0: n); out_kind as
// os2_gemm_residues.
cudaError_t launch_gemm_s8(int m, int n, int kp, const void *RA, const void *RB, int N,
                           int out_kind, void *out, int ldo, const Os2Tables *t, int *status,
                           cudaStream_t s, int b_plane_rows = 0);

// tcgen05 GEMM.  kind: 0 = mod-p int8 output (single SM), 1 = exact int32 (raw
// output and/or row/col maxima), 2 = mod-p int8 output on SM pairs (2-SM MMA),
// 3 = as 2 from int8 residue planes (widened to FP16 on chip).  prod_bound_log2: log2 of the largest |a*b| of one term
// (14 for residues, 12 for the accurate-mode magnitude planes).
cudaError_t launch_gemm_tc(int kind, int m, int n, int kp, const void *RA, const void *RB,
                           int nplanes, void *out, int ldo, int32_t *rowmax, int32_t *colmax,
                           int prod_bound_log2, const Os2Tables *t, int *status, cudaStream_t s,
                           int b_plane_rows = 0);

// Accurate-mode bound product with fused row/column maxima on the 2-SM
// kernel: magnitude planes (one FP16 plane each, values <= 64) of A (m rows)
// and B (n rows); atomicMax into rowmax[m] and colmax[n] (zeroed by the
// caller).  k is taken in segments of 4096 (64 k-blocks); with more than one
// segment, partial (int32 [m][ldp], ldp >= n a multiple of 4, 16-byte
// aligned) holds the sums between them.
cudaError_t launch_gemm_bound2(int m, int n, int kp, const void *RA, const void *RB,
                               int32_t *partial, int ldp, int32_t *rowmax, int32_t *colmax,
                               int *status, cudaStream_t s);

// Complex products: interleaved complex operands <-> stacked real operands.
cudaError_t launch_complex_stack(bool f32, int m, int n, int k, const void *A, long lda,
                                 const void *B, long ldb, void *A2, void *Bt2, cudaStream_t s);
cudaError_t launch_complex_unstack(bool f32, int m, int n, const void *C2, void *C, long ldc,
                                   cudaStream_t s);

static inline size_t os2_round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }
