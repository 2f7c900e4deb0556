/*
 * os2.h -- C ABI of libos2: Ozaki Scheme II emulation of an FP64 matrix
 * product C = A * B on one NVIDIA GB300 (sm_103a).
 *
 * The method is the one described in two web pages:
 *   [Q] Qiita, "8ビットの整数で53ビットの倍精度を組み立てる。中国剰余定理をGPUに載せた
 *       Ozaki Scheme II" (sections "行列積への当てはめ方" (the five steps),
 *       "2の累乗による整数化(手順1と5)", "256以下の法の選び方(手順2)",
 *       "誤差のないINT8行列積(手順3)", "高い精度での復元(手順4)").
 *   [G] gist.science, "Improved Scaling for Fast Mode of Ozaki Scheme II"
 *       (section "Methodik": the revised, scale-invariant fast-mode scaling).
 *
 * Steps: (1) per-row / per-column power-of-two scaling mu_i = 2^e_i,
 * nu_j = 2^f_j; (2) truncation to integers A' = trunc(mu A), B' = trunc(B nu)
 * and reduction to symmetric residues modulo N pairwise-coprime moduli
 * p_l <= 256; (3) N exact residue matrix products, each reduced mod p_l;
 * (4) Chinese-remainder reconstruction of the integer product X = A'B' in
 * [-P/2, P/2), P = prod p_l; (5) C_ij = RN(X_ij * 2^-(e_i + f_j)).
 *
 * Conventions shared by every entry point
 *  - All matrix pointers are DEVICE pointers owned by the caller (except in
 *    os2_gemm_host, whose matrices live in host memory).  The library never
 *    allocates or frees device memory.
 *  - A is m x k ROW-major with leading dimension lda >= k (A[i*lda + h]).
 *    B is k x n COLUMN-major with leading dimension ldb >= k
 *    (B[j*ldb + h] = b_hj): both operands are contiguous along k.
 *    C is m x n ROW-major with ldc >= n (C[i*ldc + j]).
 *  - num_moduli N is in [1, 20]; the moduli are the first N of
 *    256,255,253,251,247,241,239,233,229,227,223,217,211,199,197,193,191,181,179,173
 *    ([Q] "256以下の法の選び方(手順2)", footnote 6).  14-16 give about
 *    native-FP64 accuracy ([Q] "行列積の回数と性能").
 *  - 0 <= k < 2^24.  [Q] "誤差のないINT8行列積(手順3)": INT32 sums of residue
 *    products are exact only while k < 2^17, and larger k is split into
 *    blocks.  Here step 3 reduces its partial sums mod p_l block by block (at
 *    most 960 terms per block in tensor memory, 65536 in the mma.sync
 *    variant's int32 registers), so that split is built in and the mod-p
 *    products have no such limit.  Remaining limits: accurate mode k < 2^19 (its exact int32 bound
 *    product), raw int32 products from os2_gemm_residues k < 2^17.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every device-side entry point only enqueues work on it and
 *    returns; argument errors are returned synchronously before anything is
 *    enqueued.  Errors found on the device (non-finite input, a wait that
 *    timed out) are recorded in a per-device status word that
 *    os2_get_status() reads.  After any error the outputs are unspecified.
 *  - Not re-entrant on one workspace: two calls in flight at the same time
 *    must not share a workspace.
 */
#ifndef OS2_H
#define OS2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  OS2_OK = 0,
  OS2_ERR_INVALID_ARG = 1,  /* bad size, leading dimension, pointer, mode or N */
  OS2_ERR_UNSUPPORTED = 2,  /* valid but beyond a documented size limit */
  OS2_ERR_WORKSPACE = 3,    /* workspace missing or smaller than os2_workspace_size */
  OS2_ERR_NONFINITE = 4,    /* an input entry is Inf or NaN (device-detected) */
  OS2_ERR_RANGE = 5,        /* a scaled integer of os2_residues reached 2^89 */
  OS2_ERR_TIMEOUT = 6,      /* a device-side wait gave up (device-detected) */
  OS2_ERR_CUDA = 7,         /* a CUDA runtime/driver call failed */
  OS2_ERR_BOUNDS = 8        /* debug build only: a kernel's index check failed (the access
                               was skipped; see OS2_DEBUG in the build notes) */
} os2_status;

typedef enum {
  OS2_MODE_FAST = 0,      /* revised scale-invariant fast mode ([G] "Methodik") */
  OS2_MODE_ACCURATE = 1   /* bound from one extra exact matrix product ([Q] 手順1) */
} os2_mode;

typedef enum {
  OS2_GEMM_TC = 0,        /* tcgen05 2-SM tensor-core kernel, 256x256 tiles (default) */
  OS2_GEMM_SIMT = 1,      /* plain CUDA-core int32 kernel (exact reference, slow) */
  OS2_GEMM_TC_1SM = 2,    /* tcgen05 single-SM tensor-core kernel, 128x256 tiles */
  OS2_GEMM_TC_I8 = 3,     /* as OS2_GEMM_TC, from int8 residue planes in HBM (half the
                             bytes of FP16) widened to FP16 on chip by four extra warps;
                             step 2 then writes int8 planes (os2_gemm, os2_gemm_host,
                             os2_sgemm, complex products; not os2_gemm_residues) */
  OS2_GEMM_S8_SYNC = 4    /* the INT8 tensor path outside tcgen05: mma.sync.m16n8k32
                             s8 x s8 -> s32 from int8 residue planes, exact int32 sums
                             (reduced mod p every 65536 terms for mod-p output); step 2
                             then writes int8 planes, and os2_gemm_residues takes int8
                             planes for it.  About 12 times slower than OS2_GEMM_TC */
} os2_gemm_variant;

typedef enum {
  OS2_CRT_TC = 0,         /* limb sums as an FP16 tensor-core MMA per 128 entries */
  OS2_CRT_SIMT = 1,       /* limb sums as 32x32->64 multiply-adds on the CUDA cores */
  OS2_CRT_AUTO = 2        /* (default) TC alone; SIMT beside a product (see below) */
} os2_crt_variant;

typedef enum {
  OS2_OUT_MODP_INT8 = 0,  /* c_l = G_l mod p_l, symmetric, int8 [N][m][ldo] */
  OS2_OUT_RAW_INT32 = 1   /* G_l itself, int32 [N][m][ldo] */
} os2_out_kind;

/* Bytes of device workspace os2_gemm needs for these sizes (0 on bad args).
 * The workspace holds the exponents, the N FP16 residue planes of A and B
 * (N*(m+n)*ceil64(k)*2 bytes) and the N int8 product residues
 * (N*m*ceil16(n) bytes).  Must be 256-byte aligned. */
size_t os2_workspace_size(int m, int n, int k, int num_moduli, int mode);

/* The whole five-step emulated DGEMM, C = A*B ([Q] "行列積への当てはめ方": the
 * five steps applied to a matrix product; step 1 in fast mode follows [G]
 * "Methodik").  Layouts above.  Returns after
 * enqueueing on `stream`.  For m >= 4096 (unless os2_set_crt_variant selected
 * OS2_CRT_TC) the rows of A go in panels of about 2048: the CRT and unscaling
 * of one panel run on a library-owned stream (created once per device,
 * non-blocking) beside the product of the next; that stream first waits for
 * the work already on `stream`, and `stream` waits for it before the call's
 * work ends, so synchronising `stream` covers the call.  Otherwise every step
 * runs on `stream`, once over the whole problem.  Results are identical
 * either way.  Calls from several host threads are enqueued one at a time. */
os2_status os2_gemm(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                    double *C, int ldc, int num_moduli, int mode, void *workspace,
                    size_t workspace_bytes, void *stream);

/* SGEMM emulation ([G] "Improved Scaling for Fast Mode of Ozaki Scheme II",
 * "Ergebnisse": the method is evaluated for DGEMM and SGEMM).  Same five
 * steps, arguments, layouts, workspace (os2_workspace_size) and errors as
 * os2_gemm, with float A, B and C: every float is exactly a double, so the
 * exponents, integers, residues and CRT value are the ones os2_gemm computes
 * for the same entries; only the final rounding targets binary32 (RN-even,
 * subnormals, overflow to +-Inf).  Fewer moduli suffice (about 7 for FP32
 * accuracy at k ~ 10^3-10^4). */
os2_status os2_sgemm(int m, int n, int k, const float *A, int lda, const float *B, int ldb,
                     float *C, int ldc, int num_moduli, int mode, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Complex products ([G] "Bedeutung": the approach extends to ZGEMM/CGEMM).
 * A complex product is computed as the real block product
 *   [C_r | C_i] = [A_r | A_i] . [[B_r, B_i], [-B_i, B_r]]   (m x 2n x 2k),
 * so the scaling uses complex row/column norms (|a_r|^2 + |a_i|^2), every
 * integer product is exact and the CRT bound covers both parts.
 * Layouts: complex entries interleaved (re, im).  A is m x k row-major with
 * lda >= k complex entries per row; B is k x n column-major with ldb >= k
 * complex entries per column; C is m x n row-major with ldc >= n.  Workspace:
 * os2_complex_workspace_size(m, n, k, N, mode, single) bytes (single = 1 for
 * CGEMM), 256-byte aligned.  Other conventions as os2_gemm / os2_sgemm. */
size_t os2_complex_workspace_size(int m, int n, int k, int num_moduli, int mode, int single);
os2_status os2_zgemm(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                     double *C, int ldc, int num_moduli, int mode, void *workspace,
                     size_t workspace_bytes, void *stream);
os2_status os2_cgemm(int m, int n, int k, const float *A, int lda, const float *B, int ldb,
                     float *C, int ldc, int num_moduli, int mode, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Device workspace for os2_gemm_host: os2_workspace_size plus device copies
 * of A (m*k), B (k*n) and C (m*n) doubles. */
size_t os2_host_workspace_size(int m, int n, int k, int num_moduli, int mode);

/* End-to-end variant of os2_gemm whose A, B, C are HOST pointers (pinned
 * memory gives asynchronous copies; pageable memory works, with copies that
 * block the calling thread).  Results are identical to os2_gemm's.  The copies
 * overlap the kernels: A and B travel in panels (row panels of A, column
 * panels of B, about 2048 rows each) on a library-owned copy-in stream, each
 * block of C is computed on `stream` once its two panels have arrived (its
 * CRT on a library-owned stream beside the next block's product), and leaves
 * on a library-owned copy-out stream while the next block is computed.  The
 * library's streams (created once per device, non-blocking) first wait for
 * the work already enqueued on `stream`, and `stream` waits for the last copy
 * out, so synchronising `stream` covers the whole call; the caller
 * synchronises it before reading C, and must not reuse the workspace on
 * another stream before then.  Calls from several host threads are enqueued
 * one at a time. */
os2_status os2_gemm_host(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                         double *C, int ldc, int num_moduli, int mode, void *workspace,
                         size_t workspace_bytes, void *stream);

/* Step 1 alone: exponents e (m int32) and f (n int32) such that
 * mu_i = 2^e_i, nu_j = 2^f_j.  FAST: the revised formula of [G] "Methodik"
 * with an exact integer upper bound of sum_h a_ih^2 (no workspace needed:
 * pass NULL/0).  ACCURATE: needs os2_workspace_size(m,n,k,1,ACCURATE)
 * bytes. */
os2_status os2_scale(int m, int n, int k, const double *A, int lda, const double *B, int ldb,
                     int num_moduli, int mode, int32_t *e, int32_t *f, void *workspace,
                     size_t workspace_bytes, void *stream);

/* Accurate-mode step 1 split in two, for a product computed in output blocks
 * (one block per GPU, [Q] "誤差のないINT8行列積(手順3)": the moduli, the
 * residues and the reconstruction are independent per entry, and the scaling
 * is per row and per column).  os2_scale_bounds takes the block's rows of A
 * and columns of B (layouts as os2_gemm) and writes, as device int32 arrays:
 * R[m] = max_j Cbar_ij over the block's columns, K[n] = max_i Cbar_ij over its
 * rows (Cbar = Abar Bbar, the exact product of the 6-bit magnitude planes of
 * the accurate mode), and the exponent bases EA[m], EB[n] (|a_ih| < 2^EA_i; 0
 * for a row of zeros).  Workspace: os2_workspace_size(m, n, k, 1,
 * OS2_MODE_ACCURATE) bytes, 256-byte aligned.  The maxima of the whole product
 * are the MAX over the blocks that share the rows (R) or the columns (K); the
 * exponents then follow from os2_exponents_from_bounds, identical to those
 * os2_scale computes for the whole product.  k < 2^19 (else
 * OS2_ERR_UNSUPPORTED). */
os2_status os2_scale_bounds(int m, int n, int k, const double *A, int lda, const double *B,
                            int ldb, int32_t *R, int32_t *K, int32_t *EA, int32_t *EB,
                            void *workspace, size_t workspace_bytes, void *stream);

/* Accurate-mode exponents e[i] = 6 - E[i] + (largest g with bound[i] 4^g <= H),
 * e[i] = -E[i] for bound[i] = 0 ([Q] "2の累乗による整数化(手順1と5)", with the
 * bound of one extra exact product), for `count` rows or columns; device
 * int32 arrays. */
os2_status os2_exponents_from_bounds(int count, const int32_t *bound, const int32_t *E,
                                     int num_moduli, int32_t *e, void *stream);

/* Steps 2 to 5 with the exponents given (e[m] for A's rows, f[n] for B's
 * columns, device int32), for example those of os2_scale or
 * os2_exponents_from_bounds for a block of a larger product.  Arguments,
 * layouts, workspace (os2_workspace_size(m, n, k, N, OS2_MODE_FAST)) and
 * errors as os2_gemm.  Exponents larger than the scaling's can push the
 * integer product past P/2, where the reconstruction wraps: the result is
 * then unspecified (and OS2_ERR_RANGE is set if a scaled entry reaches
 * 2^89). */
os2_status os2_gemm_exponents(int m, int n, int k, const double *A, int lda, const double *B,
                              int ldb, double *C, int ldc, int num_moduli, const int32_t *e,
                              const int32_t *f, void *workspace, size_t workspace_bytes,
                              void *stream);

/* Step 2 alone for one operand ([Q] "2の累乗による整数化(手順1と5)": truncation of
 * the scaled entries to integers; [Q] "256以下の法の選び方(手順2)": their
 * symmetric residues, for p = 256 the low byte read as int8): rows x k
 * matrix X (row-major, ldx >= k; pass B
 * as its n columns), exponents exps (rows int32).  Writes N planes of FP16
 * symmetric residues, planes[(l*rows + r)*ldp + h] = sym(trunc(x_rh 2^exps_r) mod p_l),
 * for h < ldp; entries h >= k are written as 0.  ldp >= k, ldp % 64 == 0.
 * Every exponent os2_scale returns keeps |trunc(x 2^e)| below 2^84; hand-picked
 * exponents that reach 2^89 set OS2_ERR_RANGE in the status word, and the
 * residues of the 8-entry groups holding such entries are written as 0. */
os2_status os2_residues(int rows, int k, const double *X, int ldx, const int32_t *exps,
                        int num_moduli, void *planes, int ldp, void *stream);

/* Step 3 alone ([Q] "誤差のないINT8行列積(手順3)": one exact integer product of
 * the residue matrices per modulus, reduced mod p_l; larger inner dimensions
 * split into blocks): N residue matrix products from FP16 planes RA (N x m x ldp)
 * and RB (N x n x ldp), ldp % 64 == 0, k <= ldp.  out_kind selects int8
 * c_l = sym(G_l mod p_l) or raw int32 G_l; out is [N][m][ldo] with ldo >= n
 * (ldo % 16 == 0 for int8, % 4 for int32).  variant: an os2_gemm_variant
 * other than OS2_GEMM_TC_I8; with OS2_GEMM_S8_SYNC, RA and RB are int8 planes
 * (N x m x ldp and N x n x ldp bytes, residues in [-128, 127]) instead of FP16.
 * Raw int32 output with the TC variant runs the exact-accumulation kernel. */
os2_status os2_gemm_residues(int m, int n, int k, const void *RA, const void *RB, int ldp,
                             int num_moduli, int out_kind, void *out, int ldo, int variant,
                             void *stream);

/* Steps 4 and 5 ([Q] "高い精度での復元(手順4)": reconstruction of the integer
 * product from its residues beyond double precision; [Q] "繰り上がりのない計算"
 * and "秦九韶の大衍求一術": X = (sum_l c_l M_l inv_l) mod P; [Q]
 * "2の累乗による整数化(手順1と5)": the division by mu_i nu_j): from c (int8
 * [N][m][ldcres]) and the exponents, writes
 * C[i*ldc + j] = RN(X_ij * 2^-(e_i + f_j)) with X the CRT value in
 * [-P/2, P/2).  If X_out is not NULL it also receives X as 8 little-endian
 * 32-bit limbs (two's complement) per entry, X_out[(i*n + j)*8 + u]. */
os2_status os2_crt(int m, int n, const int8_t *c, int ldcres, int num_moduli, const int32_t *e,
                   const int32_t *f, double *C, int ldc, uint32_t *X_out, void *stream);

/* Host: the first num_moduli moduli into out; returns the count (0 on bad N). */
int os2_moduli(int num_moduli, int32_t *out);

/* Synchronises `stream`, returns the device status word of the current
 * device and clears it.  The word records errors only the kernels can see:
 * non-finite inputs ([Q] "行列積の回数と性能" lists Inf/NaN handling among the
 * points an emulated GEMM must settle; OS II itself gives no rule, so they
 * are rejected with OS2_ERR_NONFINITE), an out-of-range integer in
 * os2_residues (OS2_ERR_RANGE) and a device-side wait that timed out
 * (OS2_ERR_TIMEOUT).  Returns OS2_ERR_CUDA if the synchronisation or the
 * read fails. */
os2_status os2_get_status(void *stream);

/* Self-test of the device-side failure detection (the pages have no
 * counterpart: it checks this library's own safeguard).  Every mbarrier wait
 * of the tensor-core kernels gives up after a bounded number of clock cycles,
 * or when its CTA's abort flag is raised, and then records OS2_ERR_TIMEOUT.
 * This enqueues one CTA on `stream` whose wait on an mbarrier that nothing
 * arrives at runs out after `limit_cycles` SM clock cycles
 * (1 <= limit_cycles <= 2^34; 2e6 is about a millisecond).  The device status
 * word then holds OS2_ERR_TIMEOUT (read and clear it with os2_get_status) and
 * the context stays usable.  If `result` (caller-owned device memory, 8
 * int32) is not NULL it receives: [0] 1 if a satisfied wait completed, [1] 1
 * if the unsatisfied wait gave up, [2] the same for the cluster-scope wait,
 * [3] 1 if a raised abort flag ended a wait early, [4] 1 if the timed-out
 * wait lasted at least limit_cycles; [5..7] 0.  Returns OS2_ERR_INVALID_ARG
 * for a limit out of range (nothing enqueued). */
os2_status os2_wait_selftest(long long limit_cycles, int32_t *result, void *stream);

/* Selects the kernel of steps 4 and 5 (process-wide; default OS2_CRT_AUTO).
 * All give bit-identical results.  OS2_CRT_TC computes the sums
 * sum_l (c_l + 128) W_l as an FP16 tensor-core product of the residues with
 * the signed 10-bit digits of the W_l, exact in FP32; it needs rows of c that
 * are 16-byte aligned (the CUDA-core kernel is used otherwise).  It cannot run
 * beside a product (it needs TMEM and shared memory a product CTA holds), so
 * with OS2_CRT_TC os2_gemm runs in one pass (one product launch).  With
 * OS2_CRT_SIMT, os2_gemm cuts A into row panels for m >= 4096 and runs each
 * panel's reconstruction on the CUDA cores beside the next panel's product,
 * and os2_gemm_host does the same per block.  OS2_CRT_AUTO: the panels and
 * blocks as with OS2_CRT_SIMT, and the tensor-core kernel for every
 * reconstruction that runs alone (os2_crt, os2_gemm with one panel).
 * OS2_ERR_INVALID_ARG for another value. */
os2_status os2_set_crt_variant(int variant);

/* Selects the step-3 kernel used by os2_gemm and the other whole-path entry
 * points (process-wide; default OS2_GEMM_TC).  All give identical results. */
os2_status os2_set_gemm_variant(int variant);

/* Static description of a status code. */
const char *os2_status_string(int status);

/* Number of kernels os2_gemm launches for these arguments with the step-3
 * kernel currently selected (for launch accounting); 0 on bad args. */
int os2_gemm_launch_count(int m, int n, int k, int num_moduli, int mode);

/* Per-kernel timing of os2_gemm / os2_gemm_host and the other whole-path
 * entry points (a measurement aid; the pages define no such call).
 * os2_profile_start() enables it: every kernel (or group of panel launches)
 * those calls enqueue is then bracketed by two CUDA events on the stream it
 * runs on (the caller's stream or one of the library's side streams, where a
 * span includes the time it waits beside other work).  os2_profile_stop()
 * disables it, waits for the recorded events, and writes up to max_kernels
 * aggregated entries: names[i*32..] (NUL-terminated role: scale, scale_bars,
 * gemm_bound, residues, gemm_modp, crt_unscale, complex_stack,
 * complex_unstack), total_ms[i] and launches[i] (spans recorded).  Returns
 * the entry count, or -1 if an event failed.  Any output pointer may be NULL.
 * Process-wide, not thread-safe against concurrent calls on other threads. */
os2_status os2_profile_start(void);
int os2_profile_stop(int max_kernels, char *names, double *total_ms, int *launches);

/* Pipe-peak probes (a measurement aid; the pages have no counterpart): the
 * throughput ceiling of the tensor-core instructions this library can use on
 * sm_103a, from its own kernels, as a same-pipe denominator for step 3.
 *   OS2_PROBE_F16_1SM  tcgen05.mma kind::f16, cta_group::1, 128x256x16 per
 *                      instruction, one CTA per SM
 *   OS2_PROBE_F16_2SM  tcgen05.mma kind::f16, cta_group::2, 256x256x16 per
 *                      instruction, CTA pairs (the form step 3 uses)
 *   OS2_PROBE_S8_SYNC  mma.sync m16n8k32 s8 x s8 -> s32 (INT8 tensor path
 *                      outside tcgen05; sm_103a has no tcgen05 kind::i8)
 * Operands are small integers resident in shared memory (tcgen05) or
 * registers (mma.sync), so every product is exact.  Enqueues one launch of
 * `iters` rounds (each round: K = 64 per accumulator tile; for mma.sync eight
 * independent m16n8k32 per warp) on `stream` and writes to *flop (host, may be
 * NULL) the flops it performs, counting a multiply-add as 2.  With check != 0
 * the result is compared with the exact product on the CUDA cores and
 * result[0] (device int32[4], zeroed by this call) receives the mismatches,
 * result[1] the number of CTAs that checked; time only runs with check = 0
 * (result may then be NULL).  iters in [1, 2^24]; check runs of
 * OS2_PROBE_S8_SYNC need iters <= 4096 (int32 sums).  Bounded waits as in the
 * GEMM kernels (OS2_ERR_TIMEOUT in the status word on expiry). */
typedef enum {
  OS2_PROBE_F16_1SM = 0,
  OS2_PROBE_F16_2SM = 1,
  OS2_PROBE_S8_SYNC = 2
} os2_probe_kind;
os2_status os2_peak_probe(int kind, int iters, int check, int32_t *result, double *flop,
                          void *stream);

/* os2_gemm without a caller-supplied workspace, for callers that cannot
 * allocate device memory where they call it: a host library or plugin whose
 * device memory is planned and owned by another allocator (an inference
 * runtime's arena, a framework's caching allocator) and which has no
 * workspace to hand over, or a latency-critical loop that must not call
 * cudaMalloc/cudaFree because those calls can synchronise the whole device.
 * The pages have no counterpart of this call; it only changes where the
 * scratch lives.
 *
 * The scratch is one static device array of OS2_NOALLOC_SCRATCH_BYTES
 * (128 MiB) inside libos2; every GPU that loads the library holds it until
 * the process exits.  Problems whose os2_workspace_size exceeds it are
 * rejected with OS2_ERR_WORKSPACE before anything is enqueued (for example
 * m = n = k = 1024 fits for every num_moduli <= 20; at 2048^3 only
 * num_moduli <= 6 fits).  With k = 0 it only zeroes C, whatever the sizes.
 * It runs the five steps in one pass on `stream`, never through os2_gemm's
 * row-panel pipeline (which creates library streams and events on first
 * use), so for m >= 4096 it gives the same results a little more slowly.
 * The first call on a device looks up the array's device address with that
 * device current (make that first call before any stream capture); later
 * calls reuse it.  Nothing here calls cudaMalloc, cudaFree or an allocating
 * library routine.  Every call uses the same array and the array keeps the
 * previous call's contents (each call clears what it needs zeroed), so calls
 * that overlap on the GPU -- on different streams or from different threads
 * -- race and corrupt each other's results: serialise them.  Arguments,
 * layouts, errors and results are those of os2_gemm. */
#define OS2_NOALLOC_SCRATCH_BYTES (128u << 20)
os2_status os2_gemm_noalloc(int m, int n, int k, const double *A, int lda, const double *B,
                            int ldb, double *C, int ldc, int num_moduli, int mode, void *stream);

#ifdef __cplusplus
}
#endif
#endif /* OS2_H */
