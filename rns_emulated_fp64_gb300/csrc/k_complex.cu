// Complex products (ZGEMM / CGEMM) on the real path.
//
// [G] "Improved Scaling for Fast Mode of Ozaki Scheme II", "Bedeutung": the
// approach applies to complex matrix products (ZGEMM/CGEMM).  A complex
// product is the real block product
//     [C_r | C_i] = [A_r | A_i] . [[B_r, B_i], [-B_i, B_r]]
// of size m x 2n x 2k, so the five steps run unchanged on the stacked real
// operands: the scaling of a stacked row covers |a_r|^2 + |a_i|^2 (the complex
// row norm), every integer product stays exact, and the CRT bound covers the
// real and imaginary parts together.  These kernels only move data:
//   k_stack_a   A (m x k complex, interleaved)   -> A2 (m x 2k real)
//   k_stack_b   B (n columns of k complex)       -> Bt2 (2n x 2k real)
//   k_unstack_c C2 (m x 2n real)                 -> C (m x n complex, interleaved)
#include "os2_internal.cuh"

namespace {

constexpr int kThreads = 256;

template <typename T>
__global__ void k_stack_a(int m, int k, const T *__restrict__ A, long lda, T *__restrict__ A2) {
  const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (idx >= (long long)m * k) return;
  const int i = (int)(idx / k), h = (int)(idx - (long long)i * k);
  const T re = A[2 * ((size_t)i * lda + h)], im = A[2 * ((size_t)i * lda + h) + 1];
  A2[(size_t)i * 2 * k + h] = re;
  A2[(size_t)i * 2 * k + k + h] = im;
}

template <typename T>
__global__ void k_stack_b(int n, int k, const T *__restrict__ B, long ldb, T *__restrict__ Bt2) {
  const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (idx >= (long long)n * k) return;
  const int j = (int)(idx / k), h = (int)(idx - (long long)j * k);
  const T re = B[2 * ((size_t)j * ldb + h)], im = B[2 * ((size_t)j * ldb + h) + 1];
  T *rr = Bt2 + (size_t)j * 2 * k;        // column j of C_r: ( b_r ; -b_i )
  T *ri = Bt2 + (size_t)(n + j) * 2 * k;  // column j of C_i: ( b_i ;  b_r )
  rr[h] = re;
  rr[k + h] = -im;
  ri[h] = im;
  ri[k + h] = re;
}

template <typename T>
__global__ void k_unstack_c(int m, int n, const T *__restrict__ C2, T *__restrict__ C, long ldc) {
  const long long idx = (long long)blockIdx.x * kThreads + threadIdx.x;
  if (idx >= (long long)m * n) return;
  const int i = (int)(idx / n), j = (int)(idx - (long long)i * n);
  C[2 * ((size_t)i * ldc + j)] = C2[(size_t)i * 2 * n + j];
  C[2 * ((size_t)i * ldc + j) + 1] = C2[(size_t)i * 2 * n + n + j];
}

unsigned blocks(long long count) { return (unsigned)((count + kThreads - 1) / kThreads); }

}  // namespace

cudaError_t launch_complex_stack(bool f32, int m, int n, int k, const void *A, long lda,
                                 const void *B, long ldb, void *A2, void *Bt2, cudaStream_t s) {
  if ((long long)m * k > 0) {
    if (f32)
      k_stack_a<float><<<blocks((long long)m * k), kThreads, 0, s>>>(
          m, k, static_cast<const float *>(A), lda, static_cast<float *>(A2));
    else
      k_stack_a<double><<<blocks((long long)m * k), kThreads, 0, s>>>(
          m, k, static_cast<const double *>(A), lda, static_cast<double *>(A2));
  }
  if ((long long)n * k > 0) {
    if (f32)
      k_stack_b<float><<<blocks((long long)n * k), kThreads, 0, s>>>(
          n, k, static_cast<const float *>(B), ldb, static_cast<float *>(Bt2));
    else
      k_stack_b<double><<<blocks((long long)n * k), kThreads, 0, s>>>(
          n, k, static_cast<const double *>(B), ldb, static_cast<double *>(Bt2));
  }
  return cudaGetLastError();
}

cudaError_t launch_complex_unstack(bool f32, int m, int n, const void *C2, void *C, long ldc,
                                   cudaStream_t s) {
  if ((long long)m * n <= 0) return cudaSuccess;
  if (f32)
    k_unstack_c<float><<<blocks((long long)m * n), kThreads, 0, s>>>(
        m, n, static_cast<const float *>(C2), static_cast<float *>(C), ldc);
  else
    k_unstack_c<double><<<blocks((long long)m * n), kThreads, 0, s>>>(
        m, n, static_cast<const double *>(C2), static_cast<double *>(C), ldc);
  return cudaGetLastError();
}
