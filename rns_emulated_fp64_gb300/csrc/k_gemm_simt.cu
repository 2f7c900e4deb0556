// Step 3, exact reference variant on the CUDA cores: the N residue products
// G_l = R_A,l R_B,l^T accumulated in int32 ([Q] "誤差のないINT8行列積(手順3)":
// exact while the inner dimension stays below 2^17).  Slow; used to cross-check
// the tensor-core kernel and to expose raw int32 products.
#include <cuda_fp16.h>

#include "os2_internal.cuh"

namespace {

constexpr int TB = 64, TK = 32, kThreads = 256;

template <int OUT>
__global__ void __launch_bounds__(kThreads)
    k_gemm_simt(int m, int n, int kp, const __half *__restrict__ RA,
                const __half *__restrict__ RB, void *__restrict__ out, int ldo,
                const GemmConsts gc) {
  __shared__ int sA[TK][TB + 1], sB[TK][TB + 1];
  const int l = blockIdx.z;
  const __half *A = RA + (size_t)l * m * kp;
  const __half *B = RB + (size_t)l * n * kp;
  const int tm = blockIdx.y * TB, tn = blockIdx.x * TB;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  int acc[4][4] = {};
  for (int k0 = 0; k0 < kp; k0 += TK) {
    for (int idx = threadIdx.x; idx < TB * TK; idx += kThreads) {
      const int r = idx / TK, kk = idx % TK;
      sA[kk][r] = tm + r < m ? __half2int_rn(A[(size_t)(tm + r) * kp + k0 + kk]) : 0;
      sB[kk][r] = tn + r < n ? __half2int_rn(B[(size_t)(tn + r) * kp + k0 + kk]) : 0;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < TK; kk++)
#pragma unroll
      for (int a = 0; a < 4; a++)
#pragma unroll
        for (int b = 0; b < 4; b++) acc[a][b] += sA[kk][ty * 4 + a] * sB[kk][tx * 4 + b];
    __syncthreads();
  }
  const int p = (int)gc.p[l], hi = (int)gc.hi[l], lo = (int)gc.lo[l];
  for (int a = 0; a < 4; a++)
    for (int b = 0; b < 4; b++) {
      const int row = tm + ty * 4 + a, col = tn + tx * 4 + b;
      if (row >= m || col >= n) continue;
      const size_t o = ((size_t)l * m + row) * ldo + col;
      if (OUT == OS2_OUT_RAW_INT32) {
        reinterpret_cast<int32_t *>(out)[o] = acc[a][b];
      } else {
        int r = acc[a][b] % p;
        r = r > hi ? r - p : r;
        r = r < lo ? r + p : r;
        reinterpret_cast<int8_t *>(out)[o] = (int8_t)r;
      }
    }
}

}  // namespace

cudaError_t launch_gemm_simt(int m, int n, int kp, const void *RA, const void *RB, int N,
                             int out_kind, void *out, int ldo, const Os2Tables *t, cudaStream_t s) {
  if (m <= 0 || n <= 0 || N <= 0) return cudaSuccess;
  dim3 grid((n + TB - 1) / TB, (m + TB - 1) / TB, N);
  const __half *a = reinterpret_cast<const __half *>(RA);
  const __half *b = reinterpret_cast<const __half *>(RB);
  if (out_kind == OS2_OUT_RAW_INT32)
    k_gemm_simt<OS2_OUT_RAW_INT32><<<grid, kThreads, 0, s>>>(m, n, kp, a, b, out, ldo, t->gemm);
  else
    k_gemm_simt<OS2_OUT_MODP_INT8><<<grid, kThreads, 0, s>>>(m, n, kp, a, b, out, ldo, t->gemm);
  return cudaGetLastError();
}
