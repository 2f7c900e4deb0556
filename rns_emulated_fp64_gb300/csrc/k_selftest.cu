// Self-test of the device-side failure detection.
//
// Every wait of the tensor-core kernels on an mbarrier is bounded: it gives up
// after a number of clock cycles, or as soon as the CTA's abort flag is
// raised, and the kernel then records OS2_ERR_TIMEOUT in the device status
// word and returns, so a lost arrival never hangs the GPU.  This kernel makes
// those same waits run out on purpose, on an mbarrier that no thread ever
// arrives at, and reports what they did.
#include "os2_internal.cuh"
#include "ptx.cuh"

using namespace os2ptx;

namespace {

__global__ void k_wait_selftest(long long limit, int *status, int32_t *result) {
  __shared__ uint64_t bars[2];
  __shared__ int s_abort;
  if (threadIdx.x != 0) return;
  mbar_init(&bars[0], 1);  // never arrived at
  mbar_init(&bars[1], 1);  // arrived at once
  s_abort = 0;
  fence_mbar_init();
  volatile int *abort = &s_abort;
  int32_t r[8] = {0, 0, 0, 0, 0, 0, 0, 0};

  mbar_arrive(&bars[1]);
  r[0] = mbar_wait_bounded(&bars[1], 0, abort, limit) ? 1 : 0;

  const long long t0 = clock64();
  const bool done = mbar_wait_bounded(&bars[0], 0, abort, limit);
  const long long waited = clock64() - t0;
  r[1] = done ? 0 : 1;
  r[4] = waited >= limit ? 1 : 0;
  if (!done && status) atomicCAS(status, 0, OS2_ERR_TIMEOUT);

  r[2] = mbar_wait_cluster_bounded(&bars[0], 0, abort, limit) ? 0 : 1;

  // a raised abort flag ends a wait long before its limit
  s_abort = 1;
  const long long t1 = clock64();
  const bool done2 = mbar_wait_bounded(&bars[0], 0, abort, 1LL << 40);
  r[3] = (!done2 && clock64() - t1 < (1LL << 30)) ? 1 : 0;

  if (result)
    for (int i = 0; i < 8; i++) result[i] = r[i];
}

}  // namespace

cudaError_t launch_wait_selftest(long long limit, int *status, int32_t *result, cudaStream_t s) {
  k_wait_selftest<<<1, 32, 0, s>>>(limit, status, result);
  return cudaGetLastError();
}
