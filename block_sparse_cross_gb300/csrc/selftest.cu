// Diagnostic kernel for the bounded waits of the pipelines: an mbarrier wait
// that nothing can satisfy must give up after the wait limit, raise the CTA's
// abort flag (which a second waiting role observes and stops on) and report
// SPLITKV_ETIMEOUT to the host, leaving the context usable.
#include "kernels.h"
#include "tc_common.cuh"

namespace skv {

namespace {

__device__ int g_selftest_status;

__global__ void wait_probe_kernel() {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    tc::mbar_init(&bar, 1);
    abort_flag = 0;
    tc::fence_mbar_init();
  }
  __syncthreads();
  // warp 0: the role whose wait runs out (nothing ever arrives on `bar`);
  // warp 1: another role waiting on the same barrier, which stops once the
  // abort flag is up (or at its own limit)
  const bool ok = tc::mbar_wait(&bar, 0, (volatile int*)&abort_flag);
  __syncthreads();
  if (threadIdx.x == 0)
    g_selftest_status = (!ok && abort_flag) ? (int)SPLITKV_ETIMEOUT : (int)SPLITKV_OK;
}

}  // namespace

cudaError_t run_wait_probe(int* status, cudaStream_t st) {
  const int z = -1;
  cudaError_t e = cudaMemcpyToSymbolAsync(g_selftest_status, &z, sizeof(int), 0,
                                          cudaMemcpyHostToDevice, st);
  if (e != cudaSuccess) return e;
  wait_probe_kernel<<<1, 64, 0, st>>>();
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return e;
  return cudaMemcpyFromSymbol(status, g_selftest_status, sizeof(int));
}

}  // namespace skv
