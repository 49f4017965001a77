// Failure-path probe: one thread waits, with the same bounded wait the SSD
// kernels use, on an mbarrier that nothing ever arrives at.  When the bound
// runs out it records SSD_ERR_DEVICE_TIMEOUT in the status word and returns,
// so the host can check that the error surfaces without the GPU hanging.
#include "ptx.cuh"
#include "ssd_internal.cuh"

namespace ssd {
namespace {

__global__ void timeout_probe_kernel(int* status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0 && !mbar_wait(&bar, 0, limit_ns)) atomicExch(status, static_cast<int>(SSD_ERR_DEVICE_TIMEOUT));
}

}  // namespace

cudaError_t launch_timeout_probe(int* status, uint64_t limit_ns, cudaStream_t stream) {
  timeout_probe_kernel<<<1, 32, 0, stream>>>(status, limit_ns);
  return cudaGetLastError();
}

}  // namespace ssd
