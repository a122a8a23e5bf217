// A kernel whose barrier wait can never complete, run through the same
// bounded wait the tensor-core kernels use: it shows that a stuck wait ends
// with the timeout bit in the status word (and an orderly exit) instead of
// a hung GPU.
#include <cuda_runtime.h>

#include <string>

#include "plan.h"
#include "sm100.cuh"

namespace pds {
namespace {

__global__ void stuck_wait_kernel(uint32_t* status, uint64_t limit_ns, uint32_t* gave_up) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(sm100::smem_u32(&bar), 1);  // one arrival expected; none will come
    abort_flag = 0;
    sm100::mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const bool ok = sm100::mbar_wait(sm100::smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    *gave_up = ok ? 0u : 1u;
  }
}

}  // namespace

pds_status run_stuck_wait(uint32_t limit_us, cudaStream_t st, std::string* err) {
  uint32_t* dev = nullptr;  // [0] status word, [1] gave-up flag
  cudaError_t ce = cudaMallocAsync(&dev, 2 * sizeof(uint32_t), st);
  if (ce == cudaSuccess) ce = cudaMemsetAsync(dev, 0, 2 * sizeof(uint32_t), st);
  if (ce != cudaSuccess) {
    *err = std::string("stuck-wait probe setup: ") + cudaGetErrorString(ce);
    return PDS_ENOMEM;
  }
  stuck_wait_kernel<<<1, 32, 0, st>>>(dev, static_cast<uint64_t>(limit_us) * 1000ull, dev + 1);
  uint32_t host[2] = {0, 0};
  ce = cudaGetLastError();
  if (ce == cudaSuccess) ce = cudaMemcpyAsync(host, dev, sizeof(host), cudaMemcpyDeviceToHost, st);
  if (ce == cudaSuccess) ce = cudaStreamSynchronize(st);
  cudaFreeAsync(dev, st);
  if (ce != cudaSuccess) {
    *err = std::string("stuck-wait probe: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  if ((host[0] & kStatusTimeout) && host[1]) {
    *err = "the probe's bounded wait gave up after " + std::to_string(limit_us) + " us";
    return PDS_ETIMEOUT;
  }
  return PDS_OK;  // the wait completed: cannot happen, nothing arrives
}

}  // namespace pds
