// A kernel whose barrier wait can never complete, run through the same
// bounded wait the tensor-core kernels use: it shows that a stuck wait ends
// with the timeout bit in the status word (and an orderly exit) instead of
// a hung GPU.  It reports through the component entry points' status word,
// which pds_component_sync reads and clears.
#include <cuda_runtime.h>

#include <string>

#include "plan.h"
#include "sm100.cuh"

namespace pds {
namespace {

__global__ void stuck_wait_kernel(uint32_t* status, uint64_t limit_ns) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    sm100::mbar_init(sm100::smem_u32(&bar), 1);  // one arrival expected; none will come
    abort_flag = 0;
    sm100::mbar_init_fence();
  }
  __syncthreads();
  if (threadIdx.x == 0) sm100::mbar_wait(sm100::smem_u32(&bar), 0, &abort_flag, status, limit_ns);
}

}  // namespace

pds_status run_stuck_wait(uint32_t limit_us, cudaStream_t st, std::string* err) {
  uint32_t* status = component_status(err);
  if (!status) return PDS_ELAUNCH;
  stuck_wait_kernel<<<1, 32, 0, st>>>(status, static_cast<uint64_t>(limit_us) * 1000ull);
  const cudaError_t ce = cudaGetLastError();
  if (ce != cudaSuccess) {
    *err = std::string("stuck-wait probe: ") + cudaGetErrorString(ce);
    return PDS_ELAUNCH;
  }
  return PDS_OK;
}

}  // namespace pds
