// debug.cu — diagnostic kernel that exercises the engine's bounded wait.
//
// One thread waits, through the same wait_phase() every pipeline role uses, on
// an mbarrier phase that nothing will ever complete.  After limit_ns the wait
// gives up, ORPO_STATUS_TIMEOUT is OR-ed into *status and the kernel returns
// normally, so the CUDA context stays usable.  Used by the failure-detection test.
#include "../../include/orpo_head.h"
#include "engine.cuh"
#include "internal.h"

namespace orpo {
namespace {

__global__ void wait_timeout_kernel(int32_t* status, uint64_t limit_ns) {
  __shared__ SmemCtl ctl;
  if (threadIdx.x != 0) return;
  ctl.abort_flag = 0;
  mbar_init(&ctl.drain, 1);
  fence_mbar_init();
  wait_phase<1>(&ctl, &ctl.drain, 0, status, limit_ns);  // nobody arrives on this barrier
}

}  // namespace
}  // namespace orpo

extern "C" int orpo_debug_wait_timeout(int32_t* status, int64_t limit_ns, void* stream) {
  if (!status) return ORPO_ERR_NULL;
  if (limit_ns < 1000 || limit_ns > 2000000000ll) return ORPO_ERR_ARG;
  orpo::wait_timeout_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(status, (uint64_t)limit_ns);
  return cudaGetLastError() == cudaSuccess ? ORPO_OK : ORPO_ERR_CUDA;
}
