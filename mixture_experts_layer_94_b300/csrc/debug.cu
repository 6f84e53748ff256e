// debug.cu — a controlled stall for testing failure detection.
//
// One warp initialises an mbarrier that nothing ever arrives at and waits on
// it with the same bounded wait the GEMM pipeline uses, only with a short
// limit. The wait gives up, records the timeout in the workspace error word
// and the kernel returns, so the host reads MOE_ERR_TIMEOUT through
// moe_get_device_status and the CUDA context stays usable.
#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace moe {
namespace {

__global__ void __launch_bounds__(32) stall_wait_kernel(uint32_t* err, uint64_t limit_ns) {
  pdl_trigger();
  pdl_wait();
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  const uint32_t b = ptx::smem_u32(&bar);
  if (threadIdx.x == 0) {
    ptx::mbar_init(b, 1);
    abort_flag = 0;
    ptx::fence_mbarrier_init();
  }
  __syncwarp();
  if (threadIdx.x == 0) ptx::mbar_wait(b, 0, &abort_flag, err, limit_ns);  // nothing ever arrives
  __syncwarp();
}

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_debug_stall_wait(void* ws, size_t ws_bytes, uint32_t timeout_us, void* stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u) != 0 || ws_bytes < 256) return MOE_ERR_WORKSPACE;
  if (timeout_us == 0 || timeout_us > 1000000u) return MOE_ERR_INVALID_ARG;
  return moe::launch(moe::stall_wait_kernel, 1, 32, 0, static_cast<cudaStream_t>(stream), static_cast<uint32_t*>(ws),
                     (uint64_t)timeout_us * 1000ull) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}
