// Diagnostic entry point: shows that a bounded wait which runs out becomes a device
// status the host can read, with the CUDA context left usable.  The kernel waits,
// through the same acquire-and-back-off routine the SSD kernel uses to take over the
// state of the block before it, on a flag that nothing ever sets.
#include "../../include/ssm.h"

#include <cuda_runtime.h>

#include "common.cuh"
#include "ptx.cuh"

namespace ssm {
namespace {

// The flag lives in the padding of the 256-byte status header.
constexpr int kFlagWord = 32;

__global__ void bounded_wait_kernel(DeviceStatus *status, long long budget) {
    const uint32_t *flag = reinterpret_cast<const uint32_t *>(status) + kFlagWord;
    if (!ptx::wait_flag(flag, budget)) report_status(status, SSM_ERR_TIMEOUT, 90);
}

}  // namespace
}  // namespace ssm

extern "C" ssm_status ssm_check_bounded_wait(void *workspace, int64_t budget_cycles,
                                             ssm_stream_t stream) {
    if (!workspace || budget_cycles < 1 || budget_cycles > ssm::ptx::kWaitCycles)
        return SSM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(workspace) % 256 != 0) return SSM_ERR_ALIGNMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaMemsetAsync(workspace, 0, ssm::kStatusBytes, st) != cudaSuccess) return SSM_ERR_CUDA;
    ssm::bounded_wait_kernel<<<1, 1, 0, st>>>(static_cast<ssm::DeviceStatus *>(workspace),
                                              static_cast<long long>(budget_cycles));
    return cudaGetLastError() == cudaSuccess ? SSM_OK : SSM_ERR_CUDA;
}
