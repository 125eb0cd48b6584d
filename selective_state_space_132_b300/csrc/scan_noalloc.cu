// ssm_scan_fwd_noalloc: the selective scan for callers that cannot allocate.
//
// ssm_scan_fwd needs a caller-provided workspace when a long sequence is split
// over time chunks (the per-chunk end states and step sums live there).  Some
// callers cannot get one on the call path: a plugin hosted by another runtime
// that owns all device memory and exposes no allocator, a latency-critical loop
// where cudaMalloc's implicit device synchronisation is not acceptable, or a
// process that must stay inside the memory it reserved at start-up.  This entry
// point runs the same kernels with that scratch taken from a fixed buffer that is
// part of the library image instead.
//
// The buffer is a file-scope __device__ array of SSM_NOALLOC_SCRATCH_BYTES; every
// GPU that loads the library holds it until the process exits.  In host code the
// array's name is only a host-side stand-in, so its device address is looked up
// with cudaGetSymbolAddress once per device (with that device current) on the
// first call made on the device, and that address is what the kernels receive.
#include "../../include/ssm.h"

#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace ssm {
ssm_status check_scan_args(const ssm_scan_args *a);
}

namespace {

static __device__ __align__(256) unsigned char g_scan_scratch[SSM_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of g_scan_scratch on the current device (looked up once per device).
cudaError_t scratch_for_current_device(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scan_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" ssm_status ssm_scan_fwd_noalloc(const ssm_scan_args *args, ssm_stream_t stream) {
    if (!args) return SSM_ERR_INVALID_ARG;
    // Validate everything except the workspace fields, which this entry point ignores.
    ssm_scan_args a = *args;
    a.workspace = nullptr;
    a.workspace_bytes = 0;
    size_t need = 0;
    ssm_status s = ssm::check_scan_args(&a);
    if (s != SSM_OK) return s;
    s = ssm_scan_workspace_size(&a, &need);
    if (s != SSM_OK) return s;
    if (need > SSM_NOALLOC_SCRATCH_BYTES) return SSM_ERR_UNSUPPORTED;  // before any CUDA call
    if (a.batch == 0 || a.dim == 0) return ssm_scan_fwd(&a, stream);  // no launch, no scratch
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return SSM_ERR_CUDA;
    // Start from a clean status word; the chunk summaries are always written by the
    // summary pass before the output pass reads them, so they need no clearing.
    if (cudaMemsetAsync(scratch, 0, ssm::kStatusBytes, reinterpret_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return SSM_ERR_CUDA;
    a.workspace = scratch;
    a.workspace_bytes = SSM_NOALLOC_SCRATCH_BYTES;
    return ssm_scan_fwd(&a, stream);
}
