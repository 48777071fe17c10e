// conv2d_fwd_noalloc: the forward convolution for callers that cannot allocate
// device memory at all, so cannot hand conv2d_fwd a workspace.  Examples are
// plugins whose host framework owns every device allocation and offers no
// workspace hook, deployments with a fixed device-memory budget that forbid
// allocation after start-up, and latency-critical loops that must not call
// cudaMalloc/cudaFree because those calls can synchronise the whole device.
//
// The workspace (status word + one split-K semaphore per output tile) lives in
// a file-scope device array of CONV2D_NOALLOC_SCRATCH_BYTES bytes instead.
// Every GPU that loads this library holds that array until the process exits.
// In host code `g_noalloc_scratch` only names a host-side stand-in, so its
// device address is looked up with cudaGetSymbolAddress once per device (with
// that device current) on the first call made on that device and kept for the
// life of the process.  A device reset unloads the module that holds the array,
// so the kept address is only valid while the device's primary context lives.
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>
#include <mutex>

#include "conv2d.h"

namespace sgb {
size_t fwd_workspace_bytes_min(const conv2d_params* params);  // conv2d_api.cu
}

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[CONV2D_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};  // device address of the array, per device ordinal

// Device address of the scratch array on the current device (looked up once per device).
int scratch_on_current_device(void** out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CONV2D_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return CONV2D_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return CONV2D_OK;
}

}  // namespace

extern "C" int conv2d_fwd_noalloc(const conv2d_params* params, const void* x_dev, const void* w_dev,
                                  const float* bias_dev, float* y_dev, conv2d_stream_t stream)
{
    const size_t need = sgb::fwd_workspace_bytes_min(params);
    if (need == 0)  // invalid params: let the regular entry point report exactly why
        return conv2d_fwd(params, x_dev, w_dev, bias_dev, y_dev, nullptr, 0, stream);
    if (need > CONV2D_NOALLOC_SCRATCH_BYTES) return CONV2D_ERR_SCRATCH_LIMIT;
    void* scratch = nullptr;
    int rc = scratch_on_current_device(&scratch);
    if (rc != CONV2D_OK) return rc;
    // The array keeps whatever the previous call left (a timed-out call leaves
    // semaphores set), so the part this call uses is cleared first, in stream order.
    if (cudaMemsetAsync(scratch, 0, need, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    return conv2d_fwd(params, x_dev, w_dev, bias_dev, y_dev, scratch, need, stream);
}
