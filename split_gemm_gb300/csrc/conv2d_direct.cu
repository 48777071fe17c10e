// Instantiations of the direct grouped-convolution kernel (conv2d_direct.cuh),
// one per channel count of a group.
#include <cuda_runtime.h>

#include "conv2d_direct.cuh"

namespace sgb {

template <int CG>
cudaError_t launch_conv2d_direct(const DirectParams& kp, int grid, cudaStream_t stream)
{
    const long long smem = conv2d_direct_smem_bytes(kp.K, kp.R, kp.S, CG);
    if (smem > 232448) return cudaErrorInvalidValue;
    auto kern = conv2d_direct_kernel<CG>;
    if (smem > 48 * 1024) {
        cudaError_t err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
        if (err != cudaSuccess) return err;
    }
    kern<<<grid, DIRECT_THREADS, static_cast<size_t>(smem), stream>>>(kp);
    return cudaGetLastError();
}

template SGB_DIRECT_SIG(1);
template SGB_DIRECT_SIG(2);
template SGB_DIRECT_SIG(4);
template SGB_DIRECT_SIG(8);
template SGB_DIRECT_SIG(16);

}  // namespace sgb
