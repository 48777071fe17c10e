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

namespace {
__global__ void __launch_bounds__(256) expand_blockdiag_kernel(const uint4* __restrict__ w, uint4* __restrict__ wb,
                                                              int K, int taps, int cg)
{
    const long long chunks = static_cast<long long>(K) * taps * 8;  // 16-byte chunks of wb (8 per 64-channel row)
    const int cpg = cg / 8;                                          // chunks per group row of w
    for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < chunks;
         i += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long row = i >> 3;  // (k, tap)
        const int chunk = static_cast<int>(i & 7);
        const int k = static_cast<int>(row / taps);
        const int slot = (k / cg) % (64 / cg);  // k's group's place in its 64-channel block
        const int j = chunk - slot * cpg;       // chunk within the group's cg channels
        wb[i] = (j >= 0 && j < cpg) ? w[row * cpg + j] : make_uint4(0u, 0u, 0u, 0u);
    }
}
}  // namespace

cudaError_t launch_expand_blockdiag(const uint16_t* w, uint16_t* wb, int K, int taps, int cg, cudaStream_t stream)
{
    if (cg != 8 && cg != 16 && cg != 32) return cudaErrorInvalidValue;
    const long long chunks = static_cast<long long>(K) * taps * 8;
    long long grid = (chunks + 255) / 256;
    if (grid > 1184) grid = 1184;  // 8 x 148 SMs' worth; the loop covers the rest
    if (grid < 1) grid = 1;
    expand_blockdiag_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(reinterpret_cast<const uint4*>(w),
                                                                         reinterpret_cast<uint4*>(wb), K, taps, cg);
    return cudaGetLastError();
}

template SGB_DIRECT_SIG(1);
template SGB_DIRECT_SIG(2);
template SGB_DIRECT_SIG(4);
template SGB_DIRECT_SIG(8);
template SGB_DIRECT_SIG(16);

}  // namespace sgb
