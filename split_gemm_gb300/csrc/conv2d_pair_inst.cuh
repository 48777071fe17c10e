// Launchers of the CTA-pair kernel and their explicit instantiations (64-, 128- and
// 256-channel tiles) for SGB_PAIR_KBS k-blocks per stage; included by one translation
// unit per stage depth so that the variants compile in parallel.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "conv2d_pair.cuh"

namespace sgb {

namespace {

template <int BN, int KBS>
auto pair_kernel(bool fused)
{
    return fused ? conv2d_fwd_pair_kernel<BN, KBS, true> : conv2d_fwd_pair_kernel<BN, KBS, false>;
}

// The dynamic shared-memory opt-in is per device and instantiation; remember which have it.
template <int BN, int KBS>
cudaError_t pair_configure(bool fused)
{
    static unsigned long long configured[2] = {0ull, 0ull};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (__atomic_load_n(&configured[fused], __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    err = cudaFuncSetAttribute(pair_kernel<BN, KBS>(fused), cudaFuncAttributeMaxDynamicSharedMemorySize,
                               PairConfig<BN, KBS>::SMEM_BYTES);
    if (err != cudaSuccess) return err;
    if (bit) __atomic_fetch_or(&configured[fused], bit, __ATOMIC_RELEASE);
    return cudaSuccess;
}

template <int BN, int KBS>
void pair_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, cudaStream_t stream)
{
    using Cfg = PairConfig<BN, KBS>;
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg->blockDim = dim3(Cfg::THREADS);
    cfg->dynamicSmemBytes = static_cast<size_t>(Cfg::SMEM_BYTES);
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // Programmatic stream serialization: the launch may start while the previous
    // kernel drains; the kernel waits for it before touching global memory.
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg->attrs = attr;
    cfg->numAttrs = 2;
}

}  // namespace

template <int BN, int KBS>
cudaError_t launch_conv2d_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const ConvKernelParams& kp, int pairs,
                               cudaStream_t stream)
{
    const bool fused = (kp.relu | kp.out_bf16) != 0;
    cudaError_t err = pair_configure<BN, KBS>(fused);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_launch_config<BN, KBS>(&cfg, attr, pairs, stream);
    return cudaLaunchKernelEx(&cfg, pair_kernel<BN, KBS>(fused), tm_a, tm_b, kp);
}

// Clusters of two CTAs of this instantiation that the current device holds at
// once (one CTA per SM; both SMs of a pair must be free), looked up once per
// device.  0 when the query fails.
template <int BN, int KBS>
int conv2d_pair_max_resident(bool fused)
{
    static int cached[2][64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64 && __atomic_load_n(&cached[fused][dev], __ATOMIC_ACQUIRE) > 0) return cached[fused][dev];
    if (pair_configure<BN, KBS>(fused) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_launch_config<BN, KBS>(&cfg, attr, 1, nullptr);
    cfg.numAttrs = 1;  // the cluster shape only
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair_kernel<BN, KBS>(fused), &cfg) != cudaSuccess) return 0;
    if (dev < 64 && n > 0) __atomic_store_n(&cached[fused][dev], n, __ATOMIC_RELEASE);
    return n;
}

#ifndef SGB_PAIR_KBS
#error "define SGB_PAIR_KBS (k-blocks per stage) before including this file"
#endif
#if SGB_PAIR_KBS == 2
// The halo loader's kernels (two or three taps per stage) live in this translation unit.
namespace {
template <int BN, int TAPS>
auto pair_halo_kernel(bool fused)
{
    return fused ? conv2d_fwd_pair_halo_kernel<BN, TAPS, true> : conv2d_fwd_pair_halo_kernel<BN, TAPS, false>;
}

template <int BN, int TAPS>
cudaError_t pair_halo_configure(bool fused)
{
    static unsigned long long configured[2] = {0ull, 0ull};
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (bit && (__atomic_load_n(&configured[fused], __ATOMIC_ACQUIRE) & bit)) return cudaSuccess;
    err = cudaFuncSetAttribute(pair_halo_kernel<BN, TAPS>(fused), cudaFuncAttributeMaxDynamicSharedMemorySize, kMaxSmemBytes);
    if (err != cudaSuccess) return err;
    if (bit) __atomic_fetch_or(&configured[fused], bit, __ATOMIC_RELEASE);
    return cudaSuccess;
}

template <int BN, int TAPS>
void pair_halo_launch_config(cudaLaunchConfig_t* cfg, cudaLaunchAttribute* attr, int pairs, int smem,
                             cudaStream_t stream)
{
    *cfg = cudaLaunchConfig_t{};
    cfg->gridDim = dim3(static_cast<unsigned>(2 * pairs));
    cfg->blockDim = dim3(HaloPairConfig<BN, TAPS>::THREADS);
    cfg->dynamicSmemBytes = static_cast<size_t>(smem);
    cfg->stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg->attrs = attr;
    cfg->numAttrs = 2;
}
}  // namespace

template <int BN, int TAPS>
cudaError_t launch_conv2d_pair_halo(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const ConvKernelParams& kp,
                                    int pairs, cudaStream_t stream)
{
    const bool fused = (kp.relu | kp.out_bf16) != 0;
    const int smem = conv2d_pair_halo_smem_bytes<BN, TAPS>(kp.halo_bytes);
    if (smem > kMaxSmemBytes) return cudaErrorInvalidValue;
    cudaError_t err = pair_halo_configure<BN, TAPS>(fused);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_halo_launch_config<BN, TAPS>(&cfg, attr, pairs, smem, stream);
    return cudaLaunchKernelEx(&cfg, pair_halo_kernel<BN, TAPS>(fused), tm_a, tm_b, kp);
}

// Resident CTA pairs at this shared-memory size; a few sizes are remembered per device.
template <int BN, int TAPS>
int conv2d_pair_halo_max_resident(bool fused, int smem)
{
    struct Entry { int dev, fused, smem, n; };
    static Entry cache[16] = {};
    static int next = 0;
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        for (const Entry& e : cache)
            if (e.n > 0 && e.dev == dev && e.fused == static_cast<int>(fused) && e.smem == smem) return e.n;
    }
    if (pair_halo_configure<BN, TAPS>(fused) != cudaSuccess) return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    pair_halo_launch_config<BN, TAPS>(&cfg, attr, 1, smem, nullptr);
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, pair_halo_kernel<BN, TAPS>(fused), &cfg) != cudaSuccess) return 0;
    if (n > 0) {
        std::lock_guard<std::mutex> lock(mu);
        cache[next] = Entry{dev, static_cast<int>(fused), smem, n};
        next = (next + 1) % 16;
    }
    return n;
}

template SGB_PAIR_HALO_SIG(64, 2);
template SGB_PAIR_HALO_SIG(64, 3);
template SGB_PAIR_HALO_SIG(128, 2);
template SGB_PAIR_HALO_SIG(128, 3);
template SGB_PAIR_HALO_SIG(256, 2);
template SGB_PAIR_HALO_RES_SIG(64, 2);
template SGB_PAIR_HALO_RES_SIG(64, 3);
template SGB_PAIR_HALO_RES_SIG(128, 2);
template SGB_PAIR_HALO_RES_SIG(128, 3);
template SGB_PAIR_HALO_RES_SIG(256, 2);
#endif

template SGB_PAIR_SIG(64, SGB_PAIR_KBS);
template SGB_PAIR_SIG(128, SGB_PAIR_KBS);
template SGB_PAIR_SIG(256, SGB_PAIR_KBS);
template SGB_PAIR_RES_SIG(64, SGB_PAIR_KBS);
template SGB_PAIR_RES_SIG(128, SGB_PAIR_KBS);
template SGB_PAIR_RES_SIG(256, SGB_PAIR_KBS);

}  // namespace sgb
