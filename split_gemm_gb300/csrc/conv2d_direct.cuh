// Direct grouped convolution on the CUDA cores, for groups of few channels
// (C/groups = K/groups = CG in {1, 2, 4, 8, 16}; depthwise is CG = 1).
//
// With so few channels per group the implicit GEMM wastes the tensor cores: a
// 64-wide column block would hold CG useful columns and each tile's reduction
// is only R*S*CG long.  Here one thread computes the CG outputs of one (output
// pixel, group) pair in fp32 FMAs: per filter tap it loads its group's CG
// input channels (one 2..32-byte vector load) and multiplies them with the
// group's weights, which the block keeps in shared memory as fp32, laid out
// [tap][c][kk][group] so that the lanes of a warp (consecutive groups of one
// pixel, or consecutive pixels of a group) read consecutive or identical words.
// Consecutive threads take consecutive groups, then pixels, so a warp's input
// loads and output stores cover contiguous NHWC spans.  The bias, the fused
// ReLU and the bf16 output conversion happen in registers before the store.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace sgb {

constexpr int DIRECT_THREADS = 256;

struct DirectParams {
    const uint16_t* x;  // bf16 NHWC
    const uint16_t* w;  // bf16 [K][R][S][CG]
    const float* bias;  // [K] or nullptr
    float* y;           // fp32 NHWC (bf16 with out_bf16)
    int N, H, W, C, K, R, S, P, Q;
    int sh, sw, ph, pw, dh, dw;
    int G;              // groups
    int relu, out_bf16;
    long long total;    // N * P * Q * G (one thread per output pixel and group)
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// The CG channels of one group at one input position, widened to fp32.
template <int CG>
__device__ __forceinline__ void load_group(const uint16_t* p, float (&v)[CG])
{
    if constexpr (CG % 8 == 0) {
#pragma unroll
        for (int i = 0; i < CG / 8; ++i) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + i);
            const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = bf16_bits_to_float(u[j] & 0xFFFFu);
                v[8 * i + 2 * j + 1] = bf16_bits_to_float(u[j] >> 16);
            }
        }
    } else if constexpr (CG == 4) {
        const uint2 q = __ldg(reinterpret_cast<const uint2*>(p));
        v[0] = bf16_bits_to_float(q.x & 0xFFFFu);
        v[1] = bf16_bits_to_float(q.x >> 16);
        v[2] = bf16_bits_to_float(q.y & 0xFFFFu);
        v[3] = bf16_bits_to_float(q.y >> 16);
    } else if constexpr (CG == 2) {
        const uint32_t q = __ldg(reinterpret_cast<const unsigned int*>(p));
        v[0] = bf16_bits_to_float(q & 0xFFFFu);
        v[1] = bf16_bits_to_float(q >> 16);
    } else {
        v[0] = bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(p)));
    }
}

template <int CG>
__global__ void __launch_bounds__(DIRECT_THREADS) conv2d_direct_kernel(const __grid_constant__ DirectParams kp)
{
    extern __shared__ float wsm[];  // [R*S][CG][CG][G] fp32
    const int taps = kp.R * kp.S;
    const int G = kp.G;
    const int wcount = kp.K * taps * CG;
    for (int i = threadIdx.x; i < wcount; i += blockDim.x) {
        // w[k][tap][c] with k = g*CG + kk
        const int c = i % CG;
        const int t = i / CG;
        const int tap = t % taps;
        const int k = t / taps;
        const int g = k / CG;
        const int kk = k - g * CG;
        wsm[((tap * CG + c) * CG + kk) * G + g] = bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(kp.w) + i));
    }
    __syncthreads();

    for (long long idx = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; idx < kp.total;
         idx += static_cast<long long>(gridDim.x) * blockDim.x) {
        const int g = static_cast<int>(idx % G);
        const long long pix = idx / G;
        const int q = static_cast<int>(pix % kp.Q);
        const long long np = pix / kp.Q;
        const int p = static_cast<int>(np % kp.P);
        const int n = static_cast<int>(np / kp.P);
        float acc[CG];
#pragma unroll
        for (int kk = 0; kk < CG; ++kk) acc[kk] = kp.bias ? __ldg(kp.bias + g * CG + kk) : 0.0f;
        for (int r = 0; r < kp.R; ++r) {
            const int ih = p * kp.sh - kp.ph + r * kp.dh;
            if (ih < 0 || ih >= kp.H) continue;
            for (int s = 0; s < kp.S; ++s) {
                const int iw = q * kp.sw - kp.pw + s * kp.dw;
                if (iw < 0 || iw >= kp.W) continue;
                float xv[CG];
                load_group<CG>(kp.x + ((static_cast<long long>(n) * kp.H + ih) * kp.W + iw) * kp.C + g * CG, xv);
                const float* wp = wsm + ((r * kp.S + s) * CG * CG) * G + g;
#pragma unroll
                for (int c = 0; c < CG; ++c)
#pragma unroll
                    for (int kk = 0; kk < CG; ++kk) acc[kk] = fmaf(xv[c], wp[(c * CG + kk) * G], acc[kk]);
            }
        }
        if (kp.relu) {
#pragma unroll
            for (int kk = 0; kk < CG; ++kk) acc[kk] = fmaxf(acc[kk], 0.0f);
        }
        const long long at = pix * kp.K + g * CG;
        if (kp.out_bf16) {
            uint16_t* yb = reinterpret_cast<uint16_t*>(kp.y) + at;
#pragma unroll
            for (int kk = 0; kk < CG; ++kk) yb[kk] = ptx::bf16_bits(acc[kk]);
        } else if constexpr (CG % 4 == 0) {
#pragma unroll
            for (int i = 0; i < CG / 4; ++i)
                reinterpret_cast<float4*>(kp.y + at)[i] = make_float4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
        } else {
#pragma unroll
            for (int kk = 0; kk < CG; ++kk) kp.y[at + kk] = acc[kk];
        }
    }
}

// Shared memory the kernel needs: the group weights as fp32.
inline long long conv2d_direct_smem_bytes(int K, int R, int S, int CG)
{
    return static_cast<long long>(K) * R * S * CG * 4;
}

template <int CG>
cudaError_t launch_conv2d_direct(const DirectParams& kp, int grid, cudaStream_t stream);

#define SGB_DIRECT_SIG(CG_) cudaError_t launch_conv2d_direct<CG_>(const DirectParams&, int, cudaStream_t)

}  // namespace sgb
