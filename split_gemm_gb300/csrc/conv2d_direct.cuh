// Direct grouped convolution on the CUDA cores, for groups of few channels
// (C/groups = K/groups = CG in {1, 2, 4, 8, 16}; depthwise is CG = 1).
//
// With so few channels per group the implicit GEMM wastes the tensor cores: a
// 64-wide column block would hold CG useful columns and each tile's reduction
// is only R*S*CG long.  Here each thread owns one 16-byte chunk of channels
// (CH = 8 channels: 8/CG whole groups; CH = 16 for CG = 16) of PX consecutive
// output pixels of one output row, and accumulates their CH x PX outputs in
// fp32 FMAs.  Per filter tap it loads its chunk at the PX input positions (one
// vector load each) and reads each weight of its groups once from shared
// memory, for PX FMAs.  The block keeps all group weights in shared memory as
// fp32, laid out [tap][c][kk][group-in-chunk][chunk] so that the lanes of a
// warp (consecutive chunks of the same pixels) read consecutive words.
// Consecutive threads take consecutive chunks, so a warp's loads and stores
// cover contiguous NHWC spans.  The bias, the fused ReLU and the bf16 output
// conversion happen in registers before the store.
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
    int nchunk;         // C / CH channel chunks per pixel
    int qblocks;        // ceil(Q / PX) pixel blocks per output row
    int items;          // N * P * qblocks * nchunk (one thread each); < 2^31
};

template <int CG>
struct DirectCfg {
    static constexpr int CH = CG == 16 ? 16 : 8;  // channels per thread (one or two 16-byte loads)
    static constexpr int GB = CH / CG;             // groups per thread
    static constexpr int PX = CG == 16 ? 2 : 4;    // output pixels per thread
};

__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) { return __uint_as_float(b << 16); }

// CH consecutive bf16 channels (16-byte aligned) widened to fp32.
template <int CH>
__device__ __forceinline__ void load_chunk(const uint16_t* p, float (&v)[CH])
{
#pragma unroll
    for (int i = 0; i < CH / 8; ++i) {
        const uint4 q = __ldg(reinterpret_cast<const uint4*>(p) + i);
        const uint32_t u[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            v[8 * i + 2 * j] = bf16_bits_to_float(u[j] & 0xFFFFu);
            v[8 * i + 2 * j + 1] = bf16_bits_to_float(u[j] >> 16);
        }
    }
}

template <int CG>
__global__ void __launch_bounds__(DIRECT_THREADS) conv2d_direct_kernel(const __grid_constant__ DirectParams kp)
{
    using Cfg = DirectCfg<CG>;
    constexpr int CH = Cfg::CH, GB = Cfg::GB, PX = Cfg::PX;
    extern __shared__ float wsm[];  // [tap][c][kk][gi][chunk] fp32
    const int taps = kp.R * kp.S;
    const int nchunk = kp.nchunk;
    // Stage: one (filter k, tap) pair per iteration, its CG weights in one pass.
    for (int e = threadIdx.x; e < kp.K * taps; e += blockDim.x) {
        const int k = e / taps;
        const int tap = e - k * taps;
        const int g = k / CG, kk = k - (k / CG) * CG;
        const int cb = g / GB, gi = g - (g / GB) * GB;
        const uint16_t* src = kp.w + static_cast<long long>(e) * CG;
#pragma unroll
        for (int c = 0; c < CG; ++c)
            wsm[(((tap * CG + c) * CG + kk) * GB + gi) * nchunk + cb] =
                bf16_bits_to_float(__ldg(reinterpret_cast<const unsigned short*>(src) + c));
    }
    __syncthreads();

    for (int item = blockIdx.x * blockDim.x + threadIdx.x; item < kp.items; item += gridDim.x * blockDim.x) {
        const int cb = item % nchunk;
        int rest = item / nchunk;
        const int qb = rest % kp.qblocks;
        rest /= kp.qblocks;
        const int p = rest % kp.P;
        const int n = rest / kp.P;
        const int q0 = qb * PX;
        float acc[PX][CH];
#pragma unroll
        for (int i = 0; i < CH; ++i) {
            const float b = kp.bias ? __ldg(kp.bias + cb * CH + i) : 0.0f;
#pragma unroll
            for (int j = 0; j < PX; ++j) acc[j][i] = b;
        }
        for (int r = 0; r < kp.R; ++r) {
            const int ih = p * kp.sh - kp.ph + r * kp.dh;
            if (ih < 0 || ih >= kp.H) continue;
            const uint16_t* xrow = kp.x + (static_cast<long long>(n) * kp.H + ih) * kp.W * kp.C + cb * CH;
            for (int s = 0; s < kp.S; ++s) {
                float xv[PX][CH];
#pragma unroll
                for (int j = 0; j < PX; ++j) {
                    const int iw = (q0 + j) * kp.sw - kp.pw + s * kp.dw;
                    if (q0 + j < kp.Q && iw >= 0 && iw < kp.W) {
                        load_chunk<CH>(xrow + static_cast<long long>(iw) * kp.C, xv[j]);
                    } else {
#pragma unroll
                        for (int i = 0; i < CH; ++i) xv[j][i] = 0.0f;
                    }
                }
                const float* wt = wsm + (r * kp.S + s) * CG * CG * GB * nchunk + cb;
#pragma unroll
                for (int gi = 0; gi < GB; ++gi)
#pragma unroll
                    for (int c = 0; c < CG; ++c)
#pragma unroll
                        for (int kk = 0; kk < CG; ++kk) {
                            const float wv = wt[((c * CG + kk) * GB + gi) * nchunk];
#pragma unroll
                            for (int j = 0; j < PX; ++j)
                                acc[j][gi * CG + kk] = fmaf(xv[j][gi * CG + c], wv, acc[j][gi * CG + kk]);
                        }
            }
        }
#pragma unroll
        for (int j = 0; j < PX; ++j) {
            if (q0 + j >= kp.Q) break;
            const long long at = ((static_cast<long long>(n) * kp.P + p) * kp.Q + q0 + j) * kp.K + cb * CH;
            if (kp.relu) {
#pragma unroll
                for (int i = 0; i < CH; ++i) acc[j][i] = fmaxf(acc[j][i], 0.0f);
            }
            if (kp.out_bf16) {
#pragma unroll
                for (int i = 0; i < CH / 4; ++i)
                    reinterpret_cast<uint2*>(reinterpret_cast<uint16_t*>(kp.y) + at)[i] = ptx::pack_bf16x4(make_uint4(
                        __float_as_uint(acc[j][4 * i]), __float_as_uint(acc[j][4 * i + 1]),
                        __float_as_uint(acc[j][4 * i + 2]), __float_as_uint(acc[j][4 * i + 3])));
            } else {
#pragma unroll
                for (int i = 0; i < CH / 4; ++i)
                    reinterpret_cast<float4*>(kp.y + at)[i] =
                        make_float4(acc[j][4 * i], acc[j][4 * i + 1], acc[j][4 * i + 2], acc[j][4 * i + 3]);
            }
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

// Block-diagonal weight for grouped convolution on the tensor cores: groups of
// cg channels (cg = 8, 16 or 32) merged 64 / cg at a time into groups of 64.
// w [K][taps][cg] bf16 becomes wb [K][taps][64] bf16, output channel k's row
// holding its cg weights at columns ((k / cg) % (64 / cg)) * cg .. + cg - 1 of
// its 64-channel block and zeros elsewhere.  One thread per 16-byte chunk.
cudaError_t launch_expand_blockdiag(const uint16_t* w, uint16_t* wb, int K, int taps, int cg, cudaStream_t stream);

}  // namespace sgb
