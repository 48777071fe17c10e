// Epilogue building blocks shared by the convolution kernels: the 128-byte
// swizzled staging layout of a warp's 32 x 32 fp32 slab, and the slab writer
// that turns a warp's accumulator rows into coalesced 16-byte row-segment writes.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace sgb {

// Byte offset of 16-byte chunk `chunk16` of row `row` in a slab of 128-byte rows
// stored with the 128-byte swizzle (chunk index XOR row % 8): the eight chunks of
// any row, and chunk c of any eight consecutive rows, fall in distinct banks.
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk16)
{
    return static_cast<uint32_t>(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// How an epilogue writes a 32 x 32 slab of the accumulator: plain fp32 stores,
// fp32 vector atomic adds (a later split of a cut tile, or a partial-sum
// buffer), or bf16 stores (fused output conversion).
enum SlabMode : int { SLAB_F32 = 0, SLAB_RED = 1, SLAB_BF16 = 2 };

// One warp's 32 x 32 fp32 slab (lane l holds row l, columns 0..31 in v) goes out
// through the warp's swizzled 4 KB staging slot as 16-byte row-segment writes: 8
// lanes cover one 128-byte row segment, four rows per instruction.  Lane (rsub,
// chunk) = (lane / 8, lane % 8) writes rows 4*i + rsub, i < 8, at column chunk
// `chunk`; rowp[i] + slab_off is that row's byte address for this slab (offset
// to the lane's chunk), bit i of row_ok says whether the row exists, col_ok
// whether the chunk's columns do.  All eight slot reads are issued before the first
// global write so that their latencies overlap, and missing rows and columns
// are predicated off rather than branched around: the epilogue warps are few
// and their instruction stream is the critical path once the last accumulator
// is ready.
template <int MODE>
__device__ __forceinline__ void slab_out(uint32_t saddr, const uint32_t (&v)[32], const uint64_t (&rowp)[8],
                                         int64_t slab_off, uint32_t row_ok, bool col_ok, bool add_bias, float4 bias,
                                         bool relu)
{
    const int lane = threadIdx.x & 31;
    const int rsub = lane >> 3;
    const int chunk = lane & 7;
    __syncwarp();  // the previous slab's reads of the slot are done
#pragma unroll
    for (int c = 0; c < 8; ++c)
        ptx::st_shared_v4(saddr + sw128_offset(lane, c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    __syncwarp();
    uint4 val[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) val[i] = ptx::ld_shared_v4(saddr + sw128_offset(4 * i + rsub, chunk));
    if (add_bias) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            val[i].x = __float_as_uint(__uint_as_float(val[i].x) + bias.x);
            val[i].y = __float_as_uint(__uint_as_float(val[i].y) + bias.y);
            val[i].z = __float_as_uint(__uint_as_float(val[i].z) + bias.z);
            val[i].w = __float_as_uint(__uint_as_float(val[i].w) + bias.w);
        }
    }
    if (relu) {
#pragma unroll
        for (int i = 0; i < 8; ++i) val[i] = ptx::relu4(val[i]);
    }
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const bool p = col_ok && ((row_ok >> i) & 1u);
        const uint64_t at = rowp[i] + static_cast<uint64_t>(slab_off);
        if constexpr (MODE == SLAB_F32) ptx::st_global_v4_if(at, val[i], p);
        else if constexpr (MODE == SLAB_RED) ptx::red_add_v4_f32_if(at, val[i], p);
        else ptx::st_global_v2_if(at, ptx::pack_bf16x4(val[i]), p);
    }
}

}  // namespace sgb
