// Implicit-GEMM convolution for few input channels: the "row window" loader.
//
// Same GEMM as conv2d_kernel.cuh (burn PR #2545 "[Optimization] Implicit gemm
// rewrite", Changes): rows = output pixels, columns = output channels,
// reduction over the filter taps.  What changes is how the im2col operand
// reaches the tensor cores when C is small (C*2 bytes per pixel is no multiple
// of 16, so neither the im2col TMA mode nor 16-byte gathers apply; the stem
// layer of an image network, C = 3, is the usual case).
//
// A operand without im2col.  Channels are padded to Cp = 8 / stride_w (C <= Cp),
// so one staged pixel takes Cp bf16 values and the windows of two neighbouring
// output pixels of one output row start exactly stride_w * Cp * 2 = 16 bytes
// apart.  For one input row, the im2col rows of up to 128 consecutive output
// pixels are overlapping 16-byte-pitch views of ONE staged row segment: value
// kk = s*Cp + c of pixel i's window sits at byte 16*i + 2*kk.  That is the
// unswizzled K-major shared-memory layout with an 8-row group pitch of 128 B
// and a K core-matrix pitch of 16 B, so each tcgen05.mma reads its A operand
// straight from the staged row.  The S*Cp window values of one input row are
// covered by nch = ceil(S*Cp/16) MMAs of K = 16.
//
// N operand: several output rows at once.  A tcgen05.mma of 128 x N x 16 costs
// about the same time for N = 64 as for N = 256 on this part, so a tile holds
// T = 256 / BN output rows (p0 .. p0+T-1) of up to 128 pixels each and the
// accumulator is 128 x (T*BN): column block b is output row p0 + b.  Input row
// p0*sh - ph + i (window row i) meets output row p0 + b through filter row
// r = i - b*sh, so ONE MMA per (window row, K chunk) serves all T output rows if
// its B operand stacks the weights of filter rows i, i - sh, ..., i - (T-1)*sh.
// The resident weight keeps, per residue class rho = r mod sh, the filter rows
// of that class in descending order between T-1 zero blocks on each side; the
// stack for window row i is then T consecutive blocks of that sequence, one
// descriptor.  (T = 1 when dilation_h > 1: one block per filter row.)
//
// Work: a tile is (image, 128-column block, T output rows), all K <= BN output
// channels.  CTA b takes the contiguous tile range [b*Tt/G, (b+1)*Tt/G), output
// rows running fastest, so consecutive tiles share rt - T*sh staged window rows
// (rt = (T-1)*sh + (R-1)*dh + 1) and stage only T*sh new ones.  Staged rows live
// in a ring of row slots with full / empty mbarriers; the MMA thread releases a
// slot (tcgen05.commit) once no later tile of the CTA reads it.
//
// Warp roles (416 threads):
//   warps 0..7  stager: per tile, 16-byte cp.async copies of the raw bytes of its
//               new input rows (one tile ahead), then a repack into padded-
//               channel segments (zeros outside the image and at padded channels);
//   warp 8      TMEM allocator and single-thread MMA issuer;
//   warps 9..12 epilogue: TMEM -> registers (+ bias) -> swizzled shared staging
//               -> coalesced 16-byte global stores.
// Every wait is bounded as in conv2d_kernel.cuh.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "slab_store.cuh"
#include "trace.cuh"

namespace sgb {

constexpr int RW_LOAD_THREADS = 256;  // warps 0..7
constexpr int RW_MMA_WARP = 8;
constexpr int RW_EPI_WARP0 = 9;       // warps 9..12
constexpr int RW_EPI_THREADS = 128;
constexpr int RW_THREADS = 13 * 32;
constexpr int RW_TILE_M = 128;        // output pixels per output row of a tile (one MMA row block)
constexpr int RW_MAX_CLASSES = 8;     // residue classes of filter rows (stride_h <= 8 when T > 1)
constexpr int RW_REG_ROWS = 16;       // window rows whose weight descriptors the MMA thread keeps in registers
constexpr int RW_REG_CHUNKS = 4;      // K chunks per window row issued from registers
constexpr int RW_EPI_SLOT_BYTES = 32 * 32 * 4;
constexpr uint32_t RW_STATUS_TIMEOUT = 6;  // same value as CONV2D_ERR_TIMEOUT

struct RowWinParams {
    const uint16_t* x;  // bf16 NHWC
    const uint16_t* w;  // bf16 KRSC
    const float* bias;  // [K] or nullptr
    float* y;           // fp32 NHWC
    uint32_t* status;   // device status word or nullptr
    int N, H, W, C, K, R, S, P, Q;
    int sh, sw, ph, pw, dh;
    int cp_log2;       // log2 of the padded channel count Cp = 8 / stride_w
    int nch;           // 16-value reduction chunks per window row: ceil(S*Cp/16)
    int seg_elems;     // bf16 values per staged row segment: 8*127 + 16*nch
    int raw_bytes;     // bytes of one raw-copy buffer (one input row)
    int T;             // output rows per tile
    int rt;            // window rows per tile: (T-1)*sh + (R-1)*dh + 1
    int new_rows;      // rows a continuing tile stages: T*sh when reuse, else rt
    int reuse;         // consecutive tiles share window rows
    int ncls;          // residue classes of the resident weight (sh when T > 1, else 1)
    int cls_k[RW_MAX_CLASSES];     // filter rows in each class
    int cls_base[RW_MAX_CLASSES];  // first block of each class's sequence
    int nblocks;       // weight blocks per K chunk
    int row_slots;     // staged-row ring size (>= rt)
    int wtmp_filters;  // filters per weight-staging pass
    int qblocks;       // ceil(Q / 128)
    int pblocks;       // ceil(P / T)
    int tiles;         // N * qblocks * pblocks
    int grid;
    int vec_store;     // K % 4 == 0: 16-byte vector writes of y
    int relu;          // fused epilogue: ReLU after the bias
    int out_bf16;      // fused epilogue: y stored as bf16 (round to nearest even)
    uint32_t tmem_cols;  // power of two >= 2 * T * BN
    long long x_bytes;   // copies never read at or past these sizes
    long long w_bytes;
    int off_rows, off_raw, off_wtmp, off_epi, off_bar, off_tab;  // shared-memory layout (bytes from the 1024-B aligned base)
    unsigned long long wait_limit_ns;
    unsigned long long* trace;  // per-CTA phase timestamps; only written in trace builds
};

// Shared-memory layout, shared by the host (launch size) and the kernel:
// resident weight | row-slot ring | 2 x rt raw-copy buffers | weight copy area
// (wtmp_bytes, may be 0: the epilogue staging area serves instead) | epilogue
// staging | barriers | per-window-row block table.
struct RowWinLayout {
    int b_bytes, off_rows, off_raw, off_wtmp, off_epi, off_bar, off_tab, total;
};

__host__ __device__ inline int rw_align(int v, int a) { return (v + a - 1) / a * a; }

__host__ __device__ inline RowWinLayout rowwin_layout(int bn, int nch, int nblocks, int seg_elems, int row_slots,
                                                      int rt, int raw_bytes, int wtmp_bytes)
{
    RowWinLayout l;
    l.b_bytes = nch * nblocks * bn * 32;
    l.off_rows = rw_align(l.b_bytes, 128);
    l.off_raw = l.off_rows + row_slots * seg_elems * 2;
    l.off_wtmp = rw_align(l.off_raw + 2 * rt * raw_bytes, 128);
    l.off_epi = rw_align(l.off_wtmp + wtmp_bytes, 128);
    l.off_bar = l.off_epi + 4 * RW_EPI_SLOT_BYTES;
    l.off_tab = rw_align(l.off_bar + (2 * row_slots + 6) * 8 + 16, 16);
    l.total = l.off_tab + 4 * rt + 1024;  // + alignment slack of the base
    return l;
}

struct RwSmem {
    uint8_t* b;          // resident weight: nch x nblocks blocks of BN x 16 values
    uint8_t* rows;       // row_slots staged segments
    uint8_t* raw;        // 2 x rt raw-copy buffers (double-buffered by tile)
    uint8_t* epi;        // 4 epilogue staging slots
    int* tab;            // rt entries: first weight block of window row i, or -1
    uint64_t* full;      // row_slots: segment staged
    uint64_t* empty;     // row_slots: segment no longer read by any MMA
    uint64_t* acc_full;  // 2
    uint64_t* acc_empty; // 2
    uint64_t* mma_done;
    uint64_t* w_ready;   // resident weight staged (one arrive per epilogue warp)
    uint32_t* tmem_slot;
    volatile uint32_t* abort_flag;
    volatile uint32_t* epi_go;
    volatile uint32_t* ld_abort;  // stager's own verdict, read only between its barriers
};

__device__ __forceinline__ void rw_record_timeout(const RowWinParams& kp, volatile uint32_t* abort_flag)
{
    *abort_flag = 1u;
    if (kp.status) atomicMax(kp.status, RW_STATUS_TIMEOUT);
}

// Tile t -> (image, 128-column block, first output row); output rows run fastest.
struct RwTile {
    int n, qb, p0;
};
__device__ __forceinline__ RwTile rw_tile(const RowWinParams& kp, int t)
{
    const int per_img = kp.qblocks * kp.pblocks;
    RwTile o;
    o.n = t / per_img;
    const int rem = t - o.n * per_img;
    o.qb = rem / kp.pblocks;
    o.p0 = (rem - o.qb * kp.pblocks) * kp.T;
    return o;
}

// Window rows tile t stages itself: new_rows when it continues the previous
// tile of the CTA (same image and column block, next T output rows), else rt.
__device__ __forceinline__ int rw_tile_rows(const RowWinParams& kp, int t, int t_lo, const RwTile& tl)
{
    return (kp.reuse && t > t_lo && tl.p0 > 0) ? kp.new_rows : kp.rt;
}

// Byte range of x that one staged row needs: input columns [w_a, w_b) of row h.
struct RwRowSpan {
    bool ok;         // any in-image pixel at all
    int wl;          // input column of staged pixel 0 (may be negative)
    int w_a, w_b;
    long long b0;    // first needed byte
    long long a0;    // b0 rounded down to 16 (start of the raw copy)
    long long a1;    // end of the raw copy (rounded up to 16, clipped to x)
};
__device__ __forceinline__ RwRowSpan rw_row_span(const RowWinParams& kp, int n, int qb, int h)
{
    RwRowSpan sp;
    sp.wl = qb * RW_TILE_M * kp.sw - kp.pw;
    const int segpix = kp.seg_elems >> kp.cp_log2;
    sp.w_a = sp.wl > 0 ? sp.wl : 0;
    sp.w_b = sp.wl + segpix < kp.W ? sp.wl + segpix : kp.W;
    sp.ok = static_cast<unsigned>(h) < static_cast<unsigned>(kp.H) && sp.w_a < sp.w_b;
    sp.b0 = sp.a0 = sp.a1 = 0;
    if (sp.ok) {
        const long long rowpix = static_cast<long long>(n * kp.H + h) * kp.W;
        sp.b0 = (rowpix + sp.w_a) * kp.C * 2;
        const long long b1 = (rowpix + sp.w_b) * kp.C * 2;
        sp.a0 = sp.b0 & ~15ll;
        sp.a1 = (b1 + 15) & ~15ll;
        if (sp.a1 > kp.x_bytes) sp.a1 = kp.x_bytes;
    }
    return sp;
}

// 16-byte cp.async copies of [a0, a1) into a buffer; the last copy of a tensor
// may be short (the rest of its 16 bytes is zero-filled, nothing past it is read).
// Thread lt of nthreads takes chunks lt, lt + nthreads, ...
__device__ __forceinline__ void rw_copy_span(const uint8_t* base, long long a0, long long a1, uint8_t* dst, int lt,
                                             int nthreads)
{
    const int chunks = static_cast<int>((a1 - a0 + 15) >> 4);
    for (int ch = lt; ch < chunks; ch += nthreads) {
        const long long left = a1 - a0 - 16ll * ch;
        ptx::cp_async_16(dst + 16 * ch, base + a0 + 16ll * ch, left >= 16 ? 16u : static_cast<uint32_t>(left));
    }
}

// Input row of window row i of a tile whose first output row is p0.
__device__ __forceinline__ int rw_window_h(const RowWinParams& kp, int p0, int i) { return p0 * kp.sh - kp.ph + i; }

// Issues the raw copies of tile t's new rows into raw buffer set `set`.
__device__ __forceinline__ void rw_issue_tile(const RowWinParams& kp, const RwSmem& sm, int t, int t_lo, int set,
                                              int lt)
{
    const RwTile tl = rw_tile(kp, t);
    const int nr = rw_tile_rows(kp, t, t_lo, tl);
    const uint8_t* xb = reinterpret_cast<const uint8_t*>(kp.x);
    for (int k = 0; k < nr; ++k) {
        const RwRowSpan sp = rw_row_span(kp, tl.n, tl.qb, rw_window_h(kp, tl.p0, kp.rt - nr + k));
        if (sp.ok) rw_copy_span(xb, sp.a0, sp.a1, sm.raw + (set * kp.rt + k) * kp.raw_bytes, lt, RW_LOAD_THREADS);
    }
}

// Repack of tile t's new rows (raw set `set`) into row slots first_row, first_row+1, ...:
// value kk of staged pixel j of a row is channel kk % Cp of input column wl + j,
// zero outside the image or past C.  Stager warp wi repacks rows wi, wi+8, ...,
// its lanes taking consecutive 16-byte chunks.  A chunk holds 8/Cp = stride_w
// whole pixels; inside the image its 8 values sit at fixed byte offsets from
// the chunk's first pixel, so only the chunks at the row edges take the
// per-value path.
__device__ __forceinline__ void rw_repack_tile(const RowWinParams& kp, const RwSmem& sm, const RwTile& tl, int nr,
                                               int set, int first_row, int lt)
{
    const int lane = lt & 31;
    const int cpr = kp.seg_elems >> 3;  // chunks per row
    const int cpm = (1 << kp.cp_log2) - 1;
    const int ppc = 8 >> kp.cp_log2;    // pixels per chunk
    const uint32_t seg_bytes = static_cast<uint32_t>(kp.seg_elems * 2);
    int off[8];  // byte offset of value e from the chunk's first pixel, or -1 for a padded channel
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int c = e & cpm;
        off[e] = c < kp.C ? ((e >> kp.cp_log2) * kp.C + c) * 2 : -1;
    }
    for (int k = lt >> 5; k < nr; k += RW_LOAD_THREADS / 32) {
        const RwRowSpan sp = rw_row_span(kp, tl.n, tl.qb, rw_window_h(kp, tl.p0, kp.rt - nr + k));
        const uint32_t src =
            ptx::smem_addr(sm.raw + (set * kp.rt + k) * kp.raw_bytes) + static_cast<uint32_t>(sp.b0 - sp.a0);
        const uint32_t dst =
            ptx::smem_addr(sm.rows) + static_cast<uint32_t>((first_row + k) % kp.row_slots) * seg_bytes;
        for (int u = lane; u < cpr; u += 32) {
            const int w0 = sp.wl + u * ppc;  // input column of the chunk's first pixel
            uint32_t v[8];
            if (sp.ok && w0 >= sp.w_a && w0 + ppc <= sp.w_b) {
                const uint32_t base = src + static_cast<uint32_t>((w0 - sp.w_a) * kp.C * 2);
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = off[e] >= 0 ? ptx::ld_shared_u16(base + off[e]) : 0u;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int w = w0 + (e >> kp.cp_log2);
                    uint32_t val = 0;
                    if (sp.ok && off[e] >= 0 && w >= sp.w_a && w < sp.w_b)
                        val = ptx::ld_shared_u16(src + static_cast<uint32_t>(((w - sp.w_a) * kp.C + (e & cpm)) * 2));
                    v[e] = val;
                }
            }
            ptx::st_shared_v4(dst + 16 * u, v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16),
                              v[6] | (v[7] << 16));
        }
    }
}

// Resident weight.  Block `blk` of K chunk j holds, for output channel n < BN and
// value e of 16, the tap (s, c) = ((16j + e) / Cp, (16j + e) % Cp) of the block's
// filter row (zero where s >= S, c >= C, n >= K, or for a zero block), in the
// unswizzled K-major layout: 8-row groups 256 B apart, the two 8-value halves
// 128 B apart.  Run by the 128 epilogue threads before their first tile (the
// stager meanwhile fetches the first rows): the whole area is zeroed, then
// thread pair (n, half) fills the blocks that hold a filter row.  The weight is
// copied in through the epilogue staging area in passes of wtmp_filters filters.
template <int BN>
__device__ void rw_stage_weights(const RowWinParams& kp, const RwSmem& sm, int lt)
{
    const int crs = kp.C * kp.R * kp.S;
    const int cpm = (1 << kp.cp_log2) - 1;
    const uint32_t b_base = ptx::smem_addr(sm.b);
    const int kmax = kp.K < BN ? kp.K : BN;
    const uint8_t* wb = reinterpret_cast<const uint8_t*>(kp.w);
    const int units = kp.nch * kp.nblocks * BN * 2;  // 16-byte units of the resident weight
    uint8_t* tmp = kp.off_wtmp != kp.off_epi ? reinterpret_cast<uint8_t*>(sm.b) + kp.off_wtmp : sm.epi;
    for (int f0 = 0; f0 < kmax; f0 += kp.wtmp_filters) {
        const int f1 = f0 + kp.wtmp_filters < kmax ? f0 + kp.wtmp_filters : kmax;
        const long long b0 = static_cast<long long>(f0) * crs * 2;
        long long a1 = (static_cast<long long>(f1) * crs * 2 + 15) & ~15ll;
        if (a1 > kp.w_bytes) a1 = kp.w_bytes;
        const long long a0 = b0 & ~15ll;
        rw_copy_span(wb, a0, a1, tmp, lt, RW_EPI_THREADS);
        ptx::cp_async_commit();
        if (f0 == 0)  // zero blocks, padded taps and filters K..BN-1 (overlaps the first copy)
            for (int u = lt; u < units; u += RW_EPI_THREADS) ptx::st_shared_v4(b_base + 16u * u, 0u, 0u, 0u, 0u);
        ptx::cp_async_wait<0>();
        ptx::named_bar_sync(3, RW_EPI_THREADS);  // copies landed, zeroing done
        const uint32_t src = ptx::smem_addr(tmp) + static_cast<uint32_t>(b0 - a0);
        for (int pr = lt; pr < 2 * (f1 - f0); pr += RW_EPI_THREADS) {
            const int n = f0 + (pr >> 1);
            const int half = pr & 1;
            const uint32_t fsrc = src + static_cast<uint32_t>((n - f0) * crs * 2);
            const uint32_t unit = static_cast<uint32_t>((n >> 3) * 256 + half * 128 + (n & 7) * 16);
            for (int j = 0; j < kp.nch; ++j) {
                int off[8];  // byte offset of tap e inside a filter row, or -1
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int kk = j * 16 + half * 8 + e;
                    const int s = kk >> kp.cp_log2;
                    const int c = kk & cpm;
                    off[e] = (s < kp.S && c < kp.C) ? (s * kp.C + c) * 2 : -1;
                }
                for (int rho = 0; rho < kp.ncls; ++rho) {
                    const int kc = kp.cls_k[rho];
                    for (int k = 0; k < kc; ++k) {
                        const int r = kp.T > 1 ? rho + k * kp.sh : k;
                        const int blk = kp.cls_base[rho] + (kp.T - 1) + (kc - 1 - k);
                        const uint32_t rsrc = fsrc + static_cast<uint32_t>(r * kp.S * kp.C * 2);
                        uint32_t v[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) v[e] = off[e] >= 0 ? ptx::ld_shared_u16(rsrc + off[e]) : 0u;
                        ptx::st_shared_v4(b_base + static_cast<uint32_t>((j * kp.nblocks + blk) * BN * 32) + unit,
                                          v[0] | (v[1] << 16), v[2] | (v[3] << 16), v[4] | (v[5] << 16),
                                          v[6] | (v[7] << 16));
                    }
                }
            }
        }
        ptx::named_bar_sync(3, RW_EPI_THREADS);  // the copy area is reused by the next pass (and by the epilogue)
    }
}

// ---------------------------------------------------------------- stager (warps 0..7)
template <int BN>
__device__ void rw_stager(const RowWinParams& kp, const RwSmem& sm, int t_lo, int t_hi)
{
    const int lt = threadIdx.x;  // 0..255
    const int lane = lt & 31;
    uint64_t c_bar = 0, c_copy = 0, c_empty = 0, c_pack = 0;
    (void)c_bar; (void)c_copy; (void)c_empty; (void)c_pack;
    if (t_lo < t_hi) rw_issue_tile(kp, sm, t_lo, t_lo, 0, lt);
    ptx::cp_async_commit();
    int g = 0;  // stream index of the tile's first new row
    for (int t = t_lo, ti = 0; t < t_hi; ++t, ++ti) {
        if (lane == 0 && *sm.abort_flag) *sm.ld_abort = 1u;
        // (A) the previous tile's repack is done everywhere (its raw set is
        // reused below), and the abort verdict written before this point is final.
        SGB_CYCLES_BEGIN(t_bar);
        ptx::named_bar_sync(2, RW_LOAD_THREADS);
        SGB_CYCLES_END(c_bar, t_bar);
        if (*sm.ld_abort) break;
        if (t + 1 < t_hi) rw_issue_tile(kp, sm, t + 1, t_lo, (ti + 1) & 1, lt);
        ptx::cp_async_commit();
        SGB_CYCLES_BEGIN(t_copy);
        ptx::cp_async_wait<1>();  // this thread's copies of tile t have landed
        // (B) every thread's copies of tile t have landed.
        ptx::named_bar_sync(2, RW_LOAD_THREADS);
        SGB_CYCLES_END(c_copy, t_copy);
        SGB_TRACE(kp, lt == 0 && ti == 0, 21);
        const RwTile tl = rw_tile(kp, t);
        const int nr = rw_tile_rows(kp, t, t_lo, tl);
        SGB_CYCLES_BEGIN(t_empty);
        // Slots are released in row order by one thread, so the last new row's
        // slot being free implies the others are.
        int go = 1;
        if (lane == 0) {
            const int gg = g + nr - 1;
            if (!ptx::mbar_wait(&sm.empty[gg % kp.row_slots], (static_cast<uint32_t>(gg / kp.row_slots) & 1u) ^ 1u,
                                kp.wait_limit_ns)) {
                rw_record_timeout(kp, sm.abort_flag);
                *sm.ld_abort = 1u;
                go = 0;
            }
        }
        go = __shfl_sync(0xffffffffu, go, 0);
        SGB_CYCLES_END(c_empty, t_empty);
        SGB_CYCLES_BEGIN(t_pack);
        if (go) {
            rw_repack_tile(kp, sm, tl, nr, ti & 1, g, lt);
            ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
        }
        __syncwarp();
        if (lane == 0 && go)
            for (int k = 0; k < nr; ++k) ptx::mbar_arrive(&sm.full[(g + k) % kp.row_slots]);
        SGB_CYCLES_END(c_pack, t_pack);
        SGB_TRACE(kp, lt == 0 && ti == 0, 22);
        g += nr;
    }
    SGB_TRACE(kp, lt == 0, 3);
    SGB_TRACE_VALUE(kp, lt == 0, 16, c_bar);
    SGB_TRACE_VALUE(kp, lt == 0, 17, c_copy);
    SGB_TRACE_VALUE(kp, lt == 0, 18, c_empty);
    SGB_TRACE_VALUE(kp, lt == 0, 19, c_pack);
    SGB_TRACE_VALUE(kp, lt == 0, 20, static_cast<unsigned long long>(g));
    ptx::cp_async_wait_all();  // no copy may be in flight when the CTA exits
}

// Weight block (first of T consecutive ones) for window row i, or -1 when no
// filter row meets it.
__device__ __forceinline__ int rw_row_block(const RowWinParams& kp, int i)
{
    if (kp.T > 1) {
        const int rho = i % kp.sh;
        const int kc = kp.cls_k[rho];
        if (kc == 0) return -1;
        return kp.cls_base[rho] + (kp.T - 1) + (kc - 1 - i / kp.sh);
    }
    if (i % kp.dh) return -1;
    return kp.R - 1 - i / kp.dh;
}

// ---------------------------------------------------------------- MMA issuer (warp 8, one thread)
template <int BN>
__device__ void rw_mma(const RowWinParams& kp, const RwSmem& sm, uint32_t tmem_base, int t_lo, int t_hi)
{
    const uint32_t idesc = ptx::idesc_bf16_f32(RW_TILE_M, kp.T * BN);
    const uint32_t b_addr = ptx::smem_addr(sm.b);
    const uint32_t rows_addr = ptx::smem_addr(sm.rows);
    const uint32_t seg_bytes = static_cast<uint32_t>(kp.seg_elems * 2);
    const uint32_t acc_cols = static_cast<uint32_t>(kp.T * BN);
    const uint32_t chunk_bytes = static_cast<uint32_t>(kp.nblocks * BN * 32);  // one K chunk of the weight
    // Descriptor fields other than the start address.  A: pixel q, value kk at
    // byte 16*q + 2*kk -> K core matrices 16 B apart, 8-row groups 128 B apart.
    // B: T consecutive blocks of BN rows -> K halves 128 B apart, 8-row groups 256 B.
    // Descriptors are assembled from a constant high word and a low word holding
    // the start address >> 4 (addresses stay below 256 KB, so no carry into the
    // leading-offset field).
    const uint64_t a_desc0 = ptx::plain_kmajor_desc(0u, 16u, 128u);
    const uint64_t b_desc0 = ptx::plain_kmajor_desc(0u, 128u, 256u);
    const uint64_t a_hi = a_desc0 >> 32, b_hi = b_desc0 >> 32;
    const uint32_t a_lo0 = static_cast<uint32_t>(a_desc0) + (rows_addr >> 4);
    const uint32_t b_lo0 = static_cast<uint32_t>(b_desc0) + (b_addr >> 4);
    const uint32_t seg16 = seg_bytes >> 4;
    const uint32_t chunk16 = chunk_bytes >> 4;
    for (int i = 0; i < kp.rt; ++i) sm.tab[i] = rw_row_block(kp, i);
    // Kernel parameters used between MMAs live in registers: the MMA asm's
    // memory clobber would otherwise reload them after every instruction.
    const int rt = kp.rt, nch = kp.nch, row_slots = kp.row_slots;
    const bool fast_issue = rt <= RW_REG_ROWS && nch <= RW_REG_CHUNKS;
    // Low descriptor word of the first weight block of window rows 0..15 (all 1s: no filter row).
    uint32_t b_lo[RW_REG_ROWS];
#pragma unroll
    for (int i = 0; i < RW_REG_ROWS; ++i) {
        const int blk = i < kp.rt ? rw_row_block(kp, i) : -1;
        b_lo[i] = blk >= 0 ? b_lo0 + static_cast<uint32_t>(blk) * (BN * 2) : 0xFFFFFFFFu;
    }
    int g_end = 0;     // rows staged for the tiles issued so far
    int s_end = 0;     // g_end % row_slots
    int ti = 0;
    bool ok = true;
    uint64_t c_full = 0, c_acc = 0, c_issue = 0, c_rel = 0;
    (void)c_full; (void)c_acc; (void)c_issue; (void)c_rel;
    if (!ptx::mbar_wait(sm.w_ready, 0u, kp.wait_limit_ns)) {
        rw_record_timeout(kp, sm.abort_flag);
        ok = false;
    }
    for (int t = t_lo; t < t_hi && ok; ++t, ++ti) {
        const RwTile tl = rw_tile(kp, t);
        const int nr = rw_tile_rows(kp, t, t_lo, tl);
        // The stager arrives on its rows' barriers in order, so the last one
        // completing implies the others have.
        SGB_CYCLES_BEGIN(t_full);
        {
            const int g_last = g_end + nr - 1;
            if (*sm.abort_flag || !ptx::mbar_wait(&sm.full[g_last % kp.row_slots],
                                                  static_cast<uint32_t>(g_last / kp.row_slots) & 1u, kp.wait_limit_ns)) {
                if (!*sm.abort_flag) rw_record_timeout(kp, sm.abort_flag);
                break;
            }
        }
        SGB_CYCLES_END(c_full, t_full);
        g_end += nr;
        s_end += nr;
        if (s_end >= kp.row_slots) s_end -= kp.row_slots;
        const int buf = ti & 1;
        const uint32_t use = static_cast<uint32_t>(ti >> 1) & 1u;
        SGB_CYCLES_BEGIN(t_acc);
        if (!ptx::mbar_wait(&sm.acc_empty[buf], use ^ 1u, kp.wait_limit_ns)) {
            rw_record_timeout(kp, sm.abort_flag);
            break;
        }
        SGB_CYCLES_END(c_acc, t_acc);
        ptx::tc_fence_after();
        ptx::fence_proxy_async_smem();
        const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(buf) * acc_cols;
        SGB_CYCLES_BEGIN(t_issue);
        SGB_TRACE(kp, ti == 0, 23);
        SGB_TRACE(kp, ti == 1, 25);
        // Window row i of this tile is stream row g_end - rt + i.  The MMA issue
        // stalls until the tensor pipe takes the instruction, so the work between
        // two MMAs is kept to a few integer adds.
        int slot = s_end - kp.rt;
        if (slot < 0) slot += kp.row_slots;
        uint32_t accumulate = 0u;
        if (fast_issue) {
            // All descriptors of a window row are formed first, then its MMAs go
            // out back to back (only a uniform branch between them).
#pragma unroll
            for (int i = 0; i < RW_REG_ROWS; ++i) {
                if (i < rt) {
                    if (b_lo[i] != 0xFFFFFFFFu) {
                        const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(slot) * seg16;
                        uint64_t ad[RW_REG_CHUNKS], bd[RW_REG_CHUNKS];
#pragma unroll
                        for (int j = 0; j < RW_REG_CHUNKS; ++j) {
                            ad[j] = (a_hi << 32) | (a_lo + 2u * j);
                            bd[j] = (b_hi << 32) | (b_lo[i] + j * chunk16);
                        }
                        ptx::mma_bf16(tmem_d, ad[0], bd[0], idesc, accumulate);
#pragma unroll
                        for (int j = 1; j < RW_REG_CHUNKS; ++j)
                            if (j < nch) ptx::mma_bf16(tmem_d, ad[j], bd[j], idesc, 1u);
                        accumulate = 1u;
                    }
                    slot = slot + 1 == row_slots ? 0 : slot + 1;
                }
            }
        } else {
            for (int i = 0; i < kp.rt; ++i) {
                const int blk = sm.tab[i];
                if (blk >= 0) {
                    const uint32_t a_lo = a_lo0 + static_cast<uint32_t>(slot) * seg16;
                    const uint32_t bl = b_lo0 + static_cast<uint32_t>(blk) * (BN * 2);
                    for (int j = 0; j < kp.nch; ++j) {
                        ptx::mma_bf16(tmem_d, (a_hi << 32) | (a_lo + 2u * j), (b_hi << 32) | (bl + j * chunk16), idesc,
                                      accumulate);
                        accumulate = 1u;
                    }
                }
                if (++slot == kp.row_slots) slot = 0;
            }
        }
        SGB_CYCLES_END(c_issue, t_issue);
        SGB_TRACE(kp, ti == 0, 24);
        ptx::mma_commit(&sm.acc_full[buf]);
    }
    SGB_TRACE(kp, true, 5);
    SGB_TRACE_VALUE(kp, true, 4, c_full);
    SGB_TRACE_VALUE(kp, true, 6, c_acc);
    SGB_TRACE_VALUE(kp, true, 9, c_issue);
    SGB_TRACE_VALUE(kp, true, 14, c_rel);
    // No MMA may be in flight when the CTA reaches its teardown.
    ptx::mma_commit(sm.mma_done);
    ptx::mbar_wait(sm.mma_done, 0u, kp.wait_limit_ns);
}

// ---------------------------------------------------------------- epilogue (warps 9..12)
// FUSED: the fused epilogue (ReLU, bf16 output) compiled in; the plain
// instantiation carries none of its code.
template <int BN, bool FUSED>
__device__ void rw_epilogue_impl(const RowWinParams& kp, const RwSmem& sm, uint32_t tmem_base, int t_lo, int t_hi)
{
    const int et = threadIdx.x - RW_EPI_WARP0 * 32;  // 0..127
    const int lane = threadIdx.x & 31;
    const int quad = (threadIdx.x >> 5) & 3;  // TMEM lane quadrant this warp may access
    const uint32_t saddr = ptx::smem_addr(sm.epi + (et >> 5) * RW_EPI_SLOT_BYTES);
    const bool add_bias = kp.bias != nullptr;
    const uint32_t acc_cols = static_cast<uint32_t>(kp.T * BN);
    uint64_t c_wacc = 0, c_ld = 0, c_st = 0;
    (void)c_wacc; (void)c_ld; (void)c_st;
    rw_stage_weights<BN>(kp, sm, et);
    ptx::fence_proxy_async_smem();  // generic-proxy writes -> tensor-core reads
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(sm.w_ready);
    SGB_TRACE(kp, et == 0, 2);
    int g_end = 0, freed = 0, freed_slot = 0;  // row release bookkeeping (thread et == 0)
    // Bias for the vector stores: lane l adds channels 32*j + 4*(l % 8) .. +3 after the
    // slot transpose.  (The row stores of K % 4 != 0 read theirs per slab.)
    float4 bias4[BN / 32];
#pragma unroll
    for (int j = 0; j < BN / 32; ++j) {
        const int n4 = j * 32 + (lane & 7) * 4;
        bias4[j] = (add_bias && kp.vec_store && n4 < kp.K) ? __ldg(reinterpret_cast<const float4*>(kp.bias + n4))
                                                          : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    int ti = 0;
    for (int t = t_lo; t < t_hi; ++t, ++ti) {
        const RwTile tl = rw_tile(kp, t);
        const int q0 = tl.qb * RW_TILE_M;
        const int nv = kp.Q - q0 < RW_TILE_M ? kp.Q - q0 : RW_TILE_M;  // valid pixels per output row
        const int rows_valid = kp.P - tl.p0 < kp.T ? kp.P - tl.p0 : kp.T;
        const int buf = ti & 1;
        const uint32_t use = static_cast<uint32_t>(ti >> 1) & 1u;
        SGB_CYCLES_BEGIN(t_wacc);
        if (!ptx::mbar_wait(&sm.acc_full[buf], use, kp.wait_limit_ns)) rw_record_timeout(kp, sm.abort_flag);
        ptx::named_bar_sync(1, RW_EPI_THREADS);
        if (et == 0) {
            const bool go = *sm.abort_flag == 0u;
            *sm.epi_go = go ? 1u : 0u;
            if (go) {
                // Tile t's MMAs are complete: release the rows no later tile of the CTA
                // reads (stream rows below the next tile's first window row), in order.
                g_end += rw_tile_rows(kp, t, t_lo, tl);
                int lim = g_end;
                if (t + 1 < t_hi) lim = g_end + rw_tile_rows(kp, t + 1, t_lo, rw_tile(kp, t + 1)) - kp.rt;
                for (; freed < lim; ++freed) {
                    ptx::mbar_arrive(&sm.empty[freed_slot]);
                    if (++freed_slot == kp.row_slots) freed_slot = 0;
                }
            }
        }
        ptx::named_bar_sync(1, RW_EPI_THREADS);
        SGB_CYCLES_END(c_wacc, t_wacc);
        if (!*sm.epi_go) break;
        SGB_TRACE(kp, et == 0 && ti == 0, 7);
        ptx::tc_fence_after();
#pragma unroll 1
        for (int b = 0; b < rows_valid; ++b) {
            const long long m0 = (static_cast<long long>(tl.n) * kp.P + tl.p0 + b) * kp.Q + q0;
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(buf) * acc_cols + static_cast<uint32_t>(b * BN) +
                                   (static_cast<uint32_t>(quad * 32) << 16);
            const bool last_b = b == rows_valid - 1;
            if (kp.vec_store) {
                // TMEM -> registers -> this warp's 32 x 32 swizzled staging slot -> 16-byte
                // global stores, 8 lanes per 128-byte row piece, the bias added per 16-byte
                // chunk after the transpose (slab_out: slot reads batched, stores predicated).
                const int rsub = lane >> 3;
                const int chunk = lane & 7;
                const int64_t esize = (FUSED && kp.out_bf16) ? 2 : 4;
                uint64_t rowp[8];
                uint32_t row_ok = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int row = quad * 32 + 4 * i + rsub;
                    row_ok |= (row < nv ? 1u : 0u) << i;
                    rowp[i] = reinterpret_cast<uint64_t>(kp.y) +
                              static_cast<uint64_t>(((m0 + (row < nv ? row : 0)) * kp.K + chunk * 4) * esize);
                }
#pragma unroll
                for (int j = 0; j < BN / 32; ++j) {
                    uint32_t v[32];
                    SGB_CYCLES_BEGIN(t_ld);
                    ptx::tmem_ld_32x32b_x32(taddr + j * 32, v);
                    ptx::tmem_ld_wait();
                    SGB_CYCLES_END(c_ld, t_ld);
                    if (last_b && j == BN / 32 - 1) {  // accumulator drained: the MMA thread may reuse it
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&sm.acc_empty[buf]);
                    }
                    SGB_CYCLES_BEGIN(t_st);
                    const bool col_ok = j * 32 + chunk * 4 < kp.K;
                    const int64_t off = static_cast<int64_t>(j) * 32 * esize;
                    if (FUSED && kp.out_bf16)
                        slab_out<SLAB_BF16>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], FUSED && kp.relu);
                    else
                        slab_out<SLAB_F32>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], FUSED && kp.relu);
                    SGB_CYCLES_END(c_st, t_st);
                }
            } else {
                // K % 4 != 0: each thread writes its own row.
                const int row = quad * 32 + lane;
                float* yrow = kp.y + (m0 + (row < nv ? row : 0)) * kp.K;
#pragma unroll
                for (int j = 0; j < BN / 32; ++j) {
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(taddr + j * 32, v);
                    ptx::tmem_ld_wait();
                    if (last_b && j == BN / 32 - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&sm.acc_empty[buf]);
                    }
                    if (add_bias) {
                        const int n = j * 32 + lane;
                        const float bias_l = n < kp.K ? __ldg(kp.bias + n) : 0.0f;  // lane l: channel 32*j + l
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(__uint_as_float(v[e]) + __shfl_sync(0xffffffffu, bias_l, e));
                    }
                    if (row >= nv) continue;
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int n = j * 32 + e;
                        if (n >= kp.K) break;
                        float o = __uint_as_float(v[e]);
                        if (FUSED && kp.relu) o = fmaxf(o, 0.0f);
                        if (FUSED && kp.out_bf16)
                            reinterpret_cast<uint16_t*>(kp.y)[(m0 + row) * kp.K + n] = ptx::bf16_bits(o);
                        else
                            yrow[n] = o;
                    }
                }
            }
        }
    }
    SGB_TRACE(kp, et == 0, 8);
    SGB_TRACE_VALUE(kp, et == 0, 11, c_wacc);
    SGB_TRACE_VALUE(kp, et == 0, 12, c_ld);
    SGB_TRACE_VALUE(kp, et == 0, 13, c_st);
}

// ---------------------------------------------------------------- the kernel
// FUSED selects the kernel instantiation with the fused epilogue, so that the
// plain one's register allocation is not shaped by code it never runs.
template <int BN, bool FUSED>
__global__ void __launch_bounds__(RW_THREADS, 1) conv2d_rowwin_kernel(const __grid_constant__ RowWinParams kp)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    RwSmem sm;
    sm.b = smem;
    sm.rows = smem + kp.off_rows;
    sm.raw = smem + kp.off_raw;
    sm.epi = smem + kp.off_epi;
    sm.full = reinterpret_cast<uint64_t*>(smem + kp.off_bar);
    sm.empty = sm.full + kp.row_slots;
    sm.acc_full = sm.empty + kp.row_slots;
    sm.acc_empty = sm.acc_full + 2;
    sm.mma_done = sm.acc_empty + 2;
    sm.w_ready = sm.mma_done + 1;
    sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.w_ready + 1);
    sm.tab = reinterpret_cast<int*>(smem + kp.off_tab);
    sm.abort_flag = sm.tmem_slot + 1;
    sm.epi_go = sm.tmem_slot + 2;
    sm.ld_abort = sm.tmem_slot + 3;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    SGB_TRACE(kp, threadIdx.x == 0, 0);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kp.row_slots; ++i) {
            ptx::mbar_init(&sm.full[i], RW_LOAD_THREADS / 32);  // one arrive per stager warp
            ptx::mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.acc_full[i], 1);
            ptx::mbar_init(&sm.acc_empty[i], RW_EPI_THREADS);
        }
        ptx::mbar_init(sm.mma_done, 1);
        ptx::mbar_init(sm.w_ready, RW_EPI_THREADS / 32);
        *sm.abort_flag = 0u;
        *sm.epi_go = 0u;
        *sm.ld_abort = 0u;
        ptx::mbar_init_fence();
    }
    if (warp == RW_MMA_WARP) {
        ptx::tmem_alloc(sm.tmem_slot, kp.tmem_cols);
        ptx::tmem_relinquish();
    }
    if (warp == RW_MMA_WARP + 1) ptx::touch_params(&kp, static_cast<int>(sizeof(kp)));
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;
    // Global memory is touched only after the previous kernel in the stream is done.
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    SGB_TRACE(kp, threadIdx.x == 0, 1);

    const int t_lo = static_cast<int>(static_cast<long long>(blockIdx.x) * kp.tiles / kp.grid);
    const int t_hi = static_cast<int>((static_cast<long long>(blockIdx.x) + 1) * kp.tiles / kp.grid);
    if (warp < RW_MMA_WARP) {
        rw_stager<BN>(kp, sm, t_lo, t_hi);
    } else if (warp == RW_MMA_WARP) {
        if (lane == 0) rw_mma<BN>(kp, sm, tmem_base, t_lo, t_hi);
    } else {
        rw_epilogue_impl<BN, FUSED>(kp, sm, tmem_base, t_lo, t_hi);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == RW_MMA_WARP) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, kp.tmem_cols);
    }
    SGB_TRACE(kp, threadIdx.x == 0, 10);
}

// Host-side launcher (instantiated once per channel-tile width in conv2d_rowwin.cu).
template <int BN>
cudaError_t launch_conv2d_rowwin(const RowWinParams& kp, int smem_bytes, bool pdl, cudaStream_t stream)
{
    const bool fused = (kp.relu | kp.out_bf16) != 0;
    auto kern = fused ? conv2d_rowwin_kernel<BN, true> : conv2d_rowwin_kernel<BN, false>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    // Opt in once per device and instantiation to the largest dynamic shared memory any launch asks for.
    static unsigned long long configured[2] = {0ull, 0ull};
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(__atomic_load_n(&configured[fused], __ATOMIC_ACQUIRE) & bit)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 232448);
        if (err != cudaSuccess) return err;
        if (bit) __atomic_fetch_or(&configured[fused], bit, __ATOMIC_RELEASE);
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(kp.grid));
    cfg.blockDim = dim3(RW_THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, kp);
}

#define SGB_ROWWIN_SIG(BN_) cudaError_t launch_conv2d_rowwin<BN_>(const RowWinParams&, int, bool, cudaStream_t)

}  // namespace sgb
