// Implicit-GEMM 2-D convolution forward on sm_103a tensor cores.
//
// GEMM view (burn PR #2287 "Introduce autotuning to conv2d ...", Changes; burn
// PR #2545 "[Optimization] Implicit gemm rewrite", Changes):
//   row    m  = (n*P + p)*Q + q            one output pixel, M = N*P*Q rows
//   column j  = k                          one output channel, K columns
//   reduction kk = (r*S + s)*C + c         one filter tap, C*R*S terms
//   A[m][kk] = x[n][p*sh-ph+r*dh][q*sw-pw+s*dw][c] (0 outside the image) -- the
//              im2col matrix, gathered tile by tile into shared memory and never
//              written to global memory;
//   B[j][kk] = w[j][r][s][c]               -- the KRSC weight viewed as [K][C*R*S].
//
// Work decomposition (stream-K).  The output is cut into BM x BN tiles and the
// reduction into BK-wide k-blocks; a work unit is one (tile, k-block) pair and
// the units are numbered tile-major.  CTA c of G takes the contiguous unit range
// [c*U/G, (c+1)*U/G), so every CTA gets the same number of MMAs however the tile
// count falls against the SM count.  A range covers a tail of one tile, whole
// tiles, and a head of another: a tile cut by range boundaries is split over
// consecutive CTAs, its "splits" in k-block order.  Classic split-K with S
// splits is the special case G = tiles * S.
//
// Splits of a tile are reduced in place in y (NVIDIA/Fuser issue #1316
// "Split-K matmul is slow even for few partitions", Eliminating the workspace),
// ordered by a per-tile semaphore; the fp32 output is the work buffer and the
// only extra memory is one 32-bit word per tile.  Split 0 always goes first: it
// stores acc + bias.  Then, in the ordered mode, the CTAs take turns -- split j
// waits until the semaphore reads j, adds its partial tile into y and publishes
// j+1 (bitwise reproducible); in the concurrent mode every later split waits only
// for split 0, adds with vector atomic adds in L2 in whatever order the splits
// finish, and counts itself done -- a chain of two steps instead of S.  The last
// split of a tile resets its semaphore to 0.  Each CTA walks its segments in
// reverse order, so the head of a cut tile (split 0, owned by the lower CTA) is
// computed first and the tail (a later split) last: turns are normally granted
// before they are asked for.
//
// Box loader (C % 128 == 0).  An im2col-mode TMA operation costs about as much
// as a tiled one however few bytes it moves, so the box loader makes each
// operation carry more: the tile is a rectangle of output pixels (bn_img images
// x bh rows x bw columns, px = bn_img*bh*bw <= BM), and for filter tap (r, s)
// its activation rows are one tiled box of the NHWC input viewed as 5-D
// {64 channels, W, H, N, C/64}, starting at the window origin of the
// rectangle's first pixel (traversal strides sh, sw; zero fill outside the
// image gives the padding).  One box brings KC = 2 consecutive 64-channel
// chunks, and one 3-D box of the weight viewed as {64, K, C*R*S/64} brings the
// matching two k-blocks of B, so a pipeline stage holds two k-blocks.  Chunk j
// of A lands px rows after chunk j-1 (any px: the 128-byte swizzle of the TMA
// write and of the MMA read follows absolute shared-memory addresses); the MMA
// reads 128 rows from each chunk start and the rows past px are ignored by the
// epilogue.
//
// Warp roles:
//   warp 0      TMA producer (one thread): the im2col activation tiles
//               (im2col-mode or box TMA) into a STAGES-deep shared-memory ring
//               guarded by full/empty mbarriers; with a gather loader, the
//               weight tiles instead;
//   warp 1      TMEM allocator and tcgen05.mma issuer (128 x BN x 16 per
//               instruction, lane 0) into two fp32 TMEM accumulators used in
//               turn; it learns that a stage has landed from a named barrier,
//               never by touching shared memory between its MMAs;
//   warps 2..9  epilogue (2..5 with a gather loader): TMEM -> registers (+ bias)
//               -> swizzled shared staging -> coalesced 16-byte global stores
//               (vector atomic adds for later splits), while the MMA warp
//               already fills the other accumulator;
//   warps 6..9  (cp.async and scalar loaders only) im2col gather into the ring;
//   warp 10     stage waiter: waits for each stage's full barrier, releases the
//               MMA warp by the stage's named barrier;
//   warp 11     (TMA loaders) TMA producer of the weight tiles; with the halo
//               loader warps 0, 11, 12 and 13 share the weight tiles by ring
//               slot and warp 0 also loads the halos.
// The ring replaces block-wide syncs between load and MMA (burn PR #2545's
// sync-placement discussion; ROCm/rocMLIR PR #1511 "Double buffering
// improvements" splits loads and MMAs into overlapping stages the same way).
//
// Every wait is bounded (about wait_limit_ns, counted in SM cycles).  A wait
// that runs out records CONV2D_ERR_TIMEOUT in the status word; the CTA then
// drains its own in-flight copies and MMAs, frees its tensor memory and exits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "fastdiv.h"
#include "ptx.cuh"
#include "slab_store.cuh"
#include "trace.cuh"

namespace sgb {

constexpr int MMA_M = 128;       // rows per tcgen05.mma (cta_group::1); a tile has BM/128 row blocks
constexpr int BK = 64;           // reduction elements per stage: one 128-byte bf16 row
constexpr int UMMA_K = 16;       // reduction per tcgen05.mma of kind::f16
constexpr int EPI_WARP0 = 2;     // epilogue warps 2..5 (2..9 with a TMA loader)
constexpr int GATHER_WARP0 = 6;  // gather warps 6..9 (gather loaders only)
constexpr int WAITER_WARP = 10;  // waits for each stage's data, releases the MMA warp by named barrier
constexpr int STAGE_BAR0 = 2;    // named barrier of ring stage s: STAGE_BAR0 + s (1 is the epilogue's)
constexpr int GATHER_THREADS = 128;
constexpr int EPI_SLOT_BYTES = 32 * 32 * 4;  // one warp's 32 rows x 32 fp32 columns
constexpr int EPI_SLOTS = 1;                 // staging slots per epilogue warp
constexpr uint32_t STATUS_TIMEOUT = 6;  // same value as CONV2D_ERR_TIMEOUT
constexpr int kMaxSmemBytes = 232448;   // opt-in dynamic shared memory per block (227 KB)

enum LoaderKind : int {
    LOADER_TMA = 1, LOADER_CPASYNC = 2, LOADER_SCALAR = 3, LOADER_HYBRID = 4, LOADER_BOX = 6, LOADER_HALO = 7,
    // Weight gradient: the same pipeline with the GEMM dw[k][(r,s,c)] = sum_l dy[l][k] * im2col(x)[l][(r,s,c)]
    // over the output pixels l, both operands MN-major in shared memory.
    LOADER_WGRAD = 8,
    // Data gradient at stride 1: the forward convolution of dy with the weight
    // w'[c][r][s][k] = w[k][R-1-r][S-1-s][c], read straight from w by TMA as an
    // MN-major operand (channels c contiguous), the taps flipped by coordinate.
    LOADER_DGRAD = 9
};

// Which engine brings in the im2col tile of the CTA's k-block number `it`:
// the TMA unit (im2col mode) or the gather warps (cp.async).  The hybrid
// loader alternates so that both engines work in parallel.
template <int LOADER>
__device__ __forceinline__ bool a_by_tma(int it)
{
    return LOADER == LOADER_TMA || LOADER == LOADER_BOX || LOADER == LOADER_WGRAD || LOADER == LOADER_DGRAD ||
           (LOADER == LOADER_HYBRID && (it & 1) == 0);
}
template <int LOADER>
__device__ __forceinline__ bool a_by_gather(int it)
{
    return LOADER == LOADER_CPASYNC || (LOADER == LOADER_HYBRID && (it & 1) == 1);
}

struct ConvKernelParams {
    const uint16_t* x;  // bf16 NHWC
    const uint16_t* w;  // bf16 KRSC
    const float* bias;  // [K] or nullptr
    float* y;           // fp32 NHWC = [M][K] (weight gradient: dw [K][R*S*C])
    int ldy;            // elements between consecutive rows of y: K (weight gradient: R*S*C)
    uint32_t* status;   // device status word or nullptr
    uint32_t* sems;     // one per output tile (needed whenever a tile is split)
    int N, H, W, C, K, R, S, P, Q;
    int sh, sw, ph, pw, dh, dw;
    int M, CRS, num_kb;       // CRS = R*S*Cg: reduction length of one output channel; num_kb: stages per tile
    // Groups: G groups of Cg input and Kg output channels; a tile's column block
    // lies inside one group (ntpg column blocks per group).  G = 1: Cg = C, Kg = K.
    int G, Cg, Kg, ntpg;
    int m_tiles, n_tiles;
    int grid;                 // G: CTAs sharing the unit range
    long long units;          // U = m_tiles * n_tiles * num_kb
    int vec_store;            // K % 4 == 0: 16-byte vector writes of y
    // Box loader only: the tile rectangle (bn_img images x bh rows x bw columns,
    // px of its pixels) and the tile grid over (images, rows, columns).
    int bw, bh, bn_img, px, q_blocks, p_blocks;
    // Halo loader only (stride 1): virtual row pitch wv = W + 2*pw, virtual
    // pixels per image vp = P*wv, 128-pixel tiles per image tpi, halo rows hr
    // and bytes per halo buffer (64 channels x wv x hr, 1024-B multiple).
    int wv, vp, tpi, halo_rows, halo_bytes;
    int halo_tx;  // bytes one halo box delivers: 128 * wv * halo_rows (halo_bytes rounds it up to 1024)
    int debug_flags;
    int reduce_concurrent;    // 1: later splits add concurrently after split 0; 0: strict turns
    // Fused epilogue: ReLU after the bias, and y stored as bf16 (round to nearest
    // even) instead of fp32.  A tile cut between CTAs cannot be reduced in y then:
    // its splits add their partial sums into `part` (fp32 [M][K], zero outside a
    // call) and the CTA that arrives last at the tile's counter finishes it.
    int relu, out_bf16;
    float* part;
    unsigned long long wait_limit_ns;
    unsigned long long* trace;  // per-CTA phase timestamps; only written in trace builds
    // CTA-pair kernel: divisions by the loop-invariant sizes (grid = pairs,
    // units, stages per tile, column blocks, P*Q, Q, C, S).
    FastDiv fd_grid, fd_units, fd_nkb, fd_ntiles, fd_pq, fd_q, fd_c, fd_s;
    // CTA-pair halo loader: row-blocks per image, the padded row pitch, and
    // weight stages per 64-channel chunk (ceil(R*S / taps per stage)).
    FastDiv fd_tpi, fd_wv, fd_tapst;
    // CTA-pair kernels: the pairs' unit ranges are rotated by this many units
    // (0 <= unit_offset < stages per tile) so that no range starts on a tile
    // boundary (see PairWalker).
    int unit_offset;
    // Data gradient (LOADER_DGRAD).  Filter tap (r, s) of the launch (kernel order,
    // flipped) reads the original tap (dg_r0 + dg_rm*(R-1-r), dg_s0 + dg_sm*(S-1-s))
    // of a filter with dg_S columns; stride 1 is (0, 1, 0, 1, S).  At stride > 1 a
    // launch computes one output phase (dg_phase = 1): its pixel (n, i, j) is dx
    // pixel (n, dg_a + dg_sh*i, dg_b + dg_sw*j) of a dx with dg_H x dg_W pixels.
    int dg_r0, dg_rm, dg_s0, dg_sm, dg_S;
    int dg_phase, dg_H, dg_W, dg_a, dg_b, dg_sh, dg_sw;
    // CTA-pair kernels: y as a 2-D fp32 tensor {K, M} (row pitch ldy) for TMA
    // stores and reductions of 32-column x 64-row boxes in the 128-byte swizzle;
    // tma_y = 0 when it is not encoded (the epilogue then writes with st.global).
    int tma_y;
    CUtensorMap tm_y;
};


// Tile BM x BN (BM = 128 or 256 output pixels, BN = 64/128/256 channels).  A
// 256-pixel tile is loaded with one im2col operation per k-block and computed
// as two 128-row MMAs into two TMEM accumulators: the TMA unit's cost is per
// operation, so this doubles the MMA work each activation load feeds.
template <int BM, int BN, int LOADER>
struct TileConfig {
    static_assert(BM == 128 || BM == 256, "BM must be 128 or 256");
    static_assert(BN == 64 || BN == 128 || BN == 256, "BN must be 64, 128 or 256");
    static_assert(BM == 128 || LOADER == LOADER_TMA || LOADER == LOADER_BOX, "256-pixel tiles need a TMA loader");
    static constexpr bool HALO = LOADER == LOADER_HALO;
    static constexpr bool WGRAD = LOADER == LOADER_WGRAD;
    static constexpr bool DGRAD = LOADER == LOADER_DGRAD;
    static constexpr int M_SUB = BM / MMA_M;  // 128-row MMA blocks per tile
    static constexpr int KC = LOADER == LOADER_BOX ? 2 : 1;  // k-blocks per pipeline stage
    // The halo loader keeps its activations in two halo buffers outside the ring.
    static constexpr int A_STAGE_BYTES = HALO ? 0 : KC * BM * BK * 2;
    static constexpr int B_STAGE_BYTES = KC * BN * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int STAGES =
        HALO ? (BN == 64 ? 8 : 4)
        : LOADER == LOADER_BOX ? (196608 / STAGE_BYTES > 8 ? 8 : 196608 / STAGE_BYTES)
        : BM == 128 ? (BN == 256 ? 4 : (BN == 128 ? 6 : 8)) : (BN == 256 ? 3 : 4);
    static_assert(STAGES >= 2, "the ring needs at least two stages");
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 9) * 8 + 16;
    // With a TMA loader the gather warps' places go to the epilogue: 8 warps, two
    // per TMEM lane quadrant, each writing half of the tile's columns.
    static constexpr int EPI_WARPS = (LOADER == LOADER_TMA || LOADER == LOADER_BOX || HALO || WGRAD || DGRAD) ? 8 : 4;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_SLOTS * EPI_SLOT_BYTES;
    // Without the halo loader's two halo buffers (2 * kp.halo_bytes, placed after the ring).
    static constexpr int SMEM_BYTES = RING_BYTES + EPI_BYTES + BAR_BYTES + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= kMaxSmemBytes, "exceeds the per-block shared-memory limit");
    static constexpr int ACC_COLS = M_SUB * BN;                   // TMEM columns of one accumulator set
    static constexpr int NUM_ACC = 2 * ACC_COLS <= 512 ? 2 : 1;   // double-buffered when TMEM allows
    static constexpr uint32_t TMEM_COLS = NUM_ACC * ACC_COLS;
    // With a TMA loader two producer warps issue the loads: warp 0 the
    // activation tiles, warp 11 the weight tiles.  One issuing thread completes
    // only about one TMA operation per ~0.3 us whatever its size (about as long
    // as the MMAs of a 128 x 256 stage take); giving each operand its own
    // thread halves the issue time per stage.  Each operand of each ring slot
    // thus has one issuer, loading its uses in order, and a slot's parity waits
    // never run more than one phase ahead of the MMA's releases.  (Gather
    // loaders: warp 0 issues the weight tiles.)
    static constexpr bool TMA_A = LOADER == LOADER_TMA || LOADER == LOADER_BOX || HALO || WGRAD || DGRAD;
    // The halo loader's only per-stage load is the weight tile: four threads
    // (warps 0, 11, 12, 13) share them, ring slot s going to producer s % 4.
    static constexpr int HALO_NB = 4;
    static_assert(!HALO || (BM == 128 && STAGES % HALO_NB == 0), "halo loader: 128-pixel tiles, a ring of 4k slots");
    static constexpr int NPROD = HALO ? HALO_NB : TMA_A ? 2 : 1;
    static_assert(STAGES <= 8, "one named barrier per stage: ids 2 .. 9");
    static constexpr int THREADS = (WAITER_WARP + NPROD) * 32;
};

struct SmemView {
    uint8_t* a;          // STAGES x A tile
    uint8_t* b;          // STAGES x B tile
    uint8_t* epi;        // EPI_WARPS x EPI_SLOTS staging slots
    uint64_t* full;      // STAGES
    uint64_t* empty;     // STAGES
    uint64_t* acc_full;  // 2: accumulator ready for the epilogue
    uint64_t* acc_empty; // 2: accumulator drained by the epilogue
    uint64_t* mma_done;  // teardown drain of the MMA pipe
    uint8_t* halo;          // halo loader: 2 halo buffers
    uint64_t* halo_full;    // 2: halo landed
    uint64_t* halo_empty;   // 2: halo no longer read by any MMA
    uint32_t* tmem_slot;
    volatile uint32_t* abort_flag;
    volatile uint32_t* epi_go;  // epilogue decision, written by one thread between two barriers
};

__device__ __forceinline__ void record_timeout(const ConvKernelParams& kp, volatile uint32_t* abort_flag)
{
    *abort_flag = 1u;
    if (kp.status) atomicMax(kp.status, STATUS_TIMEOUT);
}

// ---------------------------------------------------------------- work partition
struct Segment {
    int tile;      // output tile index (m_tile * n_tiles + n_tile)
    int kb_begin;  // k-block range of this segment inside the tile
    int kb_end;
    int split;     // position among the CTAs sharing the tile (k-block order)
    int nsplits;   // number of CTAs sharing the tile
};

// The CTA whose unit range contains unit u: the largest c with floor(c*U/G) <= u.
__device__ __forceinline__ int cta_of_unit(long long u, long long units, int grid)
{
    return static_cast<int>(((u + 1) * grid + units - 1) / units - 1);
}

// Walks this CTA's segments from the end of its unit range to the start.
struct SegmentWalker {
    long long lo, cur;
    __device__ __forceinline__ explicit SegmentWalker(const ConvKernelParams& kp)
    {
        lo = static_cast<long long>(blockIdx.x) * kp.units / kp.grid;
        cur = (static_cast<long long>(blockIdx.x) + 1) * kp.units / kp.grid;
    }
    __device__ __forceinline__ bool next(const ConvKernelParams& kp, Segment& sg)
    {
        if (cur <= lo) return false;
        const int t = static_cast<int>((cur - 1) / kp.num_kb);
        const long long base = static_cast<long long>(t) * kp.num_kb;
        const long long seg_lo = lo > base ? lo : base;
        sg.tile = t;
        sg.kb_begin = static_cast<int>(seg_lo - base);
        sg.kb_end = static_cast<int>(cur - base);
        const int first = cta_of_unit(base, kp.units, kp.grid);
        const int last = cta_of_unit(base + kp.num_kb - 1, kp.units, kp.grid);
        sg.split = static_cast<int>(blockIdx.x) - first;
        sg.nsplits = last - first + 1;
        cur = seg_lo;
        return true;
    }
};


// Pixel (n, p, q) of GEMM row m.
__device__ __forceinline__ void decode_pixel(const ConvKernelParams& kp, int m, int& n_img, int& p, int& q)
{
    const int pq = kp.P * kp.Q;
    n_img = m / pq;
    const int rem = m - n_img * pq;
    p = rem / kp.Q;
    q = rem - p * kp.Q;
}

// Output-channel range [n0, n_end) of a tile's column block and the first input
// channel of its group (grouped convolution: output channel n sums over the
// input channels of group n / Kg only).
template <int BN>
__device__ __forceinline__ void tile_columns(const ConvKernelParams& kp, int tile, int m_tile, int& n0, int& n_end,
                                             int& c_base)
{
    const int nt = tile - m_tile * kp.n_tiles;
    const int g = nt / kp.ntpg;
    n0 = g * kp.Kg + (nt - g * kp.ntpg) * BN;
    n_end = (g + 1) * kp.Kg;
    c_base = g * kp.Cg;
}

// Box loader: first image, row and column of the rectangle of tile row-block m_tile.
__device__ __forceinline__ void box_origin(const ConvKernelParams& kp, int m_tile, int& n0, int& p0, int& q0)
{
    const int qb = m_tile % kp.q_blocks;
    const int rest = m_tile / kp.q_blocks;
    const int pb = rest % kp.p_blocks;
    n0 = (rest / kp.p_blocks) * kp.bn_img;
    p0 = pb * kp.bh;
    q0 = qb * kp.bw;
}

// Halo loader.  Each image is seen as a grid of virtual pixels with the
// padded row pitch wv = W + 2*pw (stride 1): virtual pixel j = p*wv + v of an
// image is output pixel (p, v) when v < Q, and the input value of filter tap
// (r, s) for it sits at padded linear index j + r*dh*wv + s*dw, on padded row
// (j + r*dh*wv + s*dw) / wv.  A tile is 128 consecutive virtual pixels of one
// image, so for each 64-channel chunk one tiled TMA box of whole padded input
// rows (zero fill outside the image gives the padding) holds every tap's A
// operand: tap (r, s) is the 128 rows starting r*dh*wv + s*dw rows further on.
// The reduction runs chunk-major, then over the R*S taps.
__device__ __forceinline__ void halo_kb(const ConvKernelParams& kp, int kb, int& chunk, int& tap)
{
    const int rs = kp.R * kp.S;
    chunk = kb / rs;
    tap = kb - chunk * rs;
}

// A halo use starts at a chunk's first tap or a segment's first stage, and
// ends at the chunk's last tap or the segment's last stage.
__device__ __forceinline__ bool halo_starts(const Segment& sg, int kb, int tap) { return kb == sg.kb_begin || tap == 0; }
__device__ __forceinline__ bool halo_ends(const ConvKernelParams& kp, const Segment& sg, int kb, int tap)
{
    return kb + 1 == sg.kb_end || tap + 1 == kp.R * kp.S;
}

// Image, first virtual pixel and first padded input row of tile row-block m_tile.
__device__ __forceinline__ void halo_origin(const ConvKernelParams& kp, int m_tile, int& n_img, int& j0, int& prow0)
{
    n_img = m_tile / kp.tpi;
    j0 = (m_tile - n_img * kp.tpi) * MMA_M;
    prow0 = j0 / kp.wv;
}

// GEMM row (output pixel index) of row `row` of tile row-block m_tile, or -1
// when the row lies past the output.  (n0, p0, q0) is the box origin (box
// loader only).
// Data gradient: the original filter tap (index into R*S) that kernel tap (r, s)
// reads (the taps run flipped; at stride > 1 a phase's taps are every dg_rm-th row
// and dg_sm-th column of the filter).
__device__ __forceinline__ int dgrad_tap(const ConvKernelParams& kp, int r, int s)
{
    return (kp.dg_r0 + kp.dg_rm * (kp.R - 1 - r)) * kp.dg_S + (kp.dg_s0 + kp.dg_sm * (kp.S - 1 - s));
}

template <int BM, int LOADER>
__device__ __forceinline__ int tile_row_m(const ConvKernelParams& kp, int m_tile, int row, int n0, int p0, int q0)
{
    if constexpr (LOADER == LOADER_HALO) {
        (void)n0; (void)p0; (void)q0;
        const int n = m_tile / kp.tpi;
        const int j = (m_tile - n * kp.tpi) * MMA_M + row;
        if (j >= kp.vp) return -1;
        const int p = j / kp.wv;
        const int q = j - p * kp.wv;
        if (q >= kp.Q) return -1;
        return (n * kp.P + p) * kp.Q + q;
    } else if constexpr (LOADER == LOADER_BOX) {
        if (row >= kp.px) return -1;
        const int q = q0 + row % kp.bw;
        const int t = row / kp.bw;
        const int p = p0 + t % kp.bh;
        const int n = n0 + t / kp.bh;
        if (q >= kp.Q || p >= kp.P || n >= kp.N) return -1;
        return (n * kp.P + p) * kp.Q + q;
    } else if constexpr (LOADER == LOADER_DGRAD) {
        (void)n0; (void)p0; (void)q0;
        const int m = m_tile * BM + row;
        if (m >= kp.M) return -1;
        if (!kp.dg_phase) return m;
        // Phase pixel (n, i, j) -> dx pixel (n, a + sh*i, b + sw*j).
        const int j = m % kp.Q;
        const int t = m / kp.Q;
        const int i = t % kp.P;
        const int n = t / kp.P;
        return (n * kp.dg_H + kp.dg_a + kp.dg_sh * i) * kp.dg_W + kp.dg_b + kp.dg_sw * j;
    } else {
        (void)n0; (void)p0; (void)q0;
        const int m = m_tile * BM + row;
        return m < kp.M ? m : -1;
    }
}

// ---------------------------------------------------------------- TMA producer (warp 0, one thread)
// Coordinates of the TMA loads of one segment, stage by stage: the window
// origin of the tile's first pixel, the filter tap (r, s) and channel c of the
// stage's first k-block, and the tile's first output channel.
template <int BM, int BN, int LOADER>
struct LoadCursor {
    static constexpr int KC = TileConfig<BM, BN, LOADER>::KC;
    int n_img, w_org, h_org, c, r, s, n0, kb, c_base;  // c: channel within the group
    int k0;  // weight gradient: first output channel of the tile (its dy columns)
    LoadCursor() = default;
    __device__ __forceinline__ LoadCursor(const ConvKernelParams& kp, const Segment& sg)
    {
        const int m_tile = sg.tile / kp.n_tiles;
        int n_end;
        tile_columns<BN>(kp, sg.tile, m_tile, n0, n_end, c_base);
        if constexpr (LOADER == LOADER_WGRAD) {
            // Column block (tap, channel block): G = R*S taps of Kg = C columns each.
            const int tap = c_base / kp.Cg;
            r = tap / kp.S;
            s = tap - r * kp.S;
            c = n0 - tap * kp.C;
            k0 = m_tile * BM;
            kb = sg.kb_begin;
            set_pixel_origin(kp);
            return;
        }
        int p0, q0;
        if constexpr (LOADER == LOADER_BOX) box_origin(kp, m_tile, n_img, p0, q0);
        else decode_pixel(kp, m_tile * BM, n_img, p0, q0);
        w_org = q0 * kp.sw - kp.pw;
        h_org = p0 * kp.sh - kp.ph;
        kb = sg.kb_begin;
        const int kk0 = kb * KC * BK;
        const int rs0 = kk0 / kp.Cg;
        c = kk0 - rs0 * kp.Cg;
        r = rs0 / kp.S;
        s = rs0 - r * kp.S;
    }
    // Weight gradient: window origin of output pixel kb*BK (the stage's first reduction index).
    __device__ __forceinline__ void set_pixel_origin(const ConvKernelParams& kp)
    {
        int p0, q0;
        decode_pixel(kp, kb * BK, n_img, p0, q0);
        w_org = q0 * kp.sw - kp.pw;
        h_org = p0 * kp.sh - kp.ph;
    }
    __device__ __forceinline__ void advance(const ConvKernelParams& kp)
    {
        ++kb;
        if constexpr (LOADER == LOADER_WGRAD) {
            set_pixel_origin(kp);
            return;
        }
        c += KC * BK;
        if (c >= kp.Cg) {  // the im2col loaders need Cg % 64 == 0, the box loader C % 128 == 0
            c = 0;
            if (++s == kp.S) {
                s = 0;
                ++r;
            }
        }
    }
    // The stage's loads into shared memory, completing on `bar`: the activation
    // tile (`a_tma`: by the TMA unit) and the weight tile.  One issuing thread
    // has only about one TMA operation in flight at a time, so the two loads
    // are issued by two lanes of the producer warp, A by lane 0 and B by lane 1.
    __device__ __forceinline__ void load_a(const CUtensorMap* tm_a, const ConvKernelParams& kp, uint8_t* a_dst,
                                           uint64_t* bar) const
    {
        if constexpr (LOADER == LOADER_WGRAD) {
            // dy rows kb*BK .. +63 (output pixels), output channels k0 .. k0+127 as two
            // 64-column boxes: 128-byte rows of 64 channels, 8 KB apart.
            ptx::tma_load_2d(a_dst, tm_a, bar, k0, kb * BK);
            ptx::tma_load_2d(a_dst + BK * 128, tm_a, bar, k0 + 64, kb * BK);
        } else if constexpr (LOADER == LOADER_BOX)  // KC channel chunks of the rectangle's windows at tap (r, s)
            ptx::tma_load_5d(a_dst, tm_a, bar, 0, w_org + s * kp.dw, h_org + r * kp.dh, n_img, (c_base + c) / BK);
        else
            ptx::tma_load_im2col_4d(a_dst, tm_a, bar, c_base + c, w_org, h_org, n_img,
                                    static_cast<uint16_t>(s * kp.dw), static_cast<uint16_t>(r * kp.dh));
    }
    __device__ __forceinline__ void load_b(const CUtensorMap* tm_b, const ConvKernelParams& kp, uint8_t* b_dst,
                                           uint64_t* bar) const
    {
        if constexpr (LOADER == LOADER_WGRAD) {
            // im2col boxes of the stage's 64 output pixels at tap (r, s): BN / 64 boxes of
            // 64 channels, each 64 pixel rows of 128 bytes, 8 KB apart.
#pragma unroll
            for (int i = 0; i < BN / 64; ++i)
                ptx::tma_load_im2col_4d(b_dst + i * BK * 128, tm_b, bar, c + 64 * i, w_org, h_org, n_img,
                                        static_cast<uint16_t>(s * kp.dw), static_cast<uint16_t>(r * kp.dh));
        } else if constexpr (LOADER == LOADER_DGRAD) {
            // w as {C, R*S, K}: for the flipped tap, output channels n0 + 64i .. +63 (contiguous)
            // x dy channels c .. c+63 (rows): BN / 64 boxes of 64 rows of 128 bytes, 8 KB apart.
            const int tap = dgrad_tap(kp, r, s);
#pragma unroll
            for (int i = 0; i < BN / 64; ++i) ptx::tma_load_3d(b_dst + i * BK * 128, tm_b, bar, n0 + 64 * i, tap, c);
        } else if constexpr (LOADER == LOADER_BOX) ptx::tma_load_3d(b_dst, tm_b, bar, 0, n0, kb * KC);  // KC k-blocks
        else ptx::tma_load_2d(b_dst, tm_b, bar, kb * BK, n0);
    }
    // The same reads as L2 prefetches (nothing lands in shared memory).
    __device__ __forceinline__ void prefetch(const CUtensorMap* tm_a, const CUtensorMap* tm_b,
                                             const ConvKernelParams& kp) const
    {
        if constexpr (LOADER == LOADER_WGRAD) {
            ptx::tma_prefetch_2d(tm_a, k0, kb * BK);
            ptx::tma_prefetch_2d(tm_a, k0 + 64, kb * BK);
            for (int i = 0; i < BN / 64; ++i)
                ptx::tma_prefetch_im2col_4d(tm_b, c + 64 * i, w_org, h_org, n_img, static_cast<uint16_t>(s * kp.dw),
                                            static_cast<uint16_t>(r * kp.dh));
        } else if constexpr (LOADER == LOADER_BOX) {
            ptx::tma_prefetch_5d(tm_a, 0, w_org + s * kp.dw, h_org + r * kp.dh, n_img, (c_base + c) / BK);
            ptx::tma_prefetch_3d(tm_b, 0, n0, kb * KC);
        } else if constexpr (LOADER == LOADER_DGRAD) {
            ptx::tma_prefetch_im2col_4d(tm_a, c, w_org, h_org, n_img, static_cast<uint16_t>(s * kp.dw),
                                        static_cast<uint16_t>(r * kp.dh));
            const int tap = dgrad_tap(kp, r, s);
            for (int i = 0; i < BN / 64; ++i) ptx::tma_prefetch_3d(tm_b, n0 + 64 * i, tap, c);
        } else {
            ptx::tma_prefetch_im2col_4d(tm_a, c_base + c, w_org, h_org, n_img, static_cast<uint16_t>(s * kp.dw),
                                        static_cast<uint16_t>(r * kp.dh));
            ptx::tma_prefetch_2d(tm_b, kb * BK, n0);
        }
    }
};

// Before the wait for the previous kernel: L2 prefetches of the CTA's first
// STAGES loads, so that its pipeline fills from L2 once the wait returns.  A
// prefetch moves nothing into the CTA and reads through L2, the GPU's point of
// coherence, so it cannot observe or disturb the previous kernel's writes.
template <int BM, int BN, int LOADER>
__device__ void prefetch_first_stages(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const ConvKernelParams& kp)
{
    SegmentWalker walk(kp);
    Segment sg;
    if (!walk.next(kp, sg)) return;
    if constexpr (LOADER == LOADER_HALO) {
        const int m_tile = sg.tile / kp.n_tiles;
        const int n0 = (sg.tile - m_tile * kp.n_tiles) * BN;
        int n_img, j0, prow0, chunk, tap;
        halo_origin(kp, m_tile, n_img, j0, prow0);
        halo_kb(kp, sg.kb_begin, chunk, tap);
        ptx::tma_prefetch_4d(tm_a, chunk * BK, -kp.pw, prow0 - kp.ph, n_img);
        for (int kb = sg.kb_begin; kb < sg.kb_end && kb < sg.kb_begin + TileConfig<BM, BN, LOADER>::STAGES; ++kb) {
            halo_kb(kp, kb, chunk, tap);
            ptx::tma_prefetch_2d(tm_b, tap * kp.C + chunk * BK, n0);
        }
        return;
    }
    LoadCursor<BM, BN, LOADER> cur(kp, sg);
    for (int i = 0; i < TileConfig<BM, BN, LOADER>::STAGES && cur.kb < sg.kb_end; ++i) {
        cur.prefetch(tm_a, tm_b, kp);
        cur.advance(kp);
    }
}

// TMA producer (one thread).  OPS selects what it loads: PROD_A the
// activation tiles, PROD_B the weight tiles, PROD_AB both (gather loaders'
// warp 0, which loads the weight tiles and, for the hybrid loader, the even
// stages' activations).
enum ProducerOps : int { PROD_A = 1, PROD_B = 2, PROD_AB = 3 };

template <int BM, int BN, int LOADER, int OPS>
__device__ void run_tma_producer(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const ConvKernelParams& kp,
                                 const SmemView& sm)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int A_STAGE_BYTES = Cfg::A_STAGE_BYTES;
    constexpr int KC = Cfg::KC;
    const uint32_t a_bytes = LOADER == LOADER_BOX ? static_cast<uint32_t>(KC * kp.px * BK * 2) : A_STAGE_BYTES;
    int it = 0;  // stages issued so far (all segments)
    bool ok = true;
    uint64_t wait_cycles = 0, issue_cycles = 0;
    (void)wait_cycles;
    (void)issue_cycles;
    SegmentWalker walk(kp);
    Segment sg;
    while (ok && walk.next(kp, sg)) {
        LoadCursor<BM, BN, LOADER> cur(kp, sg);
        for (; cur.kb < sg.kb_end; cur.advance(kp), ++it) {
            const int stage = it % STAGES;
            SGB_CYCLES_BEGIN(tw);
            if (*sm.abort_flag) { ok = false; break; }
            if (!ptx::mbar_wait(&sm.empty[stage], (static_cast<uint32_t>(it / STAGES) & 1u) ^ 1u, kp.wait_limit_ns)) {
                record_timeout(kp, sm.abort_flag);
                ok = false;
                break;
            }
            SGB_CYCLES_END(wait_cycles, tw);
            SGB_CYCLES_BEGIN(ti);
            const bool a_tma = (OPS & PROD_A) && a_by_tma<LOADER>(it);
            const uint32_t bytes = (a_tma ? a_bytes : 0u) + ((OPS & PROD_B) ? Cfg::B_STAGE_BYTES : 0u);
            ptx::mbar_arrive_expect_tx(&sm.full[stage], bytes);
            if (a_tma) cur.load_a(tm_a, kp, sm.a + stage * A_STAGE_BYTES, &sm.full[stage]);
            if (OPS & PROD_B) cur.load_b(tm_b, kp, sm.b + stage * Cfg::B_STAGE_BYTES, &sm.full[stage]);
            SGB_STAGE_MARK(kp, it, (OPS & PROD_A) ? 0 : 1);
            SGB_CYCLES_END(issue_cycles, ti);
        }
    }
    SGB_TRACE(kp, (OPS & PROD_A) != 0, 3);
    SGB_TRACE_VALUE(kp, (OPS & PROD_A) != 0, 2, wait_cycles);
    SGB_TRACE_VALUE(kp, (OPS & PROD_A) != 0, 18, issue_cycles);
    SGB_TRACE_VALUE(kp, OPS == PROD_B, 19, wait_cycles | (issue_cycles << 32));
    // Drain: this producer's last load of each slot must have landed before the CTA can exit.
    for (int i = it > STAGES ? it - STAGES : 0; i < it; ++i)
        ptx::mbar_wait(&sm.full[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u, kp.wait_limit_ns);
}

// ---------------------------------------------------------------- halo producers (warps 0, 11, 12, 13)
// Producer `role` loads the weight tiles of the ring slots s % HALO_NB == role;
// role 0 (warp 0) also issues the halo of each (segment, chunk).  Each ring
// slot and each halo buffer thus has one issuer, loading its uses in order.
template <int BM, int BN, int LOADER>
__device__ void run_halo_producer(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const ConvKernelParams& kp,
                                  const SmemView& sm, int role)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int NB = Cfg::HALO_NB;
    int it = 0;  // stages walked (all segments)
    int h = 0;   // halo uses issued (role 0)
    bool ok = true;
    SegmentWalker walk(kp);
    Segment sg;
    while (ok && walk.next(kp, sg)) {
        const int m_tile = sg.tile / kp.n_tiles;
        const int n0 = (sg.tile - m_tile * kp.n_tiles) * BN;
        int n_img, j0, prow0;
        halo_origin(kp, m_tile, n_img, j0, prow0);
        for (int kb = sg.kb_begin; kb < sg.kb_end; ++kb, ++it) {
            int chunk, tap;
            halo_kb(kp, kb, chunk, tap);
            if (*sm.abort_flag) { ok = false; break; }
            if (role == 0 && halo_starts(sg, kb, tap)) {
                const int slot = h & 1;
                if (!ptx::mbar_wait(&sm.halo_empty[slot], (static_cast<uint32_t>(h >> 1) & 1u) ^ 1u,
                                    kp.wait_limit_ns)) {
                    record_timeout(kp, sm.abort_flag);
                    ok = false;
                    break;
                }
                ptx::mbar_arrive_expect_tx(&sm.halo_full[slot], static_cast<uint32_t>(kp.halo_tx));
                ptx::tma_load_4d(sm.halo + slot * kp.halo_bytes, tm_a, &sm.halo_full[slot], chunk * BK, -kp.pw,
                                 prow0 - kp.ph, n_img);
                SGB_STAGE_MARK(kp, it, 0);
                ++h;
            }
            const int stage = it % STAGES;
            if (stage % NB != role) continue;
            if (!ptx::mbar_wait(&sm.empty[stage], (static_cast<uint32_t>(it / STAGES) & 1u) ^ 1u, kp.wait_limit_ns)) {
                record_timeout(kp, sm.abort_flag);
                ok = false;
                break;
            }
            ptx::mbar_arrive_expect_tx(&sm.full[stage], Cfg::B_STAGE_BYTES);
            ptx::tma_load_2d(sm.b + stage * Cfg::B_STAGE_BYTES, tm_b, &sm.full[stage], tap * kp.C + chunk * BK, n0);
            SGB_STAGE_MARK(kp, it, 1);
        }
    }
    // Drain: this thread's last halo of each buffer and last load of each of its slots must have landed.
    if (role == 0)
        for (int i = h > 2 ? h - 2 : 0; i < h; ++i)
            ptx::mbar_wait(&sm.halo_full[i & 1], static_cast<uint32_t>(i >> 1) & 1u, kp.wait_limit_ns);
    for (int i = it > STAGES ? it - STAGES : 0; i < it; ++i)
        if ((i % STAGES) % NB == role)
            ptx::mbar_wait(&sm.full[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u, kp.wait_limit_ns);
}

// ---------------------------------------------------------------- stage waiter (warp 10)
// Waits (bounded) for each ring stage's data in the MMA's order and releases
// the MMA warp through the stage's named barrier.  The MMA warp never touches
// shared memory between its MMAs: the tensor pipe queues little work, and a
// shared-memory access issued after a group of tcgen05.mma instructions
// returns only once they have drained, leaving the pipe idle for ~200 cycles
// per stage.
//
// Named-barrier generations must pair one waiter arrival with one MMA-warp
// sync, so the waiter may arrive for use u of a stage only after the MMA warp
// has passed that stage's use u - 1.  Normally the data guarantees it: use u
// was loaded after the MMA released use u - 1.  After a timeout the waiter
// stops waiting for data and waits instead for that release on the stage's
// empty barrier (the MMA warp commits every stage, issuing or not), so the MMA
// warp still runs to its end; its MMAs may then read stale data, and the
// epilogue stores nothing once the abort flag is set.
template <int BM, int BN, int LOADER>
__device__ void run_stage_waiter(const ConvKernelParams& kp, const SmemView& sm)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int STAGES = Cfg::STAGES;
    const int lane = threadIdx.x & 31;
    bool waiting = true;
    int it = 0;
    int h = 0;  // halo uses (halo loader)
    uint64_t full_cycles = 0;
    (void)full_cycles;
    SegmentWalker walk(kp);
    Segment sg;
    while (walk.next(kp, sg)) {
        for (int kb = sg.kb_begin; kb < sg.kb_end; ++kb, ++it) {
            const int stage = it % STAGES;
            const uint32_t use = static_cast<uint32_t>(it / STAGES);
            if constexpr (Cfg::HALO) {
                int chunk, tap;
                halo_kb(kp, kb, chunk, tap);
                if (halo_starts(sg, kb, tap)) {
                    if (lane == 0 && waiting &&
                        !ptx::mbar_wait(&sm.halo_full[h & 1], static_cast<uint32_t>(h >> 1) & 1u, kp.wait_limit_ns)) {
                        record_timeout(kp, sm.abort_flag);
                        waiting = false;
                    }
                    ++h;
                }
            }
            if (lane == 0) {
                SGB_CYCLES_BEGIN(tf);
                if (waiting && (*sm.abort_flag || !ptx::mbar_wait(&sm.full[stage], use & 1u, kp.wait_limit_ns))) {
                    record_timeout(kp, sm.abort_flag);
                    waiting = false;
                }
                // The MMA warp always gets this far (its only other waits are bounded),
                // so the release comes; the retry cap only bounds the loop.
                if (!waiting && use > 0)
                    for (int t = 0; t < 16 && !ptx::mbar_wait(&sm.empty[stage], (use - 1u) & 1u, kp.wait_limit_ns); ++t) {
                    }
                SGB_CYCLES_END(full_cycles, tf);
                SGB_STAGE_MARK(kp, it, 2);
            }
            __syncwarp();
            ptx::named_bar_arrive(STAGE_BAR0 + stage, 64);
        }
    }
    SGB_TRACE_VALUE(kp, lane == 0, 4, full_cycles);
}

// ---------------------------------------------------------------- MMA issuer (warp 1)
// The whole warp walks the stages (named barriers count warps); lane 0 issues.
template <int BM, int BN, int LOADER>
__device__ void run_mma_issuer(const ConvKernelParams& kp, const SmemView& sm, uint32_t tmem_base)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int A_STAGE_BYTES = Cfg::A_STAGE_BYTES;
    constexpr uint32_t IDESC = Cfg::WGRAD   ? ptx::idesc_bf16_f32_mn(MMA_M, BN)
                               : Cfg::DGRAD ? ptx::idesc_bf16_f32_bmn(MMA_M, BN)
                                            : ptx::idesc_bf16_f32(MMA_M, BN);
    const int lane = threadIdx.x & 31;
    // Weight gradient: MN-major operands, 64-element blocks along M/N 8 KB apart
    // (one 64-row TMA box each), groups of 8 reduction rows 1024 B apart.
    const uint64_t a_desc0 = Cfg::WGRAD ? ptx::sw128_mnmajor_desc(ptx::smem_addr(sm.a), BK * 128, 1024)
                                        : ptx::sw128_kmajor_desc(ptx::smem_addr(sm.a));
    const uint64_t b_desc0 = (Cfg::WGRAD || Cfg::DGRAD) ? ptx::sw128_mnmajor_desc(ptx::smem_addr(sm.b), BK * 128, 1024)
                                                        : ptx::sw128_kmajor_desc(ptx::smem_addr(sm.b));
    // Reduction step of one MMA (16 elements): 32 B along a K-major row, 16 rows of
    // 128 B in an MN-major tile.
    constexpr int KSTEP_A = Cfg::WGRAD ? UMMA_K * 128 : UMMA_K * 2;
    constexpr int KSTEP_B = (Cfg::WGRAD || Cfg::DGRAD) ? UMMA_K * 128 : UMMA_K * 2;
    const uint32_t a_chunk16 = LOADER == LOADER_BOX ? static_cast<uint32_t>(kp.px * 8) : 0u;
    const uint64_t halo_desc0 = Cfg::HALO ? ptx::sw128_kmajor_desc(ptx::smem_addr(sm.halo)) : 0ull;
    int h = 0;  // halo uses (halo loader)
    int it = 0, seg_idx = 0;
    bool issue = true;  // false once a wait has run out: keep pace with the waiter, issue nothing
    uint64_t acc_cycles = 0;
    (void)acc_cycles;
    SegmentWalker walk(kp);
    Segment sg;
    while (walk.next(kp, sg)) {
        const int buf = seg_idx % Cfg::NUM_ACC;
        const uint32_t use = static_cast<uint32_t>(seg_idx / Cfg::NUM_ACC) & 1u;
        // The epilogue must have drained this accumulator's previous segment.
        if (lane == 0 && issue) {
            SGB_CYCLES_BEGIN(ta);
            if (*sm.abort_flag || !ptx::mbar_wait(&sm.acc_empty[buf], use ^ 1u, kp.wait_limit_ns)) {
                record_timeout(kp, sm.abort_flag);
                issue = false;
            }
            SGB_CYCLES_END(acc_cycles, ta);
        }
        __syncwarp();
        ptx::tc_fence_after();
        const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(buf * Cfg::ACC_COLS);
        // Halo loader: buffer row of the tile's first virtual pixel, and the
        // filter tap (tap = r*S + fs) of the stage, stepped without divisions.
        int a_row0 = 0, tap = 0, fr = 0, fs = 0;
        if constexpr (Cfg::HALO) {
            int n_img, j0, prow0, chunk;
            halo_origin(kp, sg.tile / kp.n_tiles, n_img, j0, prow0);
            a_row0 = j0 - prow0 * kp.wv;
            halo_kb(kp, sg.kb_begin, chunk, tap);
            fr = tap / kp.S;
            fs = tap - fr * kp.S;
        }
        for (int kb = sg.kb_begin; kb < sg.kb_end; ++kb, ++it) {
            const int stage = it % STAGES;
            int halo_slot = 0;
            bool halo_last = false;
            uint64_t halo_ad = 0;
            if constexpr (Cfg::HALO) {
                if (kb == sg.kb_begin || tap == 0) ++h;
                halo_slot = (h - 1) & 1;
                halo_last = kb + 1 == sg.kb_end || tap + 1 == kp.R * kp.S;
                const int a_row = a_row0 + fr * kp.dh * kp.wv + fs * kp.dw;
                halo_ad = halo_desc0 + static_cast<uint64_t>((halo_slot * kp.halo_bytes + a_row * 128) >> 4);
                ++tap;
                if (++fs == kp.S) {
                    fs = 0;
                    ++fr;
                }
                if (tap == kp.R * kp.S) tap = fr = 0;
            }
            ptx::named_bar_sync(STAGE_BAR0 + stage, 64);
            ptx::tc_fence_after();
            if (lane == 0) SGB_STAGE_MARK(kp, it, 3);
            if (lane == 0 && issue) {
                // Gathered tiles were written through the generic proxy (cp.async);
                // order them before the tensor cores read the stage.
                if (LOADER == LOADER_CPASYNC || LOADER == LOADER_HYBRID) ptx::fence_proxy_async_smem();
                // Descriptor start addresses are address >> 4 in the low bits (no
                // carry: shared addresses < 256 KB), so an offset is added to the
                // descriptor itself; advancing along K inside a 128-B swizzled row
                // moves the start address by 32 B.  A stage with KC k-blocks holds
                // them as KC chunks, a_chunk16 apart (in 16-B units).
                const uint64_t ad =
                    Cfg::HALO ? halo_ad : a_desc0 + static_cast<uint64_t>((stage * A_STAGE_BYTES) >> 4);
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((stage * Cfg::B_STAGE_BYTES) >> 4);
                constexpr int KSTEPS = Cfg::KC * BK / UMMA_K;
                const uint32_t acc0 = kb > sg.kb_begin ? 1u : 0u;
#pragma unroll
                for (int k = 0; k < KSTEPS; ++k) {
                    const int chunk = k / (BK / UMMA_K), kin = k % (BK / UMMA_K);
                    const uint64_t bdk = bd + static_cast<uint64_t>((chunk * BN * 128 + kin * KSTEP_B) >> 4);
#pragma unroll
                    for (int sub = 0; sub < Cfg::M_SUB; ++sub)  // 128-row blocks share the B tile
                        ptx::mma_bf16(tmem_d + sub * BN,
                                      ad + static_cast<uint64_t>(chunk) * a_chunk16 +
                                          static_cast<uint64_t>((sub * MMA_M * 128 + kin * KSTEP_A) >> 4),
                                      bdk, IDESC, k > 0 ? 1u : acc0);
                }
            }
            if (lane == 0) {
                ptx::mma_commit(&sm.empty[stage]);  // every stage, issuing or not
                if (Cfg::HALO && halo_last) ptx::mma_commit(&sm.halo_empty[halo_slot]);
            }
            __syncwarp();
        }
        if (lane == 0) ptx::mma_commit(&sm.acc_full[buf]);  // also when not issuing: the epilogue must not wait out
        __syncwarp();
        ++seg_idx;
    }
    SGB_TRACE(kp, lane == 0, 5);
    SGB_TRACE_VALUE(kp, lane == 0, 6, acc_cycles);
    // No MMA may be in flight when the CTA reaches its teardown.
    if (lane == 0) {
        ptx::mma_commit(sm.mma_done);
        ptx::mbar_wait(sm.mma_done, 0u, kp.wait_limit_ns);
    }
    __syncwarp();
}

// ---------------------------------------------------------------- gather producers (warps 6..9)
// A tile by 16-byte cp.async (needs C % 8 == 0).  Thread t copies 16-byte
// chunk (t % 8) -- 8 consecutive channels -- of tile rows t/8 + 16*i, i = 0..7,
// so each warp instruction moves four whole 128-byte rows (one per pixel) and
// the filter-tap decode (r, s, c) happens once per k-block per thread.  Every
// thread hands its copies to the stage's full barrier with a non-blocking
// cp.async arrive, so the gather runs as far ahead as the ring allows; the MMA
// thread fences the async proxy after its wait (run_mma_issuer).
template <int BM, int BN, int LOADER>
__device__ void run_gather_cpasync(const ConvKernelParams& kp, const SmemView& sm)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int A_STAGE_BYTES = Cfg::A_STAGE_BYTES;
    constexpr int ROWS = BM / 16;  // tile rows per thread
    const int gt = threadIdx.x - GATHER_WARP0 * 32;
    const int lane = threadIdx.x & 31;
    const int chunk = gt & 7;
    const int row0 = gt >> 3;
    int it = 0;
    bool ok = true;
    uint64_t g_empty = 0, g_issue = 0;
    (void)g_empty; (void)g_issue;
    SegmentWalker walk(kp);
    Segment sg;
    while (ok && walk.next(kp, sg)) {
        const int m_base = (sg.tile / kp.n_tiles) * BM;
        int gn0, gn_end, c_base;
        tile_columns<BN>(kp, sg.tile, sg.tile / kp.n_tiles, gn0, gn_end, c_base);
        int ih0[ROWS], iw0[ROWS], img[ROWS];
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            const int m = m_base + row0 + 16 * i;
            int n_img = 0, p = 0, q = 0;
            if (m < kp.M) decode_pixel(kp, m, n_img, p, q);
            // Rows past M get an origin far outside the image, so every tap zero-fills.
            ih0[i] = m < kp.M ? p * kp.sh - kp.ph : -(1 << 28);
            iw0[i] = q * kp.sw - kp.pw;
            img[i] = n_img * kp.H * kp.W * kp.C;
        }
        for (int kb = sg.kb_begin; kb < sg.kb_end; ++kb, ++it) {
            const int stage = it % STAGES;
            const uint32_t parity = static_cast<uint32_t>(it / STAGES) & 1u;
            // One lane waits for the slot; the warp follows its verdict.
            int go = 0;
            SGB_CYCLES_BEGIN(t_e);
            if (lane == 0) {
                go = *sm.abort_flag == 0u;
                if (go && !ptx::mbar_wait(&sm.empty[stage], parity ^ 1u, kp.wait_limit_ns)) {
                    record_timeout(kp, sm.abort_flag);
                    go = 0;
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) { ok = false; break; }
            SGB_CYCLES_END(g_empty, t_e);
            SGB_CYCLES_BEGIN(t_i);
            if (a_by_gather<LOADER>(it)) {  // otherwise the TMA unit loads this k-block
                uint8_t* dst = sm.a + stage * A_STAGE_BYTES;
                const int kk = kb * BK + chunk * 8;
                const bool col_ok = kk < kp.CRS;
                int dih = 0, diw = 0, c = 0;
                if (col_ok) {
                    const int rs = kk / kp.Cg;
                    c = c_base + (kk - rs * kp.Cg);
                    const int r = rs / kp.S;
                    dih = r * kp.dh;
                    diw = (rs - r * kp.S) * kp.dw;
                }
#pragma unroll
                for (int i = 0; i < ROWS; ++i) {
                    const int ih = ih0[i] + dih;
                    const int iw = iw0[i] + diw;
                    const bool in = col_ok && static_cast<unsigned>(ih) < static_cast<unsigned>(kp.H) &&
                                    static_cast<unsigned>(iw) < static_cast<unsigned>(kp.W);
                    const uint16_t* src = in ? kp.x + img[i] + (ih * kp.W + iw) * kp.C + c : kp.x;
                    ptx::cp_async_16(dst + sw128_offset(row0 + 16 * i, chunk), src, in ? 16u : 0u);
                }
            }
            ptx::cp_async_arrive_noinc(&sm.full[stage]);
            SGB_CYCLES_END(g_issue, t_i);
        }
    }
    SGB_TRACE_VALUE(kp, gt == 0, 16, g_empty);
    SGB_TRACE_VALUE(kp, gt == 0, 17, g_issue);
    ptx::cp_async_wait_all();  // no copy may be in flight when the CTA exits
}

// A and B tiles element by element (any C, any C*R*S): plain loads, then
// 16-byte shared stores in the swizzled layout.
template <int BM, int BN, int LOADER>
__device__ void run_gather_scalar(const ConvKernelParams& kp, const SmemView& sm)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    static_assert(BM == GATHER_THREADS, "one tile row per gather thread");
    constexpr int STAGES = Cfg::STAGES;
    constexpr int A_STAGE_BYTES = Cfg::A_STAGE_BYTES;
    const int row = threadIdx.x - GATHER_WARP0 * 32;
    const int lane = threadIdx.x & 31;
    int it = 0;
    bool ok = true;
    SegmentWalker walk(kp);
    Segment sg;
    while (ok && walk.next(kp, sg)) {
        const int m_tile = sg.tile / kp.n_tiles;
        int n0, n_end, c_base;
        tile_columns<BN>(kp, sg.tile, m_tile, n0, n_end, c_base);
        const int m = m_tile * BM + row;
        const bool row_ok = m < kp.M;
        int n_img = 0, p = 0, q = 0;
        if (row_ok) decode_pixel(kp, m, n_img, p, q);
        const int ih0 = p * kp.sh - kp.ph;
        const int iw0 = q * kp.sw - kp.pw;
        const uint16_t* xb = kp.x + static_cast<int64_t>(n_img) * kp.H * kp.W * kp.C + c_base;
        for (int kb = sg.kb_begin; kb < sg.kb_end; ++kb, ++it) {
            const int stage = it % STAGES;
            const uint32_t parity = static_cast<uint32_t>(it / STAGES) & 1u;
            int go = 0;
            if (lane == 0) {
                go = *sm.abort_flag == 0u;
                if (go && !ptx::mbar_wait(&sm.empty[stage], parity ^ 1u, kp.wait_limit_ns)) {
                    record_timeout(kp, sm.abort_flag);
                    go = 0;
                }
            }
            if (!__shfl_sync(0xffffffffu, go, 0)) { ok = false; break; }
            const int kk0 = kb * BK;
            // A row: walk (r, s, c) incrementally from kk0.
            {
                const int rs0 = kk0 / kp.Cg;
                int c = kk0 - rs0 * kp.Cg;
                int r = rs0 / kp.S;
                int s = rs0 - r * kp.S;
                const uint32_t base = ptx::smem_addr(sm.a + stage * A_STAGE_BYTES);
#pragma unroll 1
                for (int j = 0; j < BK / 8; ++j) {
                    uint32_t packed[4];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int kk = kk0 + j * 8 + e;
                        uint32_t v = 0;
                        if (row_ok && kk < kp.CRS) {
                            const int ih = ih0 + r * kp.dh;
                            const int iw = iw0 + s * kp.dw;
                            if (static_cast<unsigned>(ih) < static_cast<unsigned>(kp.H) &&
                                static_cast<unsigned>(iw) < static_cast<unsigned>(kp.W))
                                v = __ldg(reinterpret_cast<const unsigned short*>(
                                    xb + (static_cast<int64_t>(ih) * kp.W + iw) * kp.C + c));
                        }
                        if (e & 1) packed[e >> 1] |= v << 16;
                        else packed[e >> 1] = v;
                        if (++c == kp.Cg) {
                            c = 0;
                            if (++s == kp.S) {
                                s = 0;
                                ++r;
                            }
                        }
                    }
                    ptx::st_shared_v4(base + sw128_offset(row, j), packed[0], packed[1], packed[2], packed[3]);
                }
            }
            // B rows: thread t fills weight rows t, t + 128, ...
            {
                const uint32_t base = ptx::smem_addr(sm.b + stage * Cfg::B_STAGE_BYTES);
#pragma unroll 1
                for (int b = row; b < BN; b += GATHER_THREADS) {
                    const int n = n0 + b;
                    const uint16_t* wr = kp.w + static_cast<int64_t>(n) * kp.CRS;
#pragma unroll 1
                    for (int j = 0; j < BK / 8; ++j) {
                        uint32_t packed[4];
#pragma unroll
                        for (int e = 0; e < 8; ++e) {
                            const int kk = kk0 + j * 8 + e;
                            uint32_t v = 0;
                            if (n < kp.K && kk < kp.CRS) v = __ldg(reinterpret_cast<const unsigned short*>(wr + kk));
                            if (e & 1) packed[e >> 1] |= v << 16;
                            else packed[e >> 1] = v;
                        }
                        ptx::st_shared_v4(base + sw128_offset(b, j), packed[0], packed[1], packed[2], packed[3]);
                    }
                }
            }
            ptx::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) ptx::mbar_arrive(&sm.full[stage]);
        }
    }
}

// ---------------------------------------------------------------- epilogue (warps 2..5)
// Waits (bounded) until the tile semaphore reads `split`.  One thread only.
__device__ __forceinline__ bool wait_turn(const ConvKernelParams& kp, int tile, int split,
                                          volatile uint32_t* abort_flag)
{
    const uint32_t* sem = kp.sems + tile;
    if (ptx::ld_acquire_gpu(sem) == static_cast<uint32_t>(split)) return true;
    const uint64_t t0 = ptx::clock64();
    const uint64_t limit = ptx::ns_to_cycles(kp.wait_limit_ns);
    while (ptx::ld_acquire_gpu(sem) != static_cast<uint32_t>(split)) {
        __nanosleep(32);
        if (ptx::clock64() - t0 > limit) {
            record_timeout(kp, abort_flag);
            return false;
        }
    }
    return true;
}

// Concurrent mode: waits (bounded) until split 0 of the tile has stored its part.  One thread only.
__device__ __forceinline__ bool wait_base(const ConvKernelParams& kp, int tile, volatile uint32_t* abort_flag)
{
    const uint32_t* sem = kp.sems + tile;
    if (ptx::ld_acquire_gpu(sem) != 0u) return true;
    const uint64_t t0 = ptx::clock64();
    const uint64_t limit = ptx::ns_to_cycles(kp.wait_limit_ns);
    while (ptx::ld_acquire_gpu(sem) == 0u) {
        __nanosleep(32);
        if (ptx::clock64() - t0 > limit) {
            record_timeout(kp, abort_flag);
            return false;
        }
    }
    return true;
}

// Marks this split's part of the tile done.  Ordered mode: publishes the next
// split's turn.  Concurrent mode: counts the split in; the split that completes
// the count is the last one.  The last split resets the semaphore to 0.  One
// thread only, after the CTA's writes have been fenced.
__device__ __forceinline__ void pass_turn(const ConvKernelParams& kp, const Segment& sg)
{
    if ((kp.debug_flags & 1) && sg.split == 0) return;  // test hook: never signal
    if (kp.reduce_concurrent) {
        const uint32_t before = atomicAdd(kp.sems + sg.tile, 1u);
        if (before + 1u == static_cast<uint32_t>(sg.nsplits)) atomicExch(kp.sems + sg.tile, 0u);
        return;
    }
    const uint32_t next = (sg.split + 1 == sg.nsplits) ? 0u : static_cast<uint32_t>(sg.split + 1);
    ptx::st_release_gpu(kp.sems + sg.tile, next);
}

// Finishing pass of a cut tile under the fused epilogue: the tile's complete sum
// from kp.part (read through L2), + bias, activation, conversion, store in y,
// and the part buffer reset to zero.  Same thread-to-element mapping as the
// accumulator stores.
template <int BM, int BN, int LOADER>
__device__ __forceinline__ void finish_from_part(const ConvKernelParams& kp, int m_tile, int n0, int n_end, int jbeg,
                                                 int bx_n, int bx_p, int bx_q)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int SLABS = BN / 32 / (Cfg::EPI_WARPS / 4);
    const int lane = threadIdx.x & 31;
    const int quad = (threadIdx.x >> 5) & 3;
    const int rsub = lane >> 3;
    const int chunk = lane & 7;
    uint16_t* yb = reinterpret_cast<uint16_t*>(kp.y);
    // All loads of a slab are issued before any is used: one L2 round trip per
    // slab rather than one per row.
#pragma unroll 1
    for (int sub = 0; sub < Cfg::M_SUB; ++sub) {
        const int trow0 = sub * MMA_M;
        if (kp.vec_store) {
            int mrow[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                mrow[i] = tile_row_m<BM, LOADER>(kp, m_tile, trow0 + quad * 32 + 4 * i + rsub, bx_n, bx_p, bx_q);
#pragma unroll
            for (int j = 0; j < SLABS; ++j) {
                const int col = n0 + (jbeg + j) * 32 + chunk * 4;
                if (col >= n_end) continue;
                const float4 b4 = kp.bias ? __ldg(reinterpret_cast<const float4*>(kp.bias + col)) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int h = 0; h < 8; h += 4) {  // four rows' loads in flight at a time
                    float4 v[4];
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        v[i] = mrow[h + i] >= 0
                                   ? __ldcg(reinterpret_cast<const float4*>(kp.part + static_cast<int64_t>(mrow[h + i]) * kp.ldy + col))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        if (mrow[h + i] < 0) continue;
                        const int64_t at = static_cast<int64_t>(mrow[h + i]) * kp.ldy + col;
                        __stcg(reinterpret_cast<float4*>(kp.part + at), make_float4(0.f, 0.f, 0.f, 0.f));
                        uint4 val = make_uint4(__float_as_uint(v[i].x + b4.x), __float_as_uint(v[i].y + b4.y),
                                               __float_as_uint(v[i].z + b4.z), __float_as_uint(v[i].w + b4.w));
                        if (kp.relu) val = ptx::relu4(val);
                        if (kp.out_bf16) *reinterpret_cast<uint2*>(yb + at) = ptx::pack_bf16x4(val);
                        else *reinterpret_cast<uint4*>(kp.y + at) = val;
                    }
                }
            }
        } else {
            const int m = tile_row_m<BM, LOADER>(kp, m_tile, trow0 + quad * 32 + lane, bx_n, bx_p, bx_q);
#pragma unroll
            for (int j = 0; j < SLABS; ++j) {
                const int nb = n0 + (jbeg + j) * 32;
                const int64_t at0 = static_cast<int64_t>(m < 0 ? 0 : m) * kp.ldy + nb;
                const float bias_l = (kp.bias && nb + lane < n_end) ? __ldg(kp.bias + nb + lane) : 0.0f;
#pragma unroll
                for (int h = 0; h < 32; h += 16) {  // sixteen loads in flight at a time
                    float v[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        v[e] = (m >= 0 && nb + h + e < n_end) ? __ldcg(kp.part + at0 + h + e) : 0.0f;
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const float bias = __shfl_sync(0xffffffffu, bias_l, h + e);
                        if (m < 0 || nb + h + e >= n_end) continue;
                        __stcg(kp.part + at0 + h + e, 0.0f);
                        float o = v[e] + bias;
                        if (kp.relu) o = fmaxf(o, 0.0f);
                        if (kp.out_bf16) yb[at0 + h + e] = ptx::bf16_bits(o);
                        else kp.y[at0 + h + e] = o;
                    }
                }
            }
        }
    }
}

// FUSED: the fused epilogue (ReLU, bf16 output, cut tiles through kp.part)
// compiled in; the plain instantiation carries none of its code.
template <int BM, int BN, int LOADER, bool FUSED>
__device__ void run_epilogue_impl(const ConvKernelParams& kp, const SmemView& sm, uint32_t tmem_base)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    constexpr int EPI_T = Cfg::EPI_WARPS * 32;
    // Warps of the same TMEM lane quadrant split the tile's 32-column slabs.
    constexpr int SLABS = BN / 32 / (Cfg::EPI_WARPS / 4);
    const int et = threadIdx.x - EPI_WARP0 * 32;  // 0 .. EPI_T-1
    const int ew = et >> 5;                        // epilogue warp
    const int lane = threadIdx.x & 31;
    const int quad = (threadIdx.x >> 5) & 3;  // TMEM lane quadrant this warp may access
    const int row = quad * 32 + lane;          // row of each 128-row block owned by this thread
    const int jbeg = (ew >> 2) * SLABS;        // this warp's first slab
    uint8_t* slots = sm.epi + ew * (EPI_SLOTS * EPI_SLOT_BYTES);
    int seg_idx = 0;
    uint64_t c_acc = 0, c_ld = 0, c_slot = 0, c_st = 0, c_turn = 0, c_done = 0;
    (void)c_acc; (void)c_ld; (void)c_slot; (void)c_st; (void)c_turn; (void)c_done;
    const int rsub = lane >> 3;  // vector stores: row within a group of four written per instruction
    const int chunk = lane & 7;  // vector stores: 16-byte chunk of the 128-byte row slab
    SegmentWalker walk(kp);
    Segment sg;
    while (walk.next(kp, sg)) {
        const int buf = seg_idx % Cfg::NUM_ACC;
        const uint32_t use = static_cast<uint32_t>(seg_idx / Cfg::NUM_ACC) & 1u;
        const int m_tile = sg.tile / kp.n_tiles;
        int n0, n_end, c_base_unused;
        tile_columns<BN>(kp, sg.tile, m_tile, n0, n_end, c_base_unused);
        int bx_n = 0, bx_p = 0, bx_q = 0;
        if constexpr (LOADER == LOADER_BOX) box_origin(kp, m_tile, bx_n, bx_p, bx_q);
        // Fused epilogue of a cut tile: partial sums go to kp.part, and the bias,
        // the activation and the output conversion wait for the finishing pass.
        const bool via_part = FUSED && sg.nsplits > 1;
        const bool add_bias = kp.bias != nullptr && sg.split == 0 && !via_part;
        // Bias of this warp's slabs, fetched before the accumulator wait so that
        // its latency is hidden.  Vector stores: lane holds the four columns of its
        // 16-byte chunk; row stores: lane l holds column 32*j + l.
        float4 bias4[SLABS];
        float bias_r[SLABS];
#pragma unroll
        for (int j = 0; j < SLABS; ++j) {
            const int cbase = n0 + (jbeg + j) * 32;
            bias4[j] = make_float4(0.f, 0.f, 0.f, 0.f);
            bias_r[j] = 0.f;
            if (add_bias && kp.vec_store && cbase + chunk * 4 < n_end)
                bias4[j] = __ldg(reinterpret_cast<const float4*>(kp.bias + cbase + chunk * 4));
            if (add_bias && !kp.vec_store && cbase + lane < n_end) bias_r[j] = __ldg(kp.bias + cbase + lane);
        }
        // One thread polls the accumulator barrier; the others wait at the named
        // barrier below (polling shared memory from every warp would steal issue
        // slots from the MMA warp).
        SGB_CYCLES_BEGIN(t_acc);
        if (et == 0 && !ptx::mbar_wait(&sm.acc_full[buf], use, kp.wait_limit_ns)) record_timeout(kp, sm.abort_flag);
        SGB_CYCLES_END(c_acc, t_acc);
        // One thread decides for all (including, for a later split, waiting for
        // split 0 or for its turn), so that every epilogue warp takes the same path.
        SGB_CYCLES_BEGIN(t_turn);
        ptx::named_bar_sync(1, EPI_T);
        if (et == 0) {
            bool go = *sm.abort_flag == 0u;
            if (go && sg.split > 0 && !via_part)
                go = kp.reduce_concurrent ? wait_base(kp, sg.tile, sm.abort_flag)
                                          : wait_turn(kp, sg.tile, sg.split, sm.abort_flag);
            *sm.epi_go = go ? 1u : 0u;
        }
        ptx::named_bar_sync(1, EPI_T);
        SGB_CYCLES_END(c_turn, t_turn);
        if (!*sm.epi_go) break;
        ptx::tc_fence_after();
        SGB_TRACE(kp, et == 0 && seg_idx == 0, 7);
        SGB_TRACE(kp, et == 0 && seg_idx < 4, 20 + 3 * seg_idx);  // segment: turn granted, accumulator ready

#pragma unroll 1
        for (int sub = 0; sub < Cfg::M_SUB; ++sub) {
            const uint32_t taddr = tmem_base + static_cast<uint32_t>(buf * Cfg::ACC_COLS + sub * BN) +
                                   (static_cast<uint32_t>(quad * 32) << 16);
            const int trow0 = sub * MMA_M;  // first tile row of this 128-row block
            const bool last_sub = sub == Cfg::M_SUB - 1;
            if (kp.vec_store) {
                // TMEM -> registers -> this warp's 32 x 32 swizzled staging slot ->
                // coalesced 16-byte global writes (8 lanes per 128-byte row, bias added
                // per chunk): plain stores for split 0, vector atomic adds for later
                // splits.  The writes use the load/store path, leaving the TMA unit
                // to the im2col and weight loads.
                const uint32_t saddr = ptx::smem_addr(slots);
                // Byte address of each of this lane's eight rows at the warp's first slab
                // (in the partial-sum buffer for a cut tile of a fused epilogue).
                const bool bf16_out = FUSED && kp.out_bf16 && !via_part;
                const int64_t esize = bf16_out ? 2 : 4;
                const uint64_t base = reinterpret_cast<uint64_t>(via_part ? kp.part : kp.y);
                uint64_t rowp[8];
                uint32_t row_ok = 0u;
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const int m = tile_row_m<BM, LOADER>(kp, m_tile, trow0 + quad * 32 + 4 * i + rsub, bx_n, bx_p, bx_q);
                    row_ok |= (m >= 0 ? 1u : 0u) << i;
                    rowp[i] = base + static_cast<uint64_t>(
                                         (static_cast<int64_t>(m >= 0 ? m : 0) * kp.ldy + n0 + jbeg * 32 + chunk * 4) * esize);
                }
                const int mode = bf16_out ? SLAB_BF16 : ((via_part || sg.split > 0) ? SLAB_RED : SLAB_F32);
                const bool relu = FUSED && kp.relu && !via_part;
#pragma unroll
                for (int j = 0; j < SLABS; ++j) {
                    uint32_t v[32];
                    SGB_CYCLES_BEGIN(t_ld);
                    ptx::tmem_ld_32x32b_x32(taddr + (jbeg + j) * 32, v);
                    ptx::tmem_ld_wait();
                    SGB_CYCLES_END(c_ld, t_ld);
                    if (last_sub && j == SLABS - 1) {  // accumulator drained: the MMA warp may reuse it
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&sm.acc_empty[buf]);
                    }
                    SGB_CYCLES_BEGIN(t_slot);
                    const bool col_ok = n0 + (jbeg + j) * 32 + chunk * 4 < n_end;
                    const int64_t off = static_cast<int64_t>(j) * 32 * esize;
                    if (FUSED && mode == SLAB_BF16)
                        slab_out<SLAB_BF16>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], relu);
                    else if (mode == SLAB_F32)
                        slab_out<SLAB_F32>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], relu);
                    else
                        slab_out<SLAB_RED>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], relu);
                    SGB_CYCLES_END(c_slot, t_slot);
                }
            } else {
                // K % 4 != 0: row-per-thread stores (split 0), and for later splits
                // read-add-write in turn or scalar atomic adds when concurrent.
                const int m = tile_row_m<BM, LOADER>(kp, m_tile, trow0 + row, bx_n, bx_p, bx_q);
                const bool row_ok = m >= 0;
                const bool accumulate = sg.split > 0;
                float* yrow = kp.y + static_cast<int64_t>(row_ok ? m : 0) * kp.ldy;
#pragma unroll
                for (int j = 0; j < SLABS; ++j) {
                    uint32_t v[32];
                    ptx::tmem_ld_32x32b_x32(taddr + (jbeg + j) * 32, v);
                    ptx::tmem_ld_wait();
                    if (last_sub && j == SLABS - 1) {
                        ptx::tc_fence_before();
                        ptx::mbar_arrive(&sm.acc_empty[buf]);
                    }
                    if (add_bias) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            v[e] = __float_as_uint(__uint_as_float(v[e]) + __shfl_sync(0xffffffffu, bias_r[j], e));
                    }
                    if (!row_ok) continue;
                    const int nb = n0 + (jbeg + j) * 32;
                    if (via_part) {
                        float* prow = kp.part + static_cast<int64_t>(m) * kp.ldy;
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (nb + e < n_end) atomicAdd(prow + nb + e, __uint_as_float(v[e]));
                        continue;
                    }
                    float old[32];
                    if (accumulate && !kp.reduce_concurrent) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) old[e] = nb + e < n_end ? yrow[nb + e] : 0.0f;
                    }
#pragma unroll
                    for (int e = 0; e < 32; ++e) {
                        const int n = nb + e;
                        if (n >= n_end) break;
                        float o = __uint_as_float(v[e]);
                        if (FUSED && kp.relu) o = fmaxf(o, 0.0f);
                        if (FUSED && kp.out_bf16) {  // fused epilogue: whole tiles (cut ones go through kp.part)
                            reinterpret_cast<uint16_t*>(kp.y)[static_cast<int64_t>(m) * kp.ldy + n] = ptx::bf16_bits(o);
                            continue;
                        }
                        if (accumulate && kp.reduce_concurrent) {
                            atomicAdd(yrow + n, o);
                            continue;
                        }
                        if (accumulate) o = old[e] + o;
                        yrow[n] = o;
                    }
                }
            }
        }

        if (via_part) {
            // Every thread fences its adds, then one thread counts the CTA in; the
            // CTA that completes the count (all splits' adds are then in L2) reads
            // the sums back, finishes the tile and zeroes its part of the buffer.
            __threadfence();
            ptx::named_bar_sync(1, EPI_T);
            if (et == 0) {
                const uint32_t before = atomicAdd(kp.sems + sg.tile, 1u);
                const bool last = before + 1u == static_cast<uint32_t>(sg.nsplits);
                if (last) {
                    atomicExch(kp.sems + sg.tile, 0u);
                    __threadfence();
                }
                *sm.epi_go = last ? 2u : 1u;
            }
            ptx::named_bar_sync(1, EPI_T);
            if constexpr (FUSED) {
                if (*sm.epi_go == 2u) finish_from_part<BM, BN, LOADER>(kp, m_tile, n0, n_end, jbeg, bx_n, bx_p, bx_q);
            }
        } else if (sg.nsplits > 1) {
            SGB_CYCLES_BEGIN(t_done);
            // Before the next split may read or add: split 0's stores (both modes)
            // and every split's writes in the ordered mode must be complete and
            // visible.  A later split of the concurrent mode only counts itself
            // done; nothing waits for its adds inside this launch.
            if (sg.split == 0 || !kp.reduce_concurrent) __threadfence();
            ptx::named_bar_sync(1, EPI_T);
            if (et == 0) pass_turn(kp, sg);
            SGB_CYCLES_END(c_done, t_done);
        }
        SGB_TRACE(kp, et == 0 && seg_idx < 4, 21 + 3 * seg_idx);  // segment: epilogue done
        SGB_TRACE_VALUE(kp, et == 0 && seg_idx < 4, 22 + 3 * seg_idx,
                        (static_cast<unsigned long long>(sg.kb_end - sg.kb_begin) << 16) |
                            (static_cast<unsigned long long>(sg.split) << 8) | sg.nsplits);
        ++seg_idx;
    }
    SGB_TRACE(kp, et == 0, 8);
    SGB_TRACE_VALUE(kp, et == 0, 11, c_acc);
    SGB_TRACE_VALUE(kp, et == 0, 12, c_ld);
    SGB_TRACE_VALUE(kp, et == 0, 13, c_slot);
    SGB_TRACE_VALUE(kp, et == 0, 14, c_st);
    SGB_TRACE_VALUE(kp, et == 0, 15, c_turn + (c_done << 32));
}

// ---------------------------------------------------------------- the kernel
// FUSED selects the instantiation with the fused epilogue (ReLU, bf16 output),
// so that the plain one's code and register allocation are exactly those of a
// kernel without it.
template <int BM, int BN, int LOADER, bool FUSED>
__global__ void __launch_bounds__(TileConfig<BM, BN, LOADER>::THREADS, 1)
    conv2d_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ ConvKernelParams kp)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemView sm;
    sm.a = smem;
    sm.b = smem + Cfg::STAGES * Cfg::A_STAGE_BYTES;
    sm.halo = smem + Cfg::RING_BYTES;  // halo loader: 2 buffers of kp.halo_bytes (1024-B multiples)
    const int halo_total = Cfg::HALO ? 2 * kp.halo_bytes : 0;
    sm.epi = smem + Cfg::RING_BYTES + halo_total;
    sm.full = reinterpret_cast<uint64_t*>(smem + Cfg::RING_BYTES + halo_total + Cfg::EPI_BYTES);
    sm.empty = sm.full + Cfg::STAGES;
    sm.acc_full = sm.empty + Cfg::STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.mma_done = sm.acc_empty + 2;
    sm.halo_full = sm.mma_done + 1;
    sm.halo_empty = sm.halo_full + 2;
    sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.halo_empty + 2);
    sm.abort_flag = sm.tmem_slot + 1;
    sm.epi_go = sm.tmem_slot + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    SGB_TRACE(kp, threadIdx.x == 0, 0);

    if (threadIdx.x == 0) {
        // TMA producer: one arrive (with the byte count); cp.async gather: one
        // arrive per thread (issued by its copies); scalar gather: one per warp.
        constexpr uint32_t GATHER_WARPS = GATHER_THREADS / 32;
        // Halo loader: one arrive (the weight tile's producer).
        const uint32_t full_count =
            Cfg::HALO ? 1u
            : Cfg::TMA_A ? 2u  // the activation (or output-gradient) and the weight (or im2col) producer
                                                           : (LOADER == LOADER_SCALAR ? GATHER_WARPS : 1u + GATHER_THREADS);
        for (int i = 0; i < Cfg::STAGES; ++i) {
            ptx::mbar_init(&sm.full[i], full_count);
            ptx::mbar_init(&sm.empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.acc_full[i], 1);
            ptx::mbar_init(&sm.acc_empty[i], Cfg::EPI_WARPS * 32);
        }
        ptx::mbar_init(sm.mma_done, 1);
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.halo_full[i], 1);
            ptx::mbar_init(&sm.halo_empty[i], 1);
        }
        *sm.abort_flag = 0u;
        *sm.epi_go = 0u;
        ptx::mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        if (Cfg::TMA_A || LOADER == LOADER_HYBRID) ptx::prefetch_tensormap(&tm_a);
        if (LOADER != LOADER_SCALAR) ptx::prefetch_tensormap(&tm_b);
        if constexpr (Cfg::TMA_A) prefetch_first_stages<BM, BN, LOADER>(&tm_a, &tm_b, kp);
    }
    if (warp == 1) {
        ptx::tmem_alloc(sm.tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    if (warp == 2) ptx::touch_params(&kp, static_cast<int>(sizeof(kp)));
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;
    // Everything above touches only shared memory, tensor memory, kernel
    // parameters and (by L2 prefetches) the L2 cache, so it may overlap the
    // previous kernel in the stream.  Global memory is read into the CTA or
    // written (inputs it may have written, y and the workspace it may still
    // read) only after this wait.
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    SGB_TRACE(kp, threadIdx.x == 0, 1);

    if (warp == 0) {
        if constexpr (Cfg::HALO) {
            if (lane == 0) run_halo_producer<BM, BN, LOADER>(&tm_a, &tm_b, kp, sm, 0);
        } else if constexpr (Cfg::TMA_A) {
            if (lane == 0) run_tma_producer<BM, BN, LOADER, PROD_A>(&tm_a, &tm_b, kp, sm);
        } else if constexpr (LOADER != LOADER_SCALAR) {
            if (lane == 0) run_tma_producer<BM, BN, LOADER, PROD_AB>(&tm_a, &tm_b, kp, sm);
        }
    } else if (warp == 1) {
        run_mma_issuer<BM, BN, LOADER>(kp, sm, tmem_base);
    } else if (warp < EPI_WARP0 + Cfg::EPI_WARPS) {
        run_epilogue_impl<BM, BN, LOADER, FUSED>(kp, sm, tmem_base);
    } else if (warp == WAITER_WARP) {
        run_stage_waiter<BM, BN, LOADER>(kp, sm);
    } else if (warp > WAITER_WARP) {
        if constexpr (Cfg::HALO) {  // warps 11 .. 13: weight tiles of ring slots 1 .. 3 (mod 4)
            if (lane == 0) run_halo_producer<BM, BN, LOADER>(&tm_a, &tm_b, kp, sm, warp - WAITER_WARP);
        } else if constexpr (Cfg::TMA_A) {  // warp 11: the weight tiles
            if (lane == 0) run_tma_producer<BM, BN, LOADER, PROD_B>(&tm_a, &tm_b, kp, sm);
        }
    } else {
        if constexpr (LOADER == LOADER_CPASYNC || LOADER == LOADER_HYBRID) run_gather_cpasync<BM, BN, LOADER>(kp, sm);
        if constexpr (LOADER == LOADER_SCALAR) run_gather_scalar<BM, BN, LOADER>(kp, sm);
        SGB_TRACE(kp, threadIdx.x == GATHER_WARP0 * 32, 9);
    }

    ptx::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc(tmem_base, Cfg::TMEM_COLS);
    }
    SGB_TRACE(kp, threadIdx.x == 0, 10);
}

// Overlap of consecutive launches (programmatic dependent launch) is on unless
// the environment sets CONV2D_NO_PDL=1.
inline bool pdl_enabled()
{
    static const bool on = [] {
        const char* v = std::getenv("CONV2D_NO_PDL");
        return !(v && v[0] == '1');
    }();
    return on;
}

// Dynamic shared memory of one CTA: the configuration's fixed part plus, for
// the halo loader, its two halo buffers.
template <int BM, int BN, int LOADER>
inline int conv2d_tc_smem_bytes(int halo_bytes)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    return Cfg::SMEM_BYTES + (Cfg::HALO ? 2 * halo_bytes : 0);
}

// Host-side launcher for one instantiation; explicitly instantiated in one
// translation unit per tile width so that the variants compile in parallel.
template <int BM, int BN, int LOADER>
cudaError_t launch_conv2d_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const ConvKernelParams& kp, int grid,
                             cudaStream_t stream)
{
    using Cfg = TileConfig<BM, BN, LOADER>;
    const int smem_bytes = conv2d_tc_smem_bytes<BM, BN, LOADER>(kp.halo_bytes);
    if (smem_bytes > kMaxSmemBytes) return cudaErrorInvalidValue;
    // The gradients have no fused epilogue: one instantiation.
    constexpr bool kHasFused = LOADER != LOADER_WGRAD && LOADER != LOADER_DGRAD;
    const bool fused = kHasFused && (kp.relu | kp.out_bf16) != 0;
    auto kern = fused ? conv2d_fwd_tc_kernel<BM, BN, LOADER, kHasFused> : conv2d_fwd_tc_kernel<BM, BN, LOADER, false>;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    // The dynamic shared-memory opt-in is per device and instantiation; remember which have it.
    static unsigned long long configured[2] = {0ull, 0ull};
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(__atomic_load_n(&configured[fused], __ATOMIC_ACQUIRE) & bit)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   Cfg::HALO ? kMaxSmemBytes : Cfg::SMEM_BYTES);
        if (err != cudaSuccess) return err;
        if (bit) __atomic_fetch_or(&configured[fused], bit, __ATOMIC_RELEASE);
    }
    // Programmatic stream serialization: this launch may start while the
    // previous kernel in the stream drains; the kernel waits for it (see
    // grid_dependency_wait) before touching global memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(Cfg::THREADS);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_a, tm_b, kp);
}

#define SGB_LAUNCH_SIG(BM_, BN_, L_)                                                                        \
    cudaError_t launch_conv2d_tc<BM_, BN_, L_>(const CUtensorMap&, const CUtensorMap&, const ConvKernelParams&, \
                                               int, cudaStream_t)

// Every loader with 128-pixel tiles (the halo loader's only size), the TMA loader with 256-pixel tiles, and
// the box loader with 256-pixel tiles where two k-blocks of both operands fit
// a stage twice (BN <= 128).
#define SGB_INSTANTIATE_CONV2D(BN_)                    \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_TMA);     \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_CPASYNC); \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_SCALAR);  \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_HYBRID);  \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_BOX);     \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_HALO);    \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_WGRAD);   \
    template SGB_LAUNCH_SIG(128, BN_, LOADER_DGRAD);   \
    template SGB_LAUNCH_SIG(256, BN_, LOADER_TMA);
#define SGB_INSTANTIATE_CONV2D_BOX256(BN_) template SGB_LAUNCH_SIG(256, BN_, LOADER_BOX);

// Declarations of the instantiations that live in other translation units.
#define SGB_DECLARE_CONV2D(BN_)                               \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_TMA);     \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_CPASYNC); \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_SCALAR);  \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_HYBRID);  \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_BOX);     \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_HALO);    \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_WGRAD);   \
    extern template SGB_LAUNCH_SIG(128, BN_, LOADER_DGRAD);   \
    extern template SGB_LAUNCH_SIG(256, BN_, LOADER_TMA);
#define SGB_DECLARE_CONV2D_BOX256(BN_) extern template SGB_LAUNCH_SIG(256, BN_, LOADER_BOX);

}  // namespace sgb
