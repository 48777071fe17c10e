// Implicit-GEMM 2-D convolution forward on CTA pairs (tcgen05.mma.cta_group::2).
//
// The GEMM view is the one-CTA kernel's (burn PR #2287 "Introduce autotuning to
// conv2d ...", Changes; burn PR #2545 "[Optimization] Implicit gemm rewrite",
// Changes): rows m = (n*P + p)*Q + q are output pixels, columns are output
// channels, the reduction index is kk = (r*S + s)*Cg + c (Cg = C / groups; a
// column block stays inside one group), A is the im2col matrix gathered tile by
// tile by TMA in im2col mode and B the KRSC weight viewed as [K][Cg*R*S].
//
// A tile is 256 output pixels x BN output channels, computed by a cluster of
// two CTAs on two SMs.  Each CTA loads into its own shared memory the im2col
// rows of its 128 pixels and BN/2 of the weight rows; one thread of the even
// CTA (the leader) issues 256 x BN x 16 MMAs that read A rows 0..127 and the
// first half of B from the leader and the rest from the same shared-memory
// addresses in the peer, and accumulate rows 0..127 in the leader's tensor
// memory and rows 128..255 in the peer's.  Per SM this halves the weight bytes
// moved per MMA compared with a 128-pixel tile of the same width.
//
// A pipeline stage holds two 64-wide k-blocks: per CTA, two im2col loads of
// 128 pixel rows x 64 channels and one 3-D box of BN/2 weight rows x 2
// k-blocks, so that one stage carries 1024 MMA cycles of work per SM at
// BN = 256.  A producer thread spends a roughly fixed ~0.2 us per ring stage
// (barrier wait, expect, issue) whatever the stage's size, so fewer, larger
// stages keep the producer ahead of the tensor cores.  Both CTAs' loads of a
// stage complete on the leader's full barrier (the leader's producer expects the
// bytes of both); the leader's MMA commit releases the stage in both CTAs at
// once (multicast), and the accumulator-ready signal likewise.  Each CTA's
// epilogue drains its own 128 accumulator rows and tells the leader's MMA warp
// through a remote arrive on the leader's barrier.
//
// Work split: units are (tile, stage) pairs numbered tile-major; pair c of G
// takes units [c*U/G, (c+1)*U/G) (stream-K, as in the one-CTA kernel), so all
// SM pairs get the same number of MMAs.  A tile cut between pairs is reduced in
// place in y, each 128-row half with its own semaphore (NVIDIA/Fuser issue #1316
// "Split-K matmul is slow even for few partitions", Eliminating the workspace):
// split 0 stores, later splits add; the ranges are rotated so that split 0 is
// always computed first (see PairWalker and the epilogue).
//
// Warp roles, the same in both CTAs (the MMA issuer and the stage waiter are
// idle in the peer):
//   warp 0      TMA producer (one thread) of this CTA's im2col rows;
//   warp 1      tensor-memory allocation for the pair; in the leader the MMA issuer;
//   warps 2..9  epilogue: TMEM -> registers (+ bias) -> swizzled staging -> 16-byte stores;
//   warp 10     in the leader, the stage waiter (waits for each stage's full
//               barrier and releases the MMA warp by named barrier, so the MMA
//               thread never polls shared memory between its MMAs);
//   warp 11     TMA producer (one thread) of this CTA's weight rows.
//
// Every wait is bounded; a wait that runs out records CONV2D_ERR_TIMEOUT, flags
// both CTAs of the pair, and the pair runs its loops to the end without
// issuing or storing.
#pragma once

#include "conv2d_kernel.cuh"

namespace sgb {

constexpr int PAIR_ROWS = 128;  // output pixels (GEMM rows) each CTA of the pair holds
constexpr int PAIR_TILE_M = 2 * PAIR_ROWS;
constexpr int EPI_GRP_BAR0 = 12;      // named barriers of the epilogue's two column groups (TMA stores)
constexpr int EPI_BOX_ROWS = 64;      // rows of one staged y box
constexpr int EPI_BOX_BYTES = EPI_BOX_ROWS * 128;
// 64-wide k-blocks per pipeline stage (KBS): 2 gives three 64 KB stages at BN =
// 256 with one producer thread per operand; 1 gives six 32 KB stages with two
// producer threads per operand taking alternate stages.
constexpr int PAIR_KBS_MAX = 2;

template <int BN, int KBS>
struct PairConfig {
    static_assert(BN == 64 || BN == 128 || BN == 256, "pair tiles are 256 pixels x 64, 128 or 256 channels");
    static_assert(KBS == 1 || KBS == 2, "one or two k-blocks per stage");
    static constexpr int B_ROWS = BN / 2;                  // weight rows each CTA holds
    static constexpr int A_KB = PAIR_ROWS * BK * 2;        // one k-block of this CTA's A rows: 16 KB
    static constexpr int B_KB = B_ROWS * BK * 2;           // one k-block of this CTA's B rows
    static constexpr int A_STAGE = KBS * A_KB;
    static constexpr int B_STAGE = KBS * B_KB;
    static constexpr int NPROD = KBS == 1 ? 2 : 1;  // producer threads per operand
    static constexpr int STAGE = A_STAGE + B_STAGE;
    static constexpr int STAGES = 196608 / STAGE > 8 ? 8 : 196608 / STAGE;  // 3 (BN 256), 4 (128, 64)
    static_assert(STAGES >= 3, "the ring needs at least three stages");
    static_assert(STAGES % NPROD == 0, "each producer owns whole ring slots");
    static constexpr int RING = STAGES * STAGE;
    static constexpr int EPI_WARPS = 8;
    static constexpr int EPI_T = EPI_WARPS * 32;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_SLOT_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 5) * 8 + 16;
    static constexpr int SMEM_BYTES = RING + EPI_BYTES + BAR_BYTES + 1024;  // + alignment slack
    static_assert(SMEM_BYTES <= kMaxSmemBytes, "exceeds the per-block shared-memory limit");
    static constexpr uint32_t TMEM_COLS = 2 * BN;  // two accumulators of BN fp32 columns (128 lanes)
    static constexpr int THREADS = (WAITER_WARP + 2 * NPROD) * 32;  // warps 0 .. 11 (13 with two producers per operand)
    // Both operands K-major bf16, fp32 accumulator, M = 256 across the pair.
    static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(PAIR_TILE_M, BN);
    // Accumulator-empty arrivals: every epilogue warp of both CTAs, once per segment.
    static constexpr uint32_t ACC_EMPTY_COUNT = 2 * EPI_WARPS;
};

struct PairSmem {
    uint8_t* a;          // STAGES x (2 k-blocks x 128 rows x 128 B)
    uint8_t* b;          // STAGES x (2 k-blocks x BN/2 rows x 128 B)
    uint8_t* epi;        // EPI_WARPS staging slots
    uint64_t* full;      // STAGES (used in the leader)
    uint64_t* empty;     // STAGES (both)
    uint64_t* acc_full;  // 2 (both)
    uint64_t* acc_empty; // 2 (leader)
    uint64_t* mma_done;  // 1 (leader)
    uint8_t* halo;         // halo loader: 2 buffers of kp.halo_bytes
    uint64_t* halo_full;   // 2 (leader): both CTAs' halo landed
    uint64_t* halo_empty;  // 2 (both): no MMA reads the buffer any more
    uint32_t* tmem_slot;
    volatile uint32_t* abort_flag;
    volatile uint32_t* epi_go;
};

// Records a timeout and flags both CTAs of the pair.
__device__ __forceinline__ void pair_record_timeout(const ConvKernelParams& kp, const PairSmem& sm, uint32_t rank)
{
    *sm.abort_flag = 1u;
    ptx::st_cluster_u32(ptx::mapa_shared(ptx::smem_addr(const_cast<uint32_t*>(sm.abort_flag)), rank ^ 1u), 1u);
    ptx::grid_dependency_wait();  // the status word is global memory (a no-op once waited)
    if (kp.status) atomicMax(kp.status, STATUS_TIMEOUT);
}

// This pair's segments, from the end of its unit range to the start.  kp.grid
// is the number of pairs and kp.num_kb the number of stages per tile.
//
// The units (tile, stage), numbered tile-major, are split into equal ranges
// along an axis rotated by d = kp.unit_offset: pair c takes the units
// [floor(c*U/G) + d, floor((c+1)*U/G) + d), the ones at U and above standing
// for units 0 .. d-1 (the first d stages of tile 0, whose other stages open
// pair 0's range).  The host picks d so that no range starts on a tile
// boundary: then split 0 of a cut tile -- the tile's first stages, where a
// range starts inside the tile -- is the highest segment of its pair's range
// and is computed first, so its stores are done long before the tile's later
// splits add to them, and no pair holds a split 0 as its only segment.
//
// All arithmetic is 32-bit and every division goes through a FastDiv: the host
// admits only plans with (units + d + 1) * (grid + 1) < 2^31.
struct PairWalker {
    uint32_t lo, cur, nkb, grid, units, off, tiles;
    int pair;
    __device__ __forceinline__ PairWalker(const ConvKernelParams& kp, int pair_idx)
    {
        pair = pair_idx;
        units = static_cast<uint32_t>(kp.units);
        grid = static_cast<uint32_t>(kp.grid);
        nkb = static_cast<uint32_t>(kp.num_kb);
        off = static_cast<uint32_t>(kp.unit_offset);
        tiles = units / nkb;
        lo = kp.fd_grid.div(static_cast<uint32_t>(pair) * units) + off;
        cur = kp.fd_grid.div((static_cast<uint32_t>(pair) + 1u) * units) + off;
    }
    // The pair whose range holds unit e of the rotated axis (off <= e < units + off).
    __device__ __forceinline__ uint32_t pair_of(const ConvKernelParams& kp, uint32_t e) const
    {
        const uint32_t u = e - off;
        return kp.fd_units.div((u + 1u) * grid + units - 1u) - 1u;
    }
    __device__ __forceinline__ bool next(const ConvKernelParams& kp, Segment& sg)
    {
        if (cur <= lo) return false;
        const uint32_t te = kp.fd_nkb.div(cur - 1u);  // tile index on the rotated axis
        const uint32_t base = te * nkb;
        const uint32_t seg_lo = lo > base ? lo : base;
        sg.tile = static_cast<int>(te < tiles ? te : te - tiles);
        sg.kb_begin = static_cast<int>(seg_lo - base);
        sg.kb_end = static_cast<int>(cur - base);
        if (off == 0u) {
            const uint32_t first = pair_of(kp, base);
            const uint32_t last = pair_of(kp, base + nkb - 1u);
            sg.split = pair - static_cast<int>(first);
            sg.nsplits = static_cast<int>(last - first + 1u);
        } else {
            // Tile 0 is the only tile that straddles the rotation: its stages 0 .. off-1
            // are the top of the last pair's range, the rest open pair 0's.
            const bool wrapped_tile = te == 0u || te == tiles;
            if (!wrapped_tile) {
                const uint32_t first = pair_of(kp, base);
                const uint32_t last = pair_of(kp, base + nkb - 1u);
                sg.split = pair - static_cast<int>(first);
                sg.nsplits = static_cast<int>(last - first + 1u);
            } else {
                const uint32_t last = pair_of(kp, nkb - 1u);  // the last pair holding part of stages off .. nkb-1
                sg.nsplits = static_cast<int>(last) + 2;
                sg.split = te == tiles ? 0 : pair + 1;
            }
        }
        cur = seg_lo;
        return true;
    }
};

// Tile row-block and column-block of a tile index.
__device__ __forceinline__ void pair_tile_coords(const ConvKernelParams& kp, int tile, int& m_tile, int& n_tile)
{
    m_tile = static_cast<int>(kp.fd_ntiles.div(static_cast<uint32_t>(tile)));
    n_tile = tile - m_tile * kp.n_tiles;
}

// Reduction cursor: filter tap (r, s) and channel c of a 64-wide k-block, stepped without divisions.
struct PairCursor {
    int r, s, c;
    __device__ __forceinline__ void at(const ConvKernelParams& kp, int kb)
    {
        const int kk = kb * BK;
        const int rs = static_cast<int>(kp.fd_c.div(static_cast<uint32_t>(kk)));  // fd_c divides by Cg
        c = kk - rs * kp.Cg;
        r = static_cast<int>(kp.fd_s.div(static_cast<uint32_t>(rs)));
        s = rs - r * kp.S;
    }
    __device__ __forceinline__ void step(const ConvKernelParams& kp)
    {
        c += BK;
        if (c >= kp.Cg) {
            c = 0;
            if (++s == kp.S) {
                s = 0;
                ++r;
            }
        }
    }
};

// Output channels of column block n_tile: block nb of group g = n_tile / ntpg
// covers channels g*Kg + nb*BN .. up to the group's end; its reduction reads the
// group's input channels from g*Cg.  One group: n0 = n_tile*BN, n_end <= K.
template <int BN>
__device__ __forceinline__ void pair_columns(const ConvKernelParams& kp, int n_tile, int& n0, int& n_end, int& c_base)
{
    const int g = n_tile / kp.ntpg;
    n0 = g * kp.Kg + (n_tile - g * kp.ntpg) * BN;
    const int g_end = (g + 1) * kp.Kg;
    n_end = n0 + BN < g_end ? n0 + BN : g_end;
    c_base = g * kp.Cg;
}

// Window origin of this CTA's first pixel in tile row-block m_tile (pixels
// past the output decode to images >= N, which the TMA zero-fills).
__device__ __forceinline__ void pair_origin(const ConvKernelParams& kp, int m_tile, uint32_t rank, int& n_img,
                                            int& w_org, int& h_org)
{
    const uint32_t m = static_cast<uint32_t>(m_tile * PAIR_TILE_M + static_cast<int>(rank) * PAIR_ROWS);
    n_img = static_cast<int>(kp.fd_pq.div(m));
    const uint32_t rem = m - static_cast<uint32_t>(n_img) * kp.fd_pq.d;
    const int p0 = static_cast<int>(kp.fd_q.div(rem));
    const int q0 = static_cast<int>(rem) - p0 * kp.Q;
    w_org = q0 * kp.sw - kp.pw;
    h_org = p0 * kp.sh - kp.ph;
}

// ---------------------------------------------------------------- producers (warps 0 and 11, one thread each, both CTAs)
// The TMA unit of an SM takes ~0.1 us per operation and ~0.17 us per ring
// stage of barrier traffic on the issuing thread, whatever the bytes; the
// activation loads (two im2col operations) and the weight load (one 3-D box)
// of a stage are therefore issued by two threads in different warps, each
// keeping its own pace ahead of the tensor cores.  Each operand of each slot
// has one issuer, loading its uses in order.
enum PairOperand : int { PAIR_A = 0, PAIR_B = 1 };

template <int BN, int KBS, int OP>
__device__ void pair_producer(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const ConvKernelParams& kp,
                              const PairSmem& sm, uint32_t rank, int pair, int role)
{
    using Cfg = PairConfig<BN, KBS>;
    constexpr int STAGES = Cfg::STAGES;
    const int kb_total = kp.CRS / BK;
    const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(sm.full), 0u);  // the leader's full[0]
    int it = 0;  // stages issued (all segments)
    bool ok = true;
    bool released = false;  // past the grid-dependency wait
    PairWalker walk(kp, pair);
    Segment sg;
    while (ok && walk.next(kp, sg)) {
        int m_tile, n_tile;
        pair_tile_coords(kp, sg.tile, m_tile, n_tile);
        int n_img = 0, w_org = 0, h_org = 0;
        if (OP == PAIR_A) pair_origin(kp, m_tile, rank, n_img, w_org, h_org);
        int n0, n_end, c_base;
        pair_columns<BN>(kp, n_tile, n0, n_end, c_base);
        const int b_row = n0 + static_cast<int>(rank) * Cfg::B_ROWS;
        PairCursor cur;
        if (OP == PAIR_A) cur.at(kp, sg.kb_begin * KBS);
        for (int st = sg.kb_begin; st < sg.kb_end; ++st, ++it) {
            const int slot = it % STAGES;
            const int nkb = kb_total - st * KBS < KBS ? kb_total - st * KBS : KBS;
            if (slot % Cfg::NPROD != role) {  // another producer's slot: only keep the cursor in step
                if (OP == PAIR_A)
                    for (int j = 0; j < nkb; ++j) cur.step(kp);
                continue;
            }
            if (*sm.abort_flag) { ok = false; break; }
            if (!ptx::mbar_wait_spin(&sm.empty[slot], (static_cast<uint32_t>(it / STAGES) & 1u) ^ 1u, kp.wait_limit_ns)) {
                pair_record_timeout(kp, sm, rank);
                ok = false;
                break;
            }
            const uint32_t bar = full0 + static_cast<uint32_t>(slot) * 8u;
            if (!released) {  // everything before this point reads only parameters and shared memory
                ptx::grid_dependency_wait();
                released = true;
                SGB_TRACE(kp, threadIdx.x == 0, 1);
            }
            if (OP == PAIR_A) {
                // The leader expects the activation bytes of both CTAs.
                if (rank == 0) ptx::mbar_arrive_expect_tx(&sm.full[slot], 2u * static_cast<uint32_t>(nkb * Cfg::A_KB));
                uint8_t* a_dst = sm.a + slot * Cfg::A_STAGE;
                for (int j = 0; j < nkb; ++j) {
                    ptx::tma_load_im2col_4d_pair(a_dst + j * Cfg::A_KB, tm_a, bar, c_base + cur.c, w_org, h_org, n_img,
                                                 static_cast<uint16_t>(cur.s * kp.dw), static_cast<uint16_t>(cur.r * kp.dh));
                    cur.step(kp);
                }
                SGB_PAIR_MARK(kp, it, static_cast<int>(rank));
            } else {
                // The weight box always counts both k-blocks (one past the reduction is zero-filled).
                if (rank == 0) ptx::mbar_arrive_expect_tx(&sm.full[slot], 2u * static_cast<uint32_t>(Cfg::B_STAGE));
                ptx::tma_load_3d_pair(sm.b + slot * Cfg::B_STAGE, tm_b, bar, 0, b_row, st * KBS);
                SGB_PAIR_MARK(kp, it, 5 + static_cast<int>(rank));
            }
        }
    }
    // Drain: the last load of each slot has been consumed (so it landed) once the
    // MMA's release of that use arrives on this CTA's empty barrier.
    for (int i = it > STAGES ? it - STAGES : 0; i < it; ++i)
        if ((i % STAGES) % Cfg::NPROD == role)
            ptx::mbar_wait(&sm.empty[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u, kp.wait_limit_ns);
}

// ---------------------------------------------------------------- stage waiter (warp 10, leader)
template <int BN, int KBS>
__device__ void pair_waiter(const ConvKernelParams& kp, const PairSmem& sm, int pair)
{
    using Cfg = PairConfig<BN, KBS>;
    constexpr int STAGES = Cfg::STAGES;
    const int lane = threadIdx.x & 31;
    bool waiting = true;
    int it = 0;
    PairWalker walk(kp, pair);
    Segment sg;
    while (walk.next(kp, sg)) {
        for (int st = sg.kb_begin; st < sg.kb_end; ++st, ++it) {
            const int slot = it % STAGES;
            const uint32_t use = static_cast<uint32_t>(it / STAGES);
            if (lane == 0) {
                if (waiting && (*sm.abort_flag || !ptx::mbar_wait_spin(&sm.full[slot], use & 1u, kp.wait_limit_ns))) {
                    pair_record_timeout(kp, sm, 0u);
                    waiting = false;
                }
                // After a timeout: pace the MMA warp by its own release of the previous use.
                if (!waiting && use > 0)
                    for (int t = 0; t < 16 && !ptx::mbar_wait(&sm.empty[slot], (use - 1u) & 1u, kp.wait_limit_ns); ++t) {
                    }
                SGB_PAIR_MARK(kp, it, 2);
            }
            __syncwarp();
            ptx::named_bar_arrive(STAGE_BAR0 + slot, 64);
        }
    }
}

// ---------------------------------------------------------------- MMA issuer (warp 1, leader)
template <int BN, int KBS>
__device__ void pair_mma(const ConvKernelParams& kp, const PairSmem& sm, uint32_t tmem_base, int pair)
{
    using Cfg = PairConfig<BN, KBS>;
    constexpr int STAGES = Cfg::STAGES;
    const int lane = threadIdx.x & 31;
    const int kb_total = kp.CRS / BK;
    const uint64_t a_desc0 = ptx::sw128_kmajor_desc(ptx::smem_addr(sm.a));
    const uint64_t b_desc0 = ptx::sw128_kmajor_desc(ptx::smem_addr(sm.b));
    int it = 0, seg_idx = 0;
    bool issue = true;
    PairWalker walk(kp, pair);
    Segment sg;
    while (walk.next(kp, sg)) {
        const int buf = seg_idx & 1;
        const uint32_t use = static_cast<uint32_t>(seg_idx >> 1) & 1u;
        // Both CTAs' epilogues must have drained this accumulator's previous segment.
        if (lane == 0 && issue) {
            if (*sm.abort_flag || !ptx::mbar_wait(&sm.acc_empty[buf], use ^ 1u, kp.wait_limit_ns)) {
                pair_record_timeout(kp, sm, 0u);
                issue = false;
            }
        }
        __syncwarp();
        ptx::tc_fence_after();
        const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(buf * BN);
        // The whole warp runs the stage loop (uniform control flow, no shared-memory
        // access between MMAs: such an access would wait for the queued MMAs to
        // drain); one elected lane issues each MMA and commit.
        const bool go = __shfl_sync(0xffffffffu, issue ? 1 : 0, 0) != 0;
        for (int st = sg.kb_begin; st < sg.kb_end; ++st, ++it) {
            const int slot = it % STAGES;
            ptx::named_bar_sync(STAGE_BAR0 + slot, 64);
            ptx::tc_fence_after();
            if (lane == 0) SGB_PAIR_MARK(kp, it, 3);
            if (go) {
                const int nkb = kb_total - st * KBS < KBS ? kb_total - st * KBS : KBS;
                const uint64_t ad = a_desc0 + static_cast<uint64_t>((slot * Cfg::A_STAGE) >> 4);
                const uint64_t bd = b_desc0 + static_cast<uint64_t>((slot * Cfg::B_STAGE) >> 4);
#pragma unroll
                for (int j = 0; j < KBS; ++j) {
                    if (j < nkb) {
                        ptx::mma_bf16_pair_elect_kb(tmem_d, ad + static_cast<uint64_t>((j * Cfg::A_KB) >> 4),
                                                    bd + static_cast<uint64_t>((j * Cfg::B_KB) >> 4), Cfg::IDESC,
                                                    (st > sg.kb_begin || j > 0) ? 1u : 0u);
                    }
                }
            }
            ptx::mma_commit_pair_elect(&sm.empty[slot], 0x3);  // every stage, issuing or not
            if (lane == 0) SGB_PAIR_MARK(kp, it, 4);
        }
        ptx::mma_commit_pair_elect(&sm.acc_full[buf], 0x3);
        __syncwarp();
        ++seg_idx;
    }
    // No MMA may be in flight when the pair reaches its teardown.
    ptx::mma_commit_pair_elect(sm.mma_done, 0x1);  // the lane that issued the MMAs
    if (lane == 0) ptx::mbar_wait(sm.mma_done, 0u, kp.wait_limit_ns);
    __syncwarp();
}

// ---------------------------------------------------------------- epilogue (warps 2..9, both CTAs)
// Cut tiles are reduced in place in y (NVIDIA/Fuser issue #1316, Eliminating
// the workspace), each 128-row half on its own semaphore: split 0 stores its
// partial sums with the bias and publishes; in the concurrent mode every later
// split waits only for that, adds with vector atomic adds and counts itself
// in (the last resets the semaphore to 0); in the ordered mode split j waits
// for the value j, adds, fences and publishes j + 1 (the last resets), so the
// adds land in k order: bitwise reproducible.  The rotated work split makes
// split 0 the first segment its pair computes (PairWalker), so its stores are
// complete long before a later split asks.
//
// Semaphore of one 128-row half of a tile: [row half][column block].
__device__ __forceinline__ int pair_sem_index(const ConvKernelParams& kp, int m_tile, uint32_t rank, int n_tile)
{
    return (m_tile * 2 + static_cast<int>(rank)) * kp.n_tiles + n_tile;
}

__device__ __forceinline__ void pair_pass_turn(const ConvKernelParams& kp, int sem, const Segment& sg)
{
    if ((kp.debug_flags & 1) && sg.split == 0) return;  // test hook: never signal
    if (kp.reduce_concurrent) {
        const uint32_t before = atomicAdd(kp.sems + sem, 1u);
        if (before + 1u == static_cast<uint32_t>(sg.nsplits)) atomicExch(kp.sems + sem, 0u);
        return;
    }
    const uint32_t next = (sg.split + 1 == sg.nsplits) ? 0u : static_cast<uint32_t>(sg.split + 1);
    ptx::st_release_gpu(kp.sems + sem, next);
}

// The output rows of this CTA's half of a tile.  im2col loader: GEMM rows
// m_tile*256 + rank*128 + r.  Halo loader: virtual pixels j0 + r of image
// 2*i + rank, where row-block m_tile = i*tpi + b starts at j0 = 128*b; virtual
// pixel j = p*wv + v is output pixel (p, v) when v < Q.
template <bool HALO>
struct PairRows {
    int base;   // first GEMM row (im2col) or first virtual pixel (halo)
    int n_img;  // halo: the image
    bool any;   // the half holds at least one output row
    __device__ __forceinline__ PairRows(const ConvKernelParams& kp, int m_tile, uint32_t rank)
    {
        if (HALO) {
            const int i = static_cast<int>(kp.fd_tpi.div(static_cast<uint32_t>(m_tile)));
            base = (m_tile - i * kp.tpi) * PAIR_ROWS;
            n_img = 2 * i + static_cast<int>(rank);
            any = n_img < kp.N;
        } else {
            base = m_tile * PAIR_TILE_M + static_cast<int>(rank) * PAIR_ROWS;
            n_img = 0;
            any = base < kp.M;
        }
    }
    // GEMM row (output pixel) of row r of the half, or -1.
    __device__ __forceinline__ int m(const ConvKernelParams& kp, int r) const
    {
        if (HALO) {
            const int j = base + r;
            if (j >= kp.vp) return -1;
            const int p = static_cast<int>(kp.fd_wv.div(static_cast<uint32_t>(j)));
            const int q = j - p * kp.wv;
            if (q >= kp.Q || n_img >= kp.N) return -1;
            return (n_img * kp.P + p) * kp.Q + q;
        }
        const int mm = base + r;
        return mm < kp.M ? mm : -1;
    }
};

// The output rows of a CTA's half tile are consecutive GEMM rows [m_a, m_a + cnt):
// im2col loader, rows base .. base + 127 clipped to M; halo loader, the valid
// virtual pixels of the row-block, which are consecutive output pixels of one
// image once the junk columns (q >= Q) are dropped.  cnt = 0 when there are none.
template <bool HALO>
__device__ __forceinline__ void pair_row_span(const ConvKernelParams& kp, const PairRows<HALO>& rows, int& m_a,
                                              int& cnt)
{
    m_a = 0;
    cnt = 0;
    if (!HALO) {
        m_a = rows.base;
        const int left = kp.M - rows.base;
        cnt = left < PAIR_ROWS ? (left > 0 ? left : 0) : PAIR_ROWS;
        return;
    }
    if (rows.n_img >= kp.N) return;
    const int j_first = rows.base;
    const int j_last = rows.base + PAIR_ROWS - 1 < kp.vp - 1 ? rows.base + PAIR_ROWS - 1 : kp.vp - 1;
    if (j_first > j_last) return;
    int p0 = static_cast<int>(kp.fd_wv.div(static_cast<uint32_t>(j_first)));
    int v0 = j_first - p0 * kp.wv;
    if (v0 >= kp.Q) {  // starts in a junk column: the next row's first pixel
        ++p0;
        v0 = 0;
    }
    const int p1 = static_cast<int>(kp.fd_wv.div(static_cast<uint32_t>(j_last)));
    int v1 = j_last - p1 * kp.wv;
    if (v1 >= kp.Q) v1 = kp.Q - 1;  // ends in a junk column: the row's last pixel
    const int img = rows.n_img * kp.P * kp.Q;
    m_a = img + p0 * kp.Q + v0;
    const int m_last = img + p1 * kp.Q + v1;
    cnt = m_last >= m_a ? m_last - m_a + 1 : 0;
}

// Stages one 32-column slab row (this thread's accumulator row, bias and ReLU
// applied) into row d of a 64-row staging box at `box` (1024-byte aligned), in
// the 128-byte swizzle the y tensor map expects.
__device__ __forceinline__ void stage_row(uint32_t box, int d, const uint32_t (&v)[32])
{
    const uint32_t rowb = box + static_cast<uint32_t>(d) * 128u;
#pragma unroll
    for (int c = 0; c < 8; ++c)
        ptx::st_shared_v4(rowb + static_cast<uint32_t>((c ^ (d & 7)) << 4), v[4 * c], v[4 * c + 1], v[4 * c + 2],
                          v[4 * c + 3]);
}

template <int BN, bool FUSED, bool HALO>
__device__ void pair_epilogue(const ConvKernelParams& kp, const PairSmem& sm, uint32_t tmem_base, uint32_t rank,
                              int pair)
{
    using Cfg = PairConfig<BN, 1>;  // the epilogue does not depend on the stage depth
    constexpr int SLABS = BN / 64;  // 32-column slabs per warp: two warps share each lane quadrant
    const int et = threadIdx.x - EPI_WARP0 * 32;
    const int ew = et >> 5;
    const int lane = threadIdx.x & 31;
    const int quad = (threadIdx.x >> 5) & 3;  // the TMEM lane quadrant this warp may read
    const int jbeg = (ew >> 2) * SLABS;
    const int rsub = lane >> 3;
    const int chunk = lane & 7;
    const uint32_t saddr = ptx::smem_addr(sm.epi + ew * EPI_SLOT_BYTES);
    const uint32_t acc_empty0 = ptx::mapa_shared(ptx::smem_addr(sm.acc_empty), 0u);  // the leader's
    // TMA stores: warps 2..5 and 6..9 form two column groups; each group stages a
    // slab's 128 rows in two 64-row boxes (its four warps' 4 KB slots) that one
    // thread of the group hands to the TMA unit.
    const int grp = ew >> 2;
    const bool issuer = (ew & 3) == 0 && lane == 0;
    const uint32_t box_a = ptx::smem_addr(sm.epi) + static_cast<uint32_t>(grp * 2 * EPI_BOX_BYTES);
    const uint32_t box_b = box_a + EPI_BOX_BYTES;
    const int trow = quad * 32 + lane;  // this thread's accumulator row
    bool tma_used = false;
    int seg_idx = 0;
    PairWalker walk(kp, pair);
    Segment sg;
    while (walk.next(kp, sg)) {
        const int buf = seg_idx & 1;
        const uint32_t use = static_cast<uint32_t>(seg_idx >> 1) & 1u;
        int m_tile, n_tile;
        pair_tile_coords(kp, sg.tile, m_tile, n_tile);
        const PairRows<HALO> rows(kp, m_tile, rank);
        const bool has_rows = rows.any;  // a half past the output stores nothing and takes no turn
        int n0, n_end, c_base_unused;
        pair_columns<BN>(kp, n_tile, n0, n_end, c_base_unused);
        const int sem = pair_sem_index(kp, m_tile, rank, n_tile);
        const bool cut = sg.nsplits > 1;
        const bool add_bias = kp.bias != nullptr && sg.split == 0;
        if (seg_idx == 0) ptx::grid_dependency_wait();  // bias and output are global memory
        float4 bias4[SLABS];
#pragma unroll
        for (int j = 0; j < SLABS; ++j) {
            const int col = n0 + (jbeg + j) * 32 + chunk * 4;
            bias4[j] = (add_bias && col < n_end) ? __ldg(reinterpret_cast<const float4*>(kp.bias + col))
                                                 : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        // Byte address of each of this lane's eight rows at the warp's first slab,
        // computed while the accumulator is still being produced.
        const bool bf16_out = FUSED && kp.out_bf16;
        const int64_t esize = bf16_out ? 2 : 4;
        uint64_t rowp[8];
        uint32_t row_ok = 0u;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int m = rows.m(kp, quad * 32 + 4 * i + rsub);
            row_ok |= (m >= 0 ? 1u : 0u) << i;
            rowp[i] = reinterpret_cast<uint64_t>(kp.y) +
                      static_cast<uint64_t>((static_cast<int64_t>(m >= 0 ? m : 0) * kp.ldy + n0 + jbeg * 32 + chunk * 4) *
                                            esize);
        }
        const int mode = bf16_out ? SLAB_BF16 : (sg.split == 0 ? SLAB_F32 : SLAB_RED);
        const bool relu = FUSED && kp.relu;
        const uint32_t taddr = tmem_base + static_cast<uint32_t>(buf * BN) + (static_cast<uint32_t>(quad * 32) << 16);
        // TMA path (fp32 output): box A takes span rows 0..63.  Plain stores: box B
        // takes the span's last 64 rows (overlapping A with the same values when the
        // span is shorter than 128), so the span needs at least 64 rows.  Adds (a
        // later split): box B takes rows 64..127 and rows past the span are added as
        // zeros, which leaves whatever they hold unchanged.
        int m_a, cnt;
        pair_row_span<HALO>(kp, rows, m_a, cnt);
        const bool use_tma = kp.tma_y != 0 && !bf16_out && (mode == SLAB_RED ? cnt >= 1 : cnt >= EPI_BOX_ROWS);
        const bool overlap = mode == SLAB_F32 && cnt < PAIR_ROWS;
        const int b_first = overlap ? cnt - EPI_BOX_ROWS : EPI_BOX_ROWS;  // span row at box B's row 0
        const bool need_b = overlap || cnt > EPI_BOX_ROWS;
        const int my_m = rows.m(kp, trow);
        const int idx = my_m >= 0 ? my_m - m_a : -1;  // this row's place in the span
        const int row_a = idx >= 0 && idx < EPI_BOX_ROWS ? idx : -1;
        const int row_b = idx >= b_first ? idx - b_first : -1;
        const int zero_row = mode == SLAB_RED && trow >= cnt ? trow : -1;  // padding rows cnt..127 of an add

        if (et == 0 && !ptx::mbar_wait(&sm.acc_full[buf], use, kp.wait_limit_ns)) pair_record_timeout(kp, sm, rank);
        ptx::named_bar_sync(1, Cfg::EPI_T);
        if (et == 0) {
            bool go = *sm.abort_flag == 0u;
            if (go && has_rows && cut && sg.split > 0) {  // split 0 has stored (concurrent) or it is this split's turn
                go = kp.reduce_concurrent ? wait_base(kp, sem, sm.abort_flag)
                                          : wait_turn(kp, sem, sg.split, sm.abort_flag);
                if (!go) pair_record_timeout(kp, sm, rank);  // the turn never came: flag the peer too
            }
            *sm.epi_go = go ? 1u : 0u;
        }
        ptx::named_bar_sync(1, Cfg::EPI_T);
        SGB_TRACE(kp, et == 0 && seg_idx < 4, 2 + 2 * seg_idx);  // segment: accumulator ready, turn granted
        const bool store = *sm.epi_go != 0u && has_rows;
        ptx::tc_fence_after();
#ifdef SGB_TRACE_ENABLED
        const uint64_t c0 = ptx::clock64();
#endif
#pragma unroll
        for (int j = 0; j < SLABS; ++j) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(taddr + (jbeg + j) * 32, v);
            ptx::tmem_ld_wait();
            SGB_TRACE_VALUE(kp, et == 0 && seg_idx < 2 && j < 4, 12 + 8 * seg_idx + 2 * j,
                            ptx::clock64() - c0);  // slab j in registers (SM cycles after the grant)
            if (j == SLABS - 1) {  // this warp's part of the accumulator is in registers: tell the leader
                ptx::tc_fence_before();
                __syncwarp();
                if (lane == 0) ptx::mbar_arrive_cluster_relaxed(acc_empty0 + static_cast<uint32_t>(buf) * 8u);
            }
            if (!store) continue;
            if (use_tma) {
                const int col0 = n0 + (jbeg + j) * 32;
                if (col0 >= n_end) continue;  // a slab wholly past the last column (uniform in the group)
                if (add_bias) {
#pragma unroll
                    for (int c = 0; c < 8; ++c) {
                        const float4 b4 = col0 + 4 * c < n_end ? __ldg(reinterpret_cast<const float4*>(kp.bias + col0) + c)
                                                               : make_float4(0.f, 0.f, 0.f, 0.f);
                        v[4 * c] = __float_as_uint(__uint_as_float(v[4 * c]) + b4.x);
                        v[4 * c + 1] = __float_as_uint(__uint_as_float(v[4 * c + 1]) + b4.y);
                        v[4 * c + 2] = __float_as_uint(__uint_as_float(v[4 * c + 2]) + b4.z);
                        v[4 * c + 3] = __float_as_uint(__uint_as_float(v[4 * c + 3]) + b4.w);
                    }
                }
                if (relu) {
#pragma unroll
                    for (int q = 0; q < 32; ++q) v[q] = __float_as_uint(fmaxf(__uint_as_float(v[q]), 0.0f));
                }
                if (issuer) ptx::bulk_wait_read<0>();  // the previous slab's boxes have been read
                ptx::named_bar_sync(EPI_GRP_BAR0 + grp, 128);
                if (row_a >= 0) stage_row(box_a, row_a, v);
                if (row_b >= 0) stage_row(box_b, row_b, v);
                if (zero_row >= 0) {
                    uint32_t z[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) z[q] = 0u;
                    if (zero_row < EPI_BOX_ROWS) stage_row(box_a, zero_row, z);
                    else stage_row(box_b, zero_row - EPI_BOX_ROWS, z);
                }
                ptx::fence_proxy_async_smem();
                ptx::named_bar_sync(EPI_GRP_BAR0 + grp, 128);
                if (issuer) {
                    if (mode == SLAB_RED) {
                        // Split 0's writes were seen (generic proxy) before this segment began;
                        // order that before the TMA's read-modify-writes of the same rows.
                        if (j == 0) ptx::fence_proxy_async_global();
                        ptx::tma_reduce_add_2d_s(&kp.tm_y, box_a, col0, m_a);
                        if (need_b) ptx::tma_reduce_add_2d_s(&kp.tm_y, box_b, col0, m_a + EPI_BOX_ROWS);
                    } else {
                        ptx::tma_store_2d_s(&kp.tm_y, box_a, col0, m_a);
                        if (need_b) ptx::tma_store_2d_s(&kp.tm_y, box_b, col0, m_a + b_first);
                    }
                    ptx::bulk_commit();
                }
                tma_used = true;
                continue;
            }
            const bool col_ok = n0 + (jbeg + j) * 32 + chunk * 4 < n_end;
            const int64_t off = static_cast<int64_t>(j) * 32 * esize;
            if (FUSED && mode == SLAB_BF16)
                slab_out<SLAB_BF16>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], relu);
            else if (mode == SLAB_F32)
                slab_out<SLAB_F32>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], relu);
            else
                slab_out<SLAB_RED>(saddr, v, rowp, off, row_ok, col_ok, add_bias, bias4[j], relu);
            SGB_TRACE_VALUE(kp, et == 0 && seg_idx < 2 && j < 4, 13 + 8 * seg_idx + 2 * j,
                            ptx::clock64() - c0);  // slab j's stores issued
        }
        if (store && use_tma && issuer) {
            if (cut && (sg.split == 0 || !kp.reduce_concurrent)) {
                ptx::bulk_wait_all();  // the TMA writes are performed before the turn passes
                ptx::fence_proxy_async_global();
            } else {
                ptx::bulk_wait_read<0>();  // the boxes may be reused (either path) by the next segment
            }
        }
        if (store && cut) {
            // Split 0's stores (both modes) and every split's adds in the ordered mode must be
            // performed before the next split adds.
            if (sg.split == 0 || !kp.reduce_concurrent) __threadfence();
            ptx::named_bar_sync(1, Cfg::EPI_T);
            if (et == 0) pair_pass_turn(kp, sem, sg);
        }
        SGB_TRACE(kp, et == 0 && seg_idx < 4, 3 + 2 * seg_idx);  // segment: epilogue done
        ++seg_idx;
    }
    if (tma_used && issuer) ptx::bulk_wait_all();  // no TMA store outlives the CTA
}

// ---------------------------------------------------------------- the kernel
template <int BN, int KBS, bool FUSED>
__global__ void __launch_bounds__(PairConfig<BN, KBS>::THREADS, 1)
    conv2d_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                           const __grid_constant__ ConvKernelParams kp)
{
    using Cfg = PairConfig<BN, KBS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairSmem sm;
    sm.a = smem;
    sm.b = smem + Cfg::STAGES * Cfg::A_STAGE;
    sm.epi = smem + Cfg::RING;
    sm.full = reinterpret_cast<uint64_t*>(smem + Cfg::RING + Cfg::EPI_BYTES);
    sm.empty = sm.full + Cfg::STAGES;
    sm.acc_full = sm.empty + Cfg::STAGES;
    sm.acc_empty = sm.acc_full + 2;
    sm.mma_done = sm.acc_empty + 2;
    sm.halo = nullptr;
    sm.halo_full = nullptr;
    sm.halo_empty = nullptr;
    sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.mma_done + 1);
    sm.abort_flag = sm.tmem_slot + 1;
    sm.epi_go = sm.tmem_slot + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = ptx::cluster_ctarank();
    const int pair = static_cast<int>(ptx::cluster_id_x());

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::STAGES; ++i) {
            ptx::mbar_init(&sm.full[i], 2);   // the leader's two producers (expecting both CTAs' bytes)
            ptx::mbar_init(&sm.empty[i], 1);  // the leader's MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.acc_full[i], 1);
            ptx::mbar_init(&sm.acc_empty[i], Cfg::ACC_EMPTY_COUNT);
        }
        ptx::mbar_init(sm.mma_done, 1);
        *sm.abort_flag = 0u;
        *sm.epi_go = 0u;
        ptx::mbar_init_fence();
    }
    // Only the descriptors are prefetched: L2 prefetches of the first stages would
    // queue in the SM's TMA unit ahead of the stages' own loads.
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_a);
        ptx::prefetch_tensormap(&tm_b);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(sm.tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 2) ptx::touch_params(&kp, static_cast<int>(sizeof(kp)));
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // both CTAs' barriers are initialised before any remote arrive or TMA completion
    ptx::tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;
    // Everything above touches only shared memory, tensor memory, parameters and
    // (by prefetches) L2, so it may overlap the previous kernel in the stream.
    SGB_TRACE(kp, threadIdx.x == 0, 0);
    // Each role waits for the previous kernel in the stream (griddepcontrol.wait)
    // right before its first global-memory access, after whatever setup needs
    // only parameters and shared memory: the producers before their first TMA
    // load, the epilogue before its first bias read.  The MMA issuer and the
    // stage waiter touch shared and tensor memory only.
    ptx::grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) pair_producer<BN, KBS, PAIR_A>(&tm_a, &tm_b, kp, sm, rank, pair, 0);
    } else if (warp == WAITER_WARP + 1) {
        if (lane == 0) pair_producer<BN, KBS, PAIR_B>(&tm_a, &tm_b, kp, sm, rank, pair, 0);
    } else if (Cfg::NPROD > 1 && warp == WAITER_WARP + 2) {
        if (lane == 0) pair_producer<BN, KBS, PAIR_A>(&tm_a, &tm_b, kp, sm, rank, pair, 1);
    } else if (Cfg::NPROD > 1 && warp == WAITER_WARP + 3) {
        if (lane == 0) pair_producer<BN, KBS, PAIR_B>(&tm_a, &tm_b, kp, sm, rank, pair, 1);
    } else if (warp == 1) {
        if (rank == 0) pair_mma<BN, KBS>(kp, sm, tmem_base, pair);
    } else if (warp < EPI_WARP0 + Cfg::EPI_WARPS) {
        pair_epilogue<BN, FUSED, false>(kp, sm, tmem_base, rank, pair);
    } else if (warp == WAITER_WARP) {
        if (rank == 0) pair_waiter<BN, KBS>(kp, sm, pair);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();  // neither CTA leaves while the other may still use its shared or tensor memory
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
    SGB_TRACE(kp, threadIdx.x == 0, 10);
}

// ---------------------------------------------------------------- halo loader on CTA pairs
// Stride 1.  A CTA's 128 GEMM rows are 128 consecutive virtual pixels of one
// image seen with the padded row pitch wv = W + 2*pw (virtual pixel j = p*wv + v
// is output pixel (p, v) when v < Q; the others are computed and discarded),
// and the pair takes the same block of images 2i and 2i+1, so that both CTAs'
// operands sit at the same shared-memory offsets, as the 2-CTA MMA requires.
// For each 64-channel chunk one tiled TMA box of whole padded input rows (zero
// fill gives the padding) serves all R*S filter taps: tap (r, s) reads its 128
// A rows in place, r*dh*wv + s*dw rows into the buffer (the 128-byte swizzle
// follows absolute shared-memory addresses, so any start row works).  The
// weight rows of two or three taps of one chunk come in one 4-D box per stage;
// the reduction runs chunk-major, then over the taps.  Per k-block
// this is about 0.1 TMA operation of activations (against one for the im2col
// loader) and half an operation of weights.  Under groups a column block lies
// in one group (pair_columns) and its chunks are that group's Cg input
// channels, from channel g*Cg of x and from the group's weight rows.
template <int BN, int TAPS_>
struct HaloPairConfig {
    static constexpr int B_ROWS = BN / 2;
    static constexpr int B_KB = B_ROWS * BK * 2;      // one tap's weight rows of this CTA
    // Taps (k-blocks) per stage: enough MMA work per stage that the MMA warp's
    // per-stage handshake (~0.1 us) stays small.  Two for 256-wide tiles (1024 MMA
    // cycles per SM); three for narrower ones where the ring still fits beside the
    // two halos (a 3x3 filter then takes three full stages per chunk).
    static constexpr int TAPS = TAPS_;
    static constexpr int B_STAGE = TAPS * B_KB;
    static constexpr int STAGES = 4;
    static constexpr int RING = STAGES * B_STAGE;
    static constexpr int EPI_WARPS = 8;
    static constexpr int EPI_BYTES = EPI_WARPS * EPI_SLOT_BYTES;
    static constexpr int BAR_BYTES = (2 * STAGES + 9) * 8 + 16;
    static constexpr int FIXED_SMEM = RING + EPI_BYTES + BAR_BYTES + 1024;  // + the two halo buffers
    static constexpr uint32_t TMEM_COLS = 2 * BN;
    static constexpr int THREADS = (WAITER_WARP + 2) * 32;  // warps 0 .. 11
    static constexpr uint32_t IDESC = ptx::idesc_bf16_f32(PAIR_TILE_M, BN);
};

// Chunk and first tap of stage st of a tile (TAPS taps per stage).
template <int TAPS>
__device__ __forceinline__ void halo_stage(const ConvKernelParams& kp, int st, int& chunk, int& tap0)
{
    chunk = static_cast<int>(kp.fd_tapst.div(static_cast<uint32_t>(st)));
    tap0 = TAPS * (st - chunk * static_cast<int>(kp.fd_tapst.d));
}

// First virtual pixel of the CTA's row-block and the first padded input row its halo holds.
__device__ __forceinline__ void halo_block(const ConvKernelParams& kp, int m_tile, uint32_t rank, int& n_img, int& j0,
                                           int& prow0)
{
    const int i = static_cast<int>(kp.fd_tpi.div(static_cast<uint32_t>(m_tile)));
    j0 = (m_tile - i * kp.tpi) * PAIR_ROWS;
    n_img = 2 * i + static_cast<int>(rank);
    prow0 = static_cast<int>(kp.fd_wv.div(static_cast<uint32_t>(j0)));
}

// A halo use starts at a chunk's first stage or a segment's first stage and ends
// at the chunk's last stage or the segment's last stage.
__device__ __forceinline__ bool halo_use_starts(const Segment& sg, int st, int tap0) { return st == sg.kb_begin || tap0 == 0; }
template <int TAPS>
__device__ __forceinline__ bool halo_use_ends(const ConvKernelParams& kp, const Segment& sg, int st, int tap0)
{
    return st + 1 == sg.kb_end || tap0 + TAPS >= kp.R * kp.S;
}

// L2 prefetch of this CTA's first halo and first weight stages, issued before
// the grid-dependency wait so that the loads after it find them in L2 (a
// prefetch reads nothing into the CTA, and L2 is coherent: a later load still
// sees whatever the previous kernel writes).
template <int BN, int TAPS>
__device__ void halo_pair_prefetch(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const ConvKernelParams& kp,
                                   uint32_t rank, int pair)
{
    using Cfg = HaloPairConfig<BN, TAPS>;
    PairWalker walk(kp, pair);
    Segment sg;
    if (!walk.next(kp, sg)) return;
    int m_tile, n_tile;
    pair_tile_coords(kp, sg.tile, m_tile, n_tile);
    int n_img, j0, prow0, chunk, tap0, n0, n_end, c_base;
    halo_block(kp, m_tile, rank, n_img, j0, prow0);
    halo_stage<TAPS>(kp, sg.kb_begin, chunk, tap0);
    pair_columns<BN>(kp, n_tile, n0, n_end, c_base);
    if (n_img < kp.N) ptx::tma_prefetch_4d(tm_a, c_base + chunk * BK, -kp.pw, prow0 - kp.ph, n_img);
    const int b_row = n0 + static_cast<int>(rank) * Cfg::B_ROWS;
    for (int st = sg.kb_begin; st < sg.kb_end && st < sg.kb_begin + Cfg::STAGES; ++st) {
        halo_stage<TAPS>(kp, st, chunk, tap0);
        ptx::tma_prefetch_4d(tm_b, 0, b_row, chunk, tap0);
    }
}

// Producer of the halos (warp 0, one thread, both CTAs).
template <int BN, int TAPS>
__device__ void halo_pair_producer_a(const CUtensorMap* tm_a, const ConvKernelParams& kp, const PairSmem& sm,
                                     uint32_t rank, int pair)
{
    const uint32_t hfull0 = ptx::mapa_shared(ptx::smem_addr(sm.halo_full), 0u);  // the leader's
    int h = 0;  // halo uses issued
    bool ok = true;
    PairWalker walk(kp, pair);
    Segment sg;
    while (ok && walk.next(kp, sg)) {
        int m_tile, n_tile;
        pair_tile_coords(kp, sg.tile, m_tile, n_tile);
        int n_img, j0, prow0, n0, n_end, c_base;
        halo_block(kp, m_tile, rank, n_img, j0, prow0);
        pair_columns<BN>(kp, n_tile, n0, n_end, c_base);  // the group's channels start at c_base
        for (int st = sg.kb_begin; st < sg.kb_end; ++st) {
            int chunk, tap0;
            halo_stage<TAPS>(kp, st, chunk, tap0);
            if (!halo_use_starts(sg, st, tap0)) continue;
            if (*sm.abort_flag) { ok = false; break; }
            const int slot = h & 1;
            if (!ptx::mbar_wait_spin(&sm.halo_empty[slot], (static_cast<uint32_t>(h >> 1) & 1u) ^ 1u, kp.wait_limit_ns)) {
                pair_record_timeout(kp, sm, rank);
                ok = false;
                break;
            }
            if (h == 0) {  // everything before reads only parameters and shared memory
                ptx::grid_dependency_wait();
                SGB_TRACE(kp, threadIdx.x == 0, 1);
            }
            if (rank == 0) ptx::mbar_arrive_expect_tx(&sm.halo_full[slot], 2u * static_cast<uint32_t>(kp.halo_tx));
            ptx::tma_load_4d_pair(sm.halo + slot * kp.halo_bytes, tm_a, hfull0 + static_cast<uint32_t>(slot) * 8u,
                                  c_base + chunk * BK, -kp.pw, prow0 - kp.ph, n_img);
            SGB_PAIR_MARK(kp, 200 + h, static_cast<int>(rank));
            ++h;
        }
    }
    // Drain: each buffer's last use has been released by the MMA (so it landed).
    for (int i = h > 2 ? h - 2 : 0; i < h; ++i)
        ptx::mbar_wait(&sm.halo_empty[i & 1], static_cast<uint32_t>(i >> 1) & 1u, kp.wait_limit_ns);
}

// Producer of the weight stages (warp 11, one thread, both CTAs).
template <int BN, int TAPS>
__device__ void halo_pair_producer_b(const CUtensorMap* tm_b, const ConvKernelParams& kp, const PairSmem& sm,
                                     uint32_t rank, int pair)
{
    using Cfg = HaloPairConfig<BN, TAPS>;
    constexpr int STAGES = Cfg::STAGES;
    SGB_TRACE(kp, true, 6);  // weight producer: entered
    const uint32_t full0 = ptx::mapa_shared(ptx::smem_addr(sm.full), 0u);
    int it = 0;
    bool ok = true;
    PairWalker walk(kp, pair);
    Segment sg;
    SGB_TRACE(kp, true, 7);  // weight producer: walker ready
    while (ok && walk.next(kp, sg)) {
        SGB_TRACE(kp, it == 0, 9);  // weight producer: first segment
        int m_tile, n_tile;
        pair_tile_coords(kp, sg.tile, m_tile, n_tile);
        int n0, n_end, c_base;
        pair_columns<BN>(kp, n_tile, n0, n_end, c_base);
        const int b_row = n0 + static_cast<int>(rank) * Cfg::B_ROWS;
        for (int st = sg.kb_begin; st < sg.kb_end; ++st, ++it) {
            const int slot = it % STAGES;
            if (*sm.abort_flag) { ok = false; break; }
            SGB_TRACE(kp, it == 0, 11);  // weight producer: abort flag read
            if (!ptx::mbar_wait_spin(&sm.empty[slot], (static_cast<uint32_t>(it / STAGES) & 1u) ^ 1u, kp.wait_limit_ns)) {
                pair_record_timeout(kp, sm, rank);
                ok = false;
                break;
            }
            SGB_TRACE(kp, it == 0, 30);  // weight producer: slot free
            int chunk, tap0;
            halo_stage<TAPS>(kp, st, chunk, tap0);
            SGB_TRACE(kp, it == 0, 8);  // weight producer: first stage's coordinates
            if (it == 0) ptx::grid_dependency_wait();  // everything before reads only parameters and shared memory
            // The box always counts TAPS taps (a tap past R*S reads zeros).
            if (rank == 0) ptx::mbar_arrive_expect_tx(&sm.full[slot], 2u * static_cast<uint32_t>(Cfg::B_STAGE));
            ptx::tma_load_4d_pair(sm.b + slot * Cfg::B_STAGE, tm_b, full0 + static_cast<uint32_t>(slot) * 8u, 0, b_row,
                                  chunk, tap0);
            SGB_PAIR_MARK(kp, it, 5 + static_cast<int>(rank));
        }
    }
    for (int i = it > STAGES ? it - STAGES : 0; i < it; ++i)
        ptx::mbar_wait(&sm.empty[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u, kp.wait_limit_ns);
}

// Stage waiter (warp 10, leader): the chunk's halo, then the stage's weights.
template <int BN, int TAPS>
__device__ void halo_pair_waiter(const ConvKernelParams& kp, const PairSmem& sm, int pair)
{
    constexpr int STAGES = HaloPairConfig<BN, TAPS>::STAGES;
    const int lane = threadIdx.x & 31;
    bool waiting = true;
    int it = 0, h = 0;
    PairWalker walk(kp, pair);
    Segment sg;
    while (walk.next(kp, sg)) {
        for (int st = sg.kb_begin; st < sg.kb_end; ++st, ++it) {
            const int slot = it % STAGES;
            const uint32_t use = static_cast<uint32_t>(it / STAGES);
            int chunk, tap0;
            halo_stage<TAPS>(kp, st, chunk, tap0);
            if (lane == 0) {
                if (halo_use_starts(sg, st, tap0)) {
                    if (waiting && (*sm.abort_flag ||
                                    !ptx::mbar_wait_spin(&sm.halo_full[h & 1], static_cast<uint32_t>(h >> 1) & 1u,
                                                         kp.wait_limit_ns))) {
                        pair_record_timeout(kp, sm, 0u);
                        waiting = false;
                    }
                    ++h;
                }
                if (waiting && (*sm.abort_flag || !ptx::mbar_wait_spin(&sm.full[slot], use & 1u, kp.wait_limit_ns))) {
                    pair_record_timeout(kp, sm, 0u);
                    waiting = false;
                }
                // After a timeout: pace the MMA warp by its own release of the previous use.
                if (!waiting && use > 0)
                    for (int t = 0; t < 16 && !ptx::mbar_wait(&sm.empty[slot], (use - 1u) & 1u, kp.wait_limit_ns); ++t) {
                    }
                SGB_PAIR_MARK(kp, it, 2);
            }
            __syncwarp();
            ptx::named_bar_arrive(STAGE_BAR0 + slot, 64);
        }
    }
}

// MMA issuer (warp 1, leader).
template <int BN, int TAPS>
__device__ void halo_pair_mma(const ConvKernelParams& kp, const PairSmem& sm, uint32_t tmem_base, int pair)
{
    using Cfg = HaloPairConfig<BN, TAPS>;
    constexpr int STAGES = Cfg::STAGES;
    const int lane = threadIdx.x & 31;
    const int taps = kp.R * kp.S;
    const uint64_t halo_desc0 = ptx::sw128_kmajor_desc(ptx::smem_addr(sm.halo));
    const uint64_t b_desc0 = ptx::sw128_kmajor_desc(ptx::smem_addr(sm.b));
    int it = 0, seg_idx = 0, h = 0;
    bool issue = true;
    PairWalker walk(kp, pair);
    Segment sg;
    while (walk.next(kp, sg)) {
        const int buf = seg_idx & 1;
        const uint32_t use = static_cast<uint32_t>(seg_idx >> 1) & 1u;
        if (lane == 0 && issue) {
            if (*sm.abort_flag || !ptx::mbar_wait(&sm.acc_empty[buf], use ^ 1u, kp.wait_limit_ns)) {
                pair_record_timeout(kp, sm, 0u);
                issue = false;
            }
        }
        __syncwarp();
        ptx::tc_fence_after();
        const uint32_t tmem_d = tmem_base + static_cast<uint32_t>(buf * BN);
        const bool go = __shfl_sync(0xffffffffu, issue ? 1 : 0, 0) != 0;
        int m_tile, n_tile;
        pair_tile_coords(kp, sg.tile, m_tile, n_tile);
        int n_img, j0, prow0;
        halo_block(kp, m_tile, 0u, n_img, j0, prow0);
        const int a0 = j0 - prow0 * kp.wv;  // the same in both CTAs
        for (int st = sg.kb_begin; st < sg.kb_end; ++st, ++it) {
            const int slot = it % STAGES;
            int chunk, tap0;
            halo_stage<TAPS>(kp, st, chunk, tap0);
            if (halo_use_starts(sg, st, tap0)) ++h;
            const int hslot = (h - 1) & 1;
            const bool hlast = halo_use_ends<TAPS>(kp, sg, st, tap0);
            ptx::named_bar_sync(STAGE_BAR0 + slot, 64);
            ptx::tc_fence_after();
            if (lane == 0) SGB_PAIR_MARK(kp, it, 3);
            if (go) {  // warp-uniform; one elected lane issues (see pair_mma)
#pragma unroll
                for (int jt = 0; jt < Cfg::TAPS; ++jt) {
                    const int tap = tap0 + jt;
                    if (tap < taps) {
                        const int r = static_cast<int>(kp.fd_s.div(static_cast<uint32_t>(tap)));
                        const int sx = tap - r * kp.S;
                        const int a_row = a0 + r * kp.dh * kp.wv + sx * kp.dw;
                        const uint64_t ad =
                            halo_desc0 + static_cast<uint64_t>((hslot * kp.halo_bytes + a_row * 128) >> 4);
                        const uint64_t bd = b_desc0 + static_cast<uint64_t>((slot * Cfg::B_STAGE + jt * Cfg::B_KB) >> 4);
                        static_assert(BK / UMMA_K == 4 && UMMA_K * 2 == 32, "four MMAs of 32 bytes per k-block");
                        ptx::mma_bf16_pair_elect_kb(tmem_d, ad, bd, Cfg::IDESC, (st > sg.kb_begin || jt > 0) ? 1u : 0u);
                    }
                }
            }
            ptx::mma_commit_pair_elect(&sm.empty[slot], 0x3);  // every stage, issuing or not
            if (hlast) ptx::mma_commit_pair_elect(&sm.halo_empty[hslot], 0x3);
            if (lane == 0) SGB_PAIR_MARK(kp, it, 4);
        }
        ptx::mma_commit_pair_elect(&sm.acc_full[buf], 0x3);
        __syncwarp();
        ++seg_idx;
    }
    ptx::mma_commit_pair_elect(sm.mma_done, 0x1);  // the lane that issued the MMAs
    if (lane == 0) ptx::mbar_wait(sm.mma_done, 0u, kp.wait_limit_ns);
    __syncwarp();
}

template <int BN, int TAPS, bool FUSED>
__global__ void __launch_bounds__(HaloPairConfig<BN, TAPS>::THREADS, 1)
    conv2d_fwd_pair_halo_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                                const __grid_constant__ ConvKernelParams kp)
{
    using Cfg = HaloPairConfig<BN, TAPS>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PairSmem sm;
    sm.a = nullptr;
    sm.b = smem;
    sm.halo = smem + Cfg::RING;  // 2 buffers of kp.halo_bytes (1024-byte multiples)
    sm.epi = sm.halo + 2 * kp.halo_bytes;
    sm.full = reinterpret_cast<uint64_t*>(sm.epi + Cfg::EPI_BYTES);
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
    const uint32_t rank = ptx::cluster_ctarank();
    const int pair = static_cast<int>(ptx::cluster_id_x());

    if (threadIdx.x == 0) {
        for (int i = 0; i < Cfg::STAGES; ++i) {
            ptx::mbar_init(&sm.full[i], 1);   // the leader's weight producer (expecting both CTAs' bytes)
            ptx::mbar_init(&sm.empty[i], 1);  // the leader's MMA commit
        }
        for (int i = 0; i < 2; ++i) {
            ptx::mbar_init(&sm.acc_full[i], 1);
            ptx::mbar_init(&sm.acc_empty[i], 2 * Cfg::EPI_WARPS);
            ptx::mbar_init(&sm.halo_full[i], 1);   // the leader's halo producer
            ptx::mbar_init(&sm.halo_empty[i], 1);  // the leader's MMA commit
        }
        ptx::mbar_init(sm.mma_done, 1);
        *sm.abort_flag = 0u;
        *sm.epi_go = 0u;
        ptx::mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        ptx::prefetch_tensormap(&tm_a);
        ptx::prefetch_tensormap(&tm_b);
        halo_pair_prefetch<BN, TAPS>(&tm_a, &tm_b, kp, rank, pair);
    }
    if (warp == 1) {
        ptx::tmem_alloc_pair(sm.tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish_pair();
    }
    if (warp == 2) ptx::touch_params(&kp, static_cast<int>(sizeof(kp)));
    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;
    SGB_TRACE(kp, threadIdx.x == 0, 0);
    // Each role waits for the previous kernel in the stream (griddepcontrol.wait)
    // right before its first global-memory access, after whatever setup needs
    // only parameters and shared memory: the producers before their first TMA
    // load, the epilogue before its first bias read.  The MMA issuer and the
    // stage waiter touch shared and tensor memory only.
    ptx::grid_launch_dependents();

    if (warp == 0) {
        if (lane == 0) halo_pair_producer_a<BN, TAPS>(&tm_a, kp, sm, rank, pair);
    } else if (warp == WAITER_WARP + 1) {
        if (lane == 0) halo_pair_producer_b<BN, TAPS>(&tm_b, kp, sm, rank, pair);
    } else if (warp == 1) {
        if (rank == 0) halo_pair_mma<BN, TAPS>(kp, sm, tmem_base, pair);
    } else if (warp < EPI_WARP0 + Cfg::EPI_WARPS) {
        pair_epilogue<BN, FUSED, true>(kp, sm, tmem_base, rank, pair);
    } else if (warp == WAITER_WARP) {
        if (rank == 0) halo_pair_waiter<BN, TAPS>(kp, sm, pair);
    }

    ptx::tc_fence_before();
    __syncthreads();
    ptx::cluster_sync();
    if (warp == 1) {
        ptx::tc_fence_after();
        ptx::tmem_dealloc_pair(tmem_base, Cfg::TMEM_COLS);
    }
    SGB_TRACE(kp, threadIdx.x == 0, 10);
}

template <int BN, int TAPS>
cudaError_t launch_conv2d_pair_halo(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const ConvKernelParams& kp,
                                    int pairs, cudaStream_t stream);
template <int BN, int TAPS>
int conv2d_pair_halo_max_resident(bool fused, int smem_bytes);
template <int BN, int TAPS>
inline int conv2d_pair_halo_smem_bytes(int halo_bytes)
{
    return HaloPairConfig<BN, TAPS>::FIXED_SMEM + 2 * halo_bytes;
}
#define SGB_PAIR_HALO_SIG(BN_, TAPS_)                                                                        \
    cudaError_t launch_conv2d_pair_halo<BN_, TAPS_>(const CUtensorMap&, const CUtensorMap&, const ConvKernelParams&, \
                                                    int, cudaStream_t)
#define SGB_PAIR_HALO_RES_SIG(BN_, TAPS_) int conv2d_pair_halo_max_resident<BN_, TAPS_>(bool, int)

// Host-side launcher: `pairs` clusters of two CTAs.
template <int BN, int KBS>
cudaError_t launch_conv2d_pair(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const ConvKernelParams& kp, int pairs,
                               cudaStream_t stream);

// Largest number of CTA pairs of this instantiation that can be resident at once.
template <int BN, int KBS>
int conv2d_pair_max_resident(bool fused);

#define SGB_PAIR_SIG(BN_, KBS_)                                                                              \
    cudaError_t launch_conv2d_pair<BN_, KBS_>(const CUtensorMap&, const CUtensorMap&, const ConvKernelParams&, \
                                              int, cudaStream_t)
#define SGB_PAIR_RES_SIG(BN_, KBS_) int conv2d_pair_max_resident<BN_, KBS_>(bool)

}  // namespace sgb
