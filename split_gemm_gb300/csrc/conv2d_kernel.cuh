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
// One CTA computes one BM x BN output tile over one slice of the reduction
// (split-K).  Warp roles (192 threads):
//   warp 0      TMA producer: weight tile (tiled TMA) and, for the TMA loader,
//               the im2col activation tile (im2col-mode TMA), into a STAGES-deep
//               ring of shared-memory buffers guarded by full/empty mbarriers;
//   warp 1      TMEM allocator and single-thread tcgen05.mma issuer (128 x BN x 16
//               per instruction, fp32 accumulator in tensor memory);
//   warps 2..5  gather producers for the cp.async / scalar loaders, then the
//               epilogue: TMEM -> registers (+ bias) -> shared memory -> TMA store,
//               or, under split-K, the serialised in-place reduction into y.
// The shared-memory ring replaces block-wide syncs between load and MMA (burn
// PR #2545's sync-placement discussion; ROCm/rocMLIR PR #1511 "Double buffering
// improvements" splits loads and MMAs into overlapping stages the same way).
//
// Split-K (NVIDIA/Fuser issue #1316 "Split-K matmul is slow even for few
// partitions", Eliminating the workspace): the S CTAs of one output tile take
// turns on a per-tile semaphore.  Split j waits until the semaphore reads j,
// adds its partial tile into y (split 0 stores acc + bias), then publishes j+1;
// the last split resets it to 0.  The fp32 output is the work buffer, so the
// only extra memory is one 32-bit word per tile.
//
// Every wait is bounded (about wait_limit_ns, counted in SM cycles).  A wait that runs out
// records CONV2D_ERR_TIMEOUT in the status word, and the CTA drains its own
// in-flight copies and MMAs, frees its tensor memory and exits.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>

#include "ptx.cuh"

namespace sgb {

constexpr int BM = 128;          // output pixels per tile (MMA M)
constexpr int BK = 64;           // reduction elements per stage: one 128-byte bf16 row
constexpr int UMMA_K = 16;       // reduction per tcgen05.mma of kind::f16
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int EPI_THREAD0 = 64;  // first thread of warp 2
constexpr int A_STAGE_BYTES = BM * BK * 2;
constexpr uint32_t STATUS_TIMEOUT = 6;  // same value as CONV2D_ERR_TIMEOUT

enum LoaderKind : int { LOADER_TMA = 1, LOADER_CPASYNC = 2, LOADER_SCALAR = 3 };

struct ConvKernelParams {
    const uint16_t* x;  // bf16 NHWC
    const uint16_t* w;  // bf16 KRSC
    const float* bias;  // [K] or nullptr
    float* y;           // fp32 NHWC = [M][K]
    uint32_t* status;   // device status word or nullptr
    uint32_t* sems;     // one per output tile (split-K only)
    int N, H, W, C, K, R, S, P, Q;
    int sh, sw, ph, pw, dh, dw;
    int M, CRS, num_kb;
    int splits, m_tiles, n_tiles;
    int use_tma_store;
    int debug_flags;
    unsigned long long wait_limit_ns;
    unsigned long long* trace;  // per-CTA phase timestamps; only written in trace builds
};

// Phase timestamps for profiling builds (compiled with SGB_TRACE_ENABLED):
// slot `slot` of CTA blockIdx.x gets the global timer when `cond` holds.
#ifdef SGB_TRACE_ENABLED
#define SGB_TRACE(kp, cond, slot)                                                               \
    do {                                                                                        \
        if ((kp).trace && (cond)) (kp).trace[static_cast<size_t>(blockIdx.x) * 16 + (slot)] =   \
            ::sgb::ptx::globaltimer();                                                          \
    } while (0)
#else
#define SGB_TRACE(kp, cond, slot) \
    do {                          \
    } while (0)
#endif

template <int BN>
struct TileConfig {
    static_assert(BN == 64 || BN == 128 || BN == 256, "BN must be 64, 128 or 256");
    static constexpr int B_STAGE_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_STAGE_BYTES + B_STAGE_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int RING_BYTES = STAGES * STAGE_BYTES;
    static constexpr int EPI_BYTES = BM * BN * 4;  // fp32 output tile staged for the TMA store
    static_assert(RING_BYTES >= EPI_BYTES, "output staging reuses the ring");
    static constexpr int BAR_BYTES = (2 * STAGES + 1) * 8 + 16;
    static constexpr int SMEM_BYTES = RING_BYTES + BAR_BYTES + 1024;  // + alignment slack
    static constexpr uint32_t TMEM_COLS = BN;
};

struct SmemView {
    uint8_t* a;       // STAGES x A tile
    uint8_t* b;       // STAGES x B tile
    uint64_t* full;   // STAGES
    uint64_t* empty;  // STAGES
    uint64_t* acc_full;
    uint32_t* tmem_slot;
    volatile uint32_t* abort_flag;
    volatile uint32_t* epi_go;  // epilogue decision, written by one thread between two barriers
};

__device__ __forceinline__ void record_timeout(const ConvKernelParams& kp, volatile uint32_t* abort_flag)
{
    *abort_flag = 1u;
    if (kp.status) atomicMax(kp.status, STATUS_TIMEOUT);
}

// ---------------------------------------------------------------- TMA producer (warp 0, one thread)
template <int BN, int LOADER>
__device__ void run_tma_producer(const CUtensorMap* tm_a, const CUtensorMap* tm_b, const ConvKernelParams& kp,
                                 const SmemView& sm, int m0, int n0, int kb_begin, int nkb)
{
    using Cfg = TileConfig<BN>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr uint32_t TX = (LOADER == LOADER_TMA ? A_STAGE_BYTES : 0) + Cfg::B_STAGE_BYTES;

    // Window origin of the tile's first pixel and the first (r, s, c) of this split.
    const int pq = kp.P * kp.Q;
    const int n_img = m0 / pq;
    const int rem = m0 - n_img * pq;
    const int p0 = rem / kp.Q;
    const int q0 = rem - p0 * kp.Q;
    const int w_org = q0 * kp.sw - kp.pw;
    const int h_org = p0 * kp.sh - kp.ph;
    const int kk0 = kb_begin * BK;
    const int rs0 = kk0 / kp.C;
    int c = kk0 - rs0 * kp.C;
    int r = rs0 / kp.S;
    int s = rs0 - r * kp.S;

    int issued = 0;
    for (int i = 0; i < nkb; ++i) {
        const int stage = i % STAGES;
        const uint32_t parity = static_cast<uint32_t>(i / STAGES) & 1u;
        if (*sm.abort_flag) break;
        if (!ptx::mbar_wait(&sm.empty[stage], parity ^ 1u, kp.wait_limit_ns)) {
            record_timeout(kp, sm.abort_flag);
            break;
        }
        ptx::mbar_arrive_expect_tx(&sm.full[stage], TX);
        if (LOADER == LOADER_TMA) {
            ptx::tma_load_im2col_4d(sm.a + stage * A_STAGE_BYTES, tm_a, &sm.full[stage], c, w_org, h_org, n_img,
                                    static_cast<uint16_t>(s * kp.dw), static_cast<uint16_t>(r * kp.dh));
            c += BK;
            if (c == kp.C) {
                c = 0;
                if (++s == kp.S) {
                    s = 0;
                    ++r;
                }
            }
        }
        ptx::tma_load_2d(sm.b + stage * Cfg::B_STAGE_BYTES, tm_b, &sm.full[stage], (kb_begin + i) * BK, n0);
        SGB_TRACE(kp, i == 0, 2);
        ++issued;
    }
    SGB_TRACE(kp, true, 3);
    // Drain: the last loads of each stage must have landed before the CTA can exit.
    for (int i = issued > STAGES ? issued - STAGES : 0; i < issued; ++i)
        ptx::mbar_wait(&sm.full[i % STAGES], static_cast<uint32_t>(i / STAGES) & 1u, kp.wait_limit_ns);
}

// ---------------------------------------------------------------- MMA issuer (warp 1, one thread)
template <int BN>
__device__ void run_mma_issuer(const ConvKernelParams& kp, const SmemView& sm, uint32_t tmem_d, int nkb)
{
    using Cfg = TileConfig<BN>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr uint32_t IDESC = ptx::idesc_bf16_f32(BM, BN);
    for (int i = 0; i < nkb; ++i) {
        const int stage = i % STAGES;
        const uint32_t parity = static_cast<uint32_t>(i / STAGES) & 1u;
        if (*sm.abort_flag) break;
        if (!ptx::mbar_wait(&sm.full[stage], parity, kp.wait_limit_ns)) {
            record_timeout(kp, sm.abort_flag);
            break;
        }
        ptx::tc_fence_after();
        SGB_TRACE(kp, i == 0, 4);
        const uint32_t a_addr = ptx::smem_addr(sm.a + stage * A_STAGE_BYTES);
        const uint32_t b_addr = ptx::smem_addr(sm.b + stage * Cfg::B_STAGE_BYTES);
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
            // Advancing along K inside a 128-B swizzled row moves the start address by 32 B.
            const uint64_t ad = ptx::sw128_kmajor_desc(a_addr + k * UMMA_K * 2);
            const uint64_t bd = ptx::sw128_kmajor_desc(b_addr + k * UMMA_K * 2);
            ptx::mma_bf16(tmem_d, ad, bd, IDESC, (i > 0 || k > 0) ? 1u : 0u);
        }
        ptx::mma_commit(&sm.empty[stage]);
    }
    // Signals the epilogue, and (waiting on it here too) guarantees no MMA is in
    // flight when the CTA reaches its teardown.
    SGB_TRACE(kp, true, 5);
    ptx::mma_commit(sm.acc_full);
    ptx::mbar_wait(sm.acc_full, 0u, kp.wait_limit_ns);
    SGB_TRACE(kp, true, 6);
}

// ---------------------------------------------------------------- gather producers (warps 2..5)
__device__ __forceinline__ uint32_t sw128_offset(int row, int chunk16)
{
    return static_cast<uint32_t>(row * 128 + ((chunk16 ^ (row & 7)) << 4));
}

// A tile by 16-byte cp.async: each thread owns one tile row (output pixel); a
// 16-byte chunk is 8 consecutive channels of one filter tap (needs C % 8 == 0).
template <int BN>
__device__ void run_gather_cpasync(const ConvKernelParams& kp, const SmemView& sm, int m0, int kb_begin, int nkb)
{
    using Cfg = TileConfig<BN>;
    constexpr int STAGES = Cfg::STAGES;
    constexpr int LAG = STAGES - 1 < 3 ? STAGES - 1 : 3;  // stages in flight per thread
    const int row = threadIdx.x - EPI_THREAD0;
    const int m = m0 + row;
    const bool row_ok = m < kp.M;
    int n_img = 0, p = 0, q = 0;
    if (row_ok) {
        const int pq = kp.P * kp.Q;
        n_img = m / pq;
        const int rem = m - n_img * pq;
        p = rem / kp.Q;
        q = rem - p * kp.Q;
    }
    const int ih0 = p * kp.sh - kp.ph;
    const int iw0 = q * kp.sw - kp.pw;
    const uint16_t* xb = kp.x + static_cast<int64_t>(n_img) * kp.H * kp.W * kp.C;

    int issued = 0, arrived = 0;
    for (int i = 0; i < nkb; ++i) {
        const int stage = i % STAGES;
        const uint32_t parity = static_cast<uint32_t>(i / STAGES) & 1u;
        if (*sm.abort_flag) break;
        if (!ptx::mbar_wait(&sm.empty[stage], parity ^ 1u, kp.wait_limit_ns)) {
            record_timeout(kp, sm.abort_flag);
            break;
        }
        uint8_t* dst = sm.a + stage * A_STAGE_BYTES;
        const int kk0 = (kb_begin + i) * BK;
#pragma unroll
        for (int j = 0; j < BK / 8; ++j) {
            const int kk = kk0 + j * 8;
            const void* src = kp.x;
            uint32_t bytes = 0;
            if (row_ok && kk < kp.CRS) {
                const int rs = kk / kp.C;
                const int c = kk - rs * kp.C;
                const int r = rs / kp.S;
                const int s = rs - r * kp.S;
                const int ih = ih0 + r * kp.dh;
                const int iw = iw0 + s * kp.dw;
                if (static_cast<unsigned>(ih) < static_cast<unsigned>(kp.H) &&
                    static_cast<unsigned>(iw) < static_cast<unsigned>(kp.W)) {
                    src = xb + (static_cast<int64_t>(ih) * kp.W + iw) * kp.C + c;
                    bytes = 16;
                }
            }
            ptx::cp_async_16(dst + sw128_offset(row, j), src, bytes);
        }
        ptx::cp_async_commit();
        ++issued;
        if (issued - arrived > LAG) {
            ptx::cp_async_wait<LAG>();
            ptx::fence_proxy_async_smem();
            ptx::mbar_arrive(&sm.full[arrived % STAGES]);
            ++arrived;
        }
    }
    ptx::cp_async_wait_all();
    ptx::fence_proxy_async_smem();
    while (arrived < issued) {
        ptx::mbar_arrive(&sm.full[arrived % STAGES]);
        ++arrived;
    }
}

// A and B tiles element by element (any C, any C*R*S): plain loads, then
// 16-byte shared stores in the swizzled layout.
template <int BN>
__device__ void run_gather_scalar(const ConvKernelParams& kp, const SmemView& sm, int m0, int n0, int kb_begin,
                                  int nkb)
{
    using Cfg = TileConfig<BN>;
    constexpr int STAGES = Cfg::STAGES;
    const int row = threadIdx.x - EPI_THREAD0;
    const int m = m0 + row;
    const bool row_ok = m < kp.M;
    int n_img = 0, p = 0, q = 0;
    if (row_ok) {
        const int pq = kp.P * kp.Q;
        n_img = m / pq;
        const int rem = m - n_img * pq;
        p = rem / kp.Q;
        q = rem - p * kp.Q;
    }
    const int ih0 = p * kp.sh - kp.ph;
    const int iw0 = q * kp.sw - kp.pw;
    const uint16_t* xb = kp.x + static_cast<int64_t>(n_img) * kp.H * kp.W * kp.C;

    for (int i = 0; i < nkb; ++i) {
        const int stage = i % STAGES;
        const uint32_t parity = static_cast<uint32_t>(i / STAGES) & 1u;
        if (*sm.abort_flag) break;
        if (!ptx::mbar_wait(&sm.empty[stage], parity ^ 1u, kp.wait_limit_ns)) {
            record_timeout(kp, sm.abort_flag);
            break;
        }
        const int kk0 = (kb_begin + i) * BK;
        // A row: walk (r, s, c) incrementally from kk0.
        {
            const int rs0 = kk0 / kp.C;
            int c = kk0 - rs0 * kp.C;
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
                    if (++c == kp.C) {
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
            for (int b = row; b < BN; b += EPI_THREADS) {
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
        ptx::mbar_arrive(&sm.full[stage]);
    }
}

// ---------------------------------------------------------------- epilogue (warps 2..5)
// Waits (thread et == 0, bounded) until the tile semaphore reads `split`.
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

// Publishes the next split's turn (the last split resets the semaphore to 0).
__device__ __forceinline__ void pass_turn(const ConvKernelParams& kp, int tile, int split)
{
    const bool skip = (kp.debug_flags & 1) && split == 0;  // test hook: never signal
    if (skip) return;
    const uint32_t next = (split + 1 == kp.splits) ? 0u : static_cast<uint32_t>(split + 1);
    ptx::st_release_gpu(kp.sems + tile, next);
}

template <int BN>
__device__ void run_epilogue(const CUtensorMap* tm_y, const ConvKernelParams& kp, const SmemView& sm,
                             uint32_t tmem_base, int m0, int n0, int split, int tile)
{
    const int et = threadIdx.x - EPI_THREAD0;  // 0..127
    const int quad = (threadIdx.x >> 5) & 3;   // TMEM lane quadrant this warp may access
    const int row = quad * 32 + (threadIdx.x & 31);
    const int m = m0 + row;
    const bool row_ok = m < kp.M;
    const bool add_bias = kp.bias != nullptr && split == 0;
    const bool serial = kp.splits > 1;

    const bool acc_ready = ptx::mbar_wait(sm.acc_full, 0u, kp.wait_limit_ns);
    if (!acc_ready) record_timeout(kp, sm.abort_flag);
    // One thread decides for all 128, so that every epilogue warp takes the same
    // path through the named barriers below.
    ptx::named_bar_sync(1, EPI_THREADS);
    if (et == 0) *sm.epi_go = (*sm.abort_flag == 0u) ? 1u : 0u;
    ptx::named_bar_sync(1, EPI_THREADS);
    if (!*sm.epi_go) return;
    SGB_TRACE(kp, et == 0, 7);
    ptx::tc_fence_after();
    const uint32_t taddr = tmem_base + (static_cast<uint32_t>(quad * 32) << 16);

    if (kp.use_tma_store) {
        // TMEM -> registers (+bias) -> 128-B swizzled shared slabs of 32 columns.
        // Split 0 (or no split) stores each slab as soon as it is complete; later
        // splits stage every slab, wait for their turn, then let the TMA unit add
        // the slabs into y in place.
        uint8_t* stage_base = sm.a;  // the ring is idle once the accumulator is complete
        const bool store_now = split == 0;
#pragma unroll 1
        for (int j = 0; j < BN / 32; ++j) {
            uint32_t v[32];
            ptx::tmem_ld_32x32b_x32(taddr + j * 32, v);
            ptx::tmem_ld_wait();
            if (add_bias) {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    const int n = n0 + j * 32 + e;
                    const float b = n < kp.K ? __ldg(kp.bias + n) : 0.0f;
                    v[e] = __float_as_uint(__uint_as_float(v[e]) + b);
                }
            }
            const uint32_t slab = ptx::smem_addr(stage_base + j * (BM * 128));
#pragma unroll
            for (int c = 0; c < 8; ++c)
                ptx::st_shared_v4(slab + sw128_offset(row, c), v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
            ptx::fence_proxy_async_smem();
            if (store_now) {
                ptx::named_bar_sync(1, EPI_THREADS);
                if (et == 0) {
                    ptx::tma_store_2d(tm_y, stage_base + j * (BM * 128), n0 + j * 32, m0);
                    ptx::bulk_commit();
                }
            }
        }
        if (!store_now) {
            ptx::named_bar_sync(1, EPI_THREADS);
            if (et == 0 && wait_turn(kp, tile, split, sm.abort_flag)) {
                ptx::fence_proxy_async_global();
#pragma unroll 1
                for (int j = 0; j < BN / 32; ++j)
                    ptx::tma_reduce_add_2d(tm_y, stage_base + j * (BM * 128), n0 + j * 32, m0);
                ptx::bulk_commit();
                ptx::bulk_wait_all();
                ptx::fence_proxy_async_global();
                __threadfence();
                pass_turn(kp, tile, split);
            }
        } else if (et == 0) {
            if (serial) {
                ptx::bulk_wait_all();  // writes done before the next split may add to them
                ptx::fence_proxy_async_global();
                __threadfence();
                pass_turn(kp, tile, split);
            } else {
                ptx::bulk_wait_read_all();
            }
        }
        SGB_TRACE(kp, et == 0, 8);
        return;
    }

    // K % 4 != 0: row-per-thread stores (split 0 / no split) or read-add-write
    // (later splits, in turn).
    if (serial && split > 0) {
        if (et == 0) *sm.epi_go = wait_turn(kp, tile, split, sm.abort_flag) ? 1u : 0u;
        ptx::named_bar_sync(1, EPI_THREADS);
        if (!*sm.epi_go) return;
    }
    const bool accumulate = split > 0;
    float* yrow = kp.y + static_cast<int64_t>(row_ok ? m : 0) * kp.K;
#pragma unroll 1
    for (int j = 0; j < BN / 32; ++j) {
        uint32_t v[32];
        ptx::tmem_ld_32x32b_x32(taddr + j * 32, v);
        ptx::tmem_ld_wait();
        if (!row_ok) continue;
        const int nb = n0 + j * 32;
        float old[32];
        if (accumulate) {
#pragma unroll
            for (int e = 0; e < 32; ++e) old[e] = nb + e < kp.K ? yrow[nb + e] : 0.0f;
        }
#pragma unroll
        for (int e = 0; e < 32; ++e) {
            const int n = nb + e;
            if (n >= kp.K) break;
            float o = __uint_as_float(v[e]);
            if (add_bias) o += __ldg(kp.bias + n);
            if (accumulate) o = old[e] + o;
            yrow[n] = o;
        }
    }
    if (serial) {
        __threadfence();
        ptx::named_bar_sync(1, EPI_THREADS);
        if (et == 0) pass_turn(kp, tile, split);
    }
    SGB_TRACE(kp, et == 0, 8);
}

// ---------------------------------------------------------------- the kernel
template <int BN, int LOADER>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    conv2d_fwd_tc_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                         const __grid_constant__ CUtensorMap tm_y, const ConvKernelParams kp)
{
    using Cfg = TileConfig<BN>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    SmemView sm;
    sm.a = smem;
    sm.b = smem + Cfg::STAGES * A_STAGE_BYTES;
    sm.full = reinterpret_cast<uint64_t*>(smem + Cfg::RING_BYTES);
    sm.empty = sm.full + Cfg::STAGES;
    sm.acc_full = sm.empty + Cfg::STAGES;
    sm.tmem_slot = reinterpret_cast<uint32_t*>(sm.acc_full + 1);
    sm.abort_flag = sm.tmem_slot + 1;
    sm.epi_go = sm.tmem_slot + 2;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int tiles = kp.m_tiles * kp.n_tiles;
    // Split-major block order: every split-j CTA has a lower id than any
    // split-(j+1) CTA, so a tile's predecessors are scheduled first.
    const int split = blockIdx.x / tiles;
    const int tile = blockIdx.x - split * tiles;
    const int m_tile = tile / kp.n_tiles;
    const int n_tile = tile - m_tile * kp.n_tiles;
    const int m0 = m_tile * BM;
    const int n0 = n_tile * BN;
    const int kb_begin = static_cast<int>(static_cast<int64_t>(split) * kp.num_kb / kp.splits);
    const int kb_end = static_cast<int>(static_cast<int64_t>(split + 1) * kp.num_kb / kp.splits);
    const int nkb = kb_end - kb_begin;
    SGB_TRACE(kp, threadIdx.x == 0, 0);

    if (threadIdx.x == 0) {
        const uint32_t full_count =
            LOADER == LOADER_TMA ? 1u : (LOADER == LOADER_CPASYNC ? 1u + EPI_THREADS : EPI_THREADS);
        for (int i = 0; i < Cfg::STAGES; ++i) {
            ptx::mbar_init(&sm.full[i], full_count);
            ptx::mbar_init(&sm.empty[i], 1);
        }
        ptx::mbar_init(sm.acc_full, 1);
        *sm.abort_flag = 0u;
        *sm.epi_go = 0u;
        ptx::mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        if (LOADER == LOADER_TMA) ptx::prefetch_tensormap(&tm_a);
        if (LOADER != LOADER_SCALAR) ptx::prefetch_tensormap(&tm_b);
        if (kp.use_tma_store) ptx::prefetch_tensormap(&tm_y);
    }
    if (warp == 1) {
        ptx::tmem_alloc(sm.tmem_slot, Cfg::TMEM_COLS);
        ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    __syncthreads();
    ptx::tc_fence_after();
    const uint32_t tmem_base = *sm.tmem_slot;
    // Everything above touches only shared memory, tensor memory and kernel
    // parameters, so it may overlap the previous kernel in the stream.  Global
    // memory (inputs it may have written, y and the workspace it may still read)
    // is touched only after this wait.
    ptx::grid_launch_dependents();
    ptx::grid_dependency_wait();
    SGB_TRACE(kp, threadIdx.x == 0, 1);

    if (warp == 0) {
        if (lane == 0 && LOADER != LOADER_SCALAR)
            run_tma_producer<BN, LOADER>(&tm_a, &tm_b, kp, sm, m0, n0, kb_begin, nkb);
    } else if (warp == 1) {
        if (lane == 0) run_mma_issuer<BN>(kp, sm, tmem_base, nkb);
    } else {
        if (LOADER == LOADER_CPASYNC) run_gather_cpasync<BN>(kp, sm, m0, kb_begin, nkb);
        if (LOADER == LOADER_SCALAR) run_gather_scalar<BN>(kp, sm, m0, n0, kb_begin, nkb);
        SGB_TRACE(kp, threadIdx.x == EPI_THREAD0, 9);
        run_epilogue<BN>(&tm_y, kp, sm, tmem_base, m0, n0, split, tile);
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

// Host-side launcher for one instantiation; explicitly instantiated in one
// translation unit per tile width so that the variants compile in parallel.
template <int BN, int LOADER>
cudaError_t launch_conv2d_tc(const CUtensorMap& tm_a, const CUtensorMap& tm_b, const CUtensorMap& tm_y,
                             const ConvKernelParams& kp, int grid, cudaStream_t stream)
{
    auto kern = conv2d_fwd_tc_kernel<BN, LOADER>;
    constexpr int smem = TileConfig<BN>::SMEM_BYTES;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    // The dynamic shared-memory opt-in is per device; remember which devices have it.
    static unsigned long long configured = 0ull;
    const unsigned long long bit = dev < 64 ? (1ull << dev) : 0ull;
    if (!bit || !(__atomic_load_n(&configured, __ATOMIC_ACQUIRE) & bit)) {
        err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (err != cudaSuccess) return err;
        if (bit) __atomic_fetch_or(&configured, bit, __ATOMIC_RELEASE);
    }
    // Programmatic stream serialization: this launch may start while the
    // previous kernel in the stream drains; the kernel waits for it (see
    // grid_dependency_wait) before touching global memory.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(NUM_THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl_enabled() ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tm_a, tm_b, tm_y, kp);
}

#define SGB_LAUNCH_SIG(BN_, L_)                                                                                  \
    cudaError_t launch_conv2d_tc<BN_, L_>(const CUtensorMap&, const CUtensorMap&, const CUtensorMap&,          \
                                          const ConvKernelParams&, int, cudaStream_t)

#define SGB_INSTANTIATE_CONV2D(BN_)                 \
    template SGB_LAUNCH_SIG(BN_, LOADER_TMA);       \
    template SGB_LAUNCH_SIG(BN_, LOADER_CPASYNC);   \
    template SGB_LAUNCH_SIG(BN_, LOADER_SCALAR);

// Declarations of the instantiations that live in other translation units.
#define SGB_DECLARE_CONV2D(BN_)                          \
    extern template SGB_LAUNCH_SIG(BN_, LOADER_TMA);     \
    extern template SGB_LAUNCH_SIG(BN_, LOADER_CPASYNC); \
    extern template SGB_LAUNCH_SIG(BN_, LOADER_SCALAR);

}  // namespace sgb
