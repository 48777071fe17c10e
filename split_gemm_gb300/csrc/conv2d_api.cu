// Host side of the C ABI declared in include/conv2d.h: argument validation,
// output shape, the tile / split / loader heuristic, TMA descriptor encoding
// and the kernel launch.  No device memory is allocated here.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "conv2d.h"
#include "conv2d_direct.cuh"
#include "conv2d_kernel.cuh"
#include "conv2d_pair.cuh"
#include "conv2d_rowwin.cuh"

namespace sgb {
SGB_DECLARE_CONV2D(64)
SGB_DECLARE_CONV2D(128)
SGB_DECLARE_CONV2D(256)
SGB_DECLARE_CONV2D_BOX256(64)
SGB_DECLARE_CONV2D_BOX256(128)
extern template SGB_ROWWIN_SIG(64);
extern template SGB_ROWWIN_SIG(128);
extern template SGB_ROWWIN_SIG(256);
extern template SGB_DIRECT_SIG(1);
extern template SGB_DIRECT_SIG(2);
extern template SGB_DIRECT_SIG(4);
extern template SGB_DIRECT_SIG(8);
extern template SGB_DIRECT_SIG(16);
extern template SGB_PAIR_SIG(64, 1);
extern template SGB_PAIR_SIG(128, 1);
extern template SGB_PAIR_SIG(256, 1);
extern template SGB_PAIR_SIG(64, 2);
extern template SGB_PAIR_SIG(128, 2);
extern template SGB_PAIR_SIG(256, 2);
extern template SGB_PAIR_RES_SIG(64, 1);
extern template SGB_PAIR_RES_SIG(128, 1);
extern template SGB_PAIR_RES_SIG(256, 1);
extern template SGB_PAIR_RES_SIG(64, 2);
extern template SGB_PAIR_RES_SIG(128, 2);
extern template SGB_PAIR_RES_SIG(256, 2);
extern template SGB_PAIR_HALO_SIG(64, 2);
extern template SGB_PAIR_HALO_SIG(64, 3);
extern template SGB_PAIR_HALO_SIG(128, 2);
extern template SGB_PAIR_HALO_SIG(128, 3);
extern template SGB_PAIR_HALO_SIG(256, 2);
extern template SGB_PAIR_HALO_RES_SIG(64, 2);
extern template SGB_PAIR_HALO_RES_SIG(64, 3);
extern template SGB_PAIR_HALO_RES_SIG(128, 2);
extern template SGB_PAIR_HALO_RES_SIG(128, 3);
extern template SGB_PAIR_HALO_RES_SIG(256, 2);
}  // namespace sgb

namespace {

using sgb::BK;
constexpr int64_t kMinTileM = 128;  // the narrowest tile height (sizes the semaphore array)

constexpr int64_t kIndexLimit = (int64_t(1) << 31) - 1;
constexpr size_t kStatusBytes = 256;  // status word, padded so the semaphores start 256-B aligned
constexpr unsigned long long kDefaultWaitNs = 1000000000ull;  // 1 s
constexpr long long kSmemDirectLimit = 232448;  // dynamic shared memory one CTA may opt in to

thread_local int g_last_launches = 0;

#ifdef SGB_TRACE_ENABLED
unsigned long long* g_trace = nullptr;  // profiling builds only: per-CTA phase timestamps
#endif

// ------------------------------------------------------------------ shape
struct Shape {
    int64_t n, h, w, c, k, r, s;
    int64_t sh, sw, ph, pw, dh, dw;
    int64_t g, cg, kg;  // groups; input and output channels per group
    int64_t p, q, m, crs;  // crs = R*S*Cg: the reduction length of one output channel
};

int64_t out_extent(int64_t in, int64_t pad, int64_t dil, int64_t ker, int64_t stride)
{
    const int64_t span = dil * (ker - 1) + 1;
    const int64_t room = in + 2 * pad - span;
    if (room < 0) return 0;
    return room / stride + 1;
}

int make_shape(const conv2d_params* prm, Shape* sh)
{
    if (!prm) return CONV2D_ERR_INVALID;
    if (prm->n < 0 || prm->k < 0 || prm->h < 1 || prm->w < 1 || prm->c < 1 || prm->r < 1 || prm->s < 1)
        return CONV2D_ERR_INVALID;
    // Groups split the channels into equal consecutive groups (both C and K).
    if (prm->groups < 1 || prm->c % prm->groups != 0 || prm->k % prm->groups != 0) return CONV2D_ERR_INVALID;
    if (prm->stride_h < 1 || prm->stride_w < 1 || prm->dil_h < 1 || prm->dil_w < 1 || prm->pad_h < 0 ||
        prm->pad_w < 0)
        return CONV2D_ERR_INVALID;
    sh->n = prm->n; sh->h = prm->h; sh->w = prm->w; sh->c = prm->c;
    sh->k = prm->k; sh->r = prm->r; sh->s = prm->s;
    sh->sh = prm->stride_h; sh->sw = prm->stride_w;
    sh->ph = prm->pad_h; sh->pw = prm->pad_w;
    sh->dh = prm->dil_h; sh->dw = prm->dil_w;
    sh->g = prm->groups;
    sh->cg = sh->c / sh->g;
    sh->kg = sh->k / sh->g;
    // Guard the extent arithmetic itself against overflow before using it.
    if (sh->h > kIndexLimit || sh->w > kIndexLimit || sh->r > kIndexLimit || sh->s > kIndexLimit ||
        sh->c > kIndexLimit || sh->n > kIndexLimit || sh->k > kIndexLimit)
        return CONV2D_ERR_UNSUPPORTED;
    sh->p = out_extent(sh->h, sh->ph, sh->dh, sh->r, sh->sh);
    sh->q = out_extent(sh->w, sh->pw, sh->dw, sh->s, sh->sw);
    if (sh->p < 1 || sh->q < 1) return CONV2D_ERR_INVALID;
    sh->crs = sh->cg * sh->r * sh->s;
    sh->m = sh->n * sh->p * sh->q;
    // 32-bit device indexing: every element count must fit in int32.
    if (sh->crs > kIndexLimit || sh->n * sh->h * sh->w * sh->c > kIndexLimit || sh->m > kIndexLimit ||
        sh->m * sh->k > kIndexLimit || sh->k * sh->crs > kIndexLimit)
        return CONV2D_ERR_UNSUPPORTED;
    return CONV2D_OK;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ------------------------------------------------------------------ device facts
int sm_count_current()
{
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64 && cached[dev] > 0) return cached[dev];
    int sms = 0;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cached[dev] = sms;
    return sms;
}

// ------------------------------------------------------------------ TMA encoders (driver entry points)
PFN_cuTensorMapEncodeTiled_v12000 g_encode_tiled = nullptr;
PFN_cuTensorMapEncodeIm2col_v12000 g_encode_im2col = nullptr;
std::once_flag g_encode_once;

bool load_encoders()
{
    std::call_once(g_encode_once, [] {
        cudaDriverEntryPointQueryResult q{};
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_tiled = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeIm2col", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode_im2col = reinterpret_cast<PFN_cuTensorMapEncodeIm2col_v12000>(fn);
    });
    return g_encode_tiled != nullptr && g_encode_im2col != nullptr;
}

// im2col-mode TMA limits for a rank-4 tensor: bounding-box corners in [-128, 127],
// per-tap offsets that fit the instruction's offset field, traversal strides <= 8.
bool tma_im2col_eligible(const Shape& s)
{
    if (s.cg % BK != 0) return false;  // each 64-channel box stays inside one group
    const int64_t lo_w = -s.pw, lo_h = -s.ph;
    const int64_t up_w = s.pw - (s.s - 1) * s.dw, up_h = s.ph - (s.r - 1) * s.dh;
    auto in8 = [](int64_t v) { return v >= -128 && v <= 127; };
    if (!in8(lo_w) || !in8(lo_h) || !in8(up_w) || !in8(up_h)) return false;
    if ((s.s - 1) * s.dw > 255 || (s.r - 1) * s.dh > 255) return false;
    if (s.sh > 8 || s.sw > 8) return false;
    return true;
}

// ------------------------------------------------------------------ box loader (tile = rectangle of pixels)
constexpr int kBoxChunks = 2;  // 64-channel chunks (k-blocks) per box, as in the kernel's TileConfig::KC

struct BoxGeom {
    int bw, bh, bn_img, px;      // rectangle: bn_img images x bh rows x bw columns, px pixels
    int q_blocks, p_blocks, n_blocks;
    int64_t m_tiles;
};

// Rectangle of at most bm output pixels for the box loader, or false when the
// shape does not allow one: a box spans at most 256 elements per dimension
// (bw * stride_w, bh * stride_h), the traversal strides are at most 8, and two
// 64-channel chunks must divide C.  The pixel count px needs no rounding: the
// second chunk of a box lands px 128-byte rows after the first, and the
// 128-byte swizzle of both the TMA write and the MMA read follows absolute
// shared-memory addresses, so a chunk may start at any row.
bool box_geometry(const Shape& s, int bm, BoxGeom* g)
{
    if (s.g != 1 || s.c % (kBoxChunks * BK) != 0 || s.sw > 8 || s.sh > 8) return false;
    const int64_t wmax = 256 / s.sw, hmax = 256 / s.sh;
    int64_t bw, bh = 1, bn = 1;
    if (s.q >= bm || s.q > wmax) {
        // Part of one output row per tile, split evenly, rounded up to 8 pixels.
        const int64_t cap = bm < wmax ? bm : wmax;
        const int64_t qb = cdiv(s.q, cap);
        bw = (cdiv(s.q, qb) + 7) / 8 * 8;
        if (bw > cap) bw = cap / 8 * 8;
    } else if (s.p * s.q > bm) {
        // Whole rows: as many as fit, balanced over the row blocks.
        bw = s.q;
        int64_t rows = bm / s.q;
        if (rows > hmax) rows = hmax;
        const int64_t pb = cdiv(s.p, rows);
        bh = cdiv(s.p, pb);
    } else {
        // Whole images.
        bw = s.q;
        bh = s.p;
        bn = bm / (s.p * s.q);
        if (bn > s.n) bn = s.n;
    }
    if (bw < 1 || bh < 1 || bn < 1) return false;
    const int64_t px = bw * bh * bn;
    if (px > bm || bw > wmax || bh > hmax) return false;
    g->bw = static_cast<int>(bw);
    g->bh = static_cast<int>(bh);
    g->bn_img = static_cast<int>(bn);
    g->px = static_cast<int>(px);
    g->q_blocks = static_cast<int>(cdiv(s.q, bw));
    g->p_blocks = static_cast<int>(cdiv(s.p, bh));
    g->n_blocks = static_cast<int>(cdiv(s.n, bn));
    g->m_tiles = static_cast<int64_t>(g->q_blocks) * g->p_blocks * g->n_blocks;
    return true;
}

// ------------------------------------------------------------------ row-window loader (few channels)
constexpr int kSmemLimit = 232448;  // dynamic shared memory one CTA may opt in to

struct RowWinCfg {
    int bn, cp_log2, nch, seg_elems, raw_bytes, T, rt, new_rows, reuse, ncls, nblocks, row_slots, wtmp_filters;
    int cls_k[sgb::RW_MAX_CLASSES], cls_base[sgb::RW_MAX_CLASSES];
    int qblocks, pblocks, tiles;
    uint32_t tmem_cols;
    sgb::RowWinLayout lay;
};

// The row-window kernel's sizes for this shape, or false when it does not
// apply: the padded pixel (Cp = 8 / stride_w channels) must hold C, the window
// must be contiguous along W (dil_w == 1), all K channels must fit one channel
// tile, and the resident weight plus one tile's window rows must fit in shared
// memory.  T output rows share each MMA (T*BN <= 256); T drops to 1 for
// dil_h > 1 or stride_h > 8, and further down while shared memory is short.
bool rowwin_config(const Shape& s, int bn_force, RowWinCfg* o)
{
    if (s.g != 1 || s.dw != 1 || s.r > 64 || s.s > 64 || s.dh > 64) return false;
    int cp_log2;
    switch (s.sw) {
        case 1: cp_log2 = 3; break;
        case 2: cp_log2 = 2; break;
        case 4: cp_log2 = 1; break;
        case 8: cp_log2 = 0; break;
        default: return false;
    }
    const int64_t cp = int64_t(1) << cp_log2;
    if (s.c > cp || s.k > 256) return false;
    const int bn = bn_force ? bn_force : (s.k <= 64 ? 64 : (s.k <= 128 ? 128 : 256));
    if (bn != 64 && bn != 128 && bn != 256) return false;
    if (bn < s.k) return false;
    o->bn = bn;
    o->cp_log2 = cp_log2;
    o->nch = static_cast<int>(cdiv(s.s * cp, 16));
    o->seg_elems = 8 * (sgb::RW_TILE_M - 1) + 16 * o->nch;
    const int64_t segpix = o->seg_elems / cp;
    o->raw_bytes = static_cast<int>((segpix * s.c * 2 + 32 + 15) / 16 * 16);
    o->qblocks = static_cast<int>(cdiv(s.q, sgb::RW_TILE_M));
    const int64_t crs_bytes = s.crs * 2;
    int t_max = 256 / bn;
    if (s.dh != 1 || s.sh > sgb::RW_MAX_CLASSES) t_max = 1;
    if (t_max > s.p) t_max = static_cast<int>(s.p);
    for (int T = t_max; T >= 1; --T) {
        const int64_t rt = (T - 1) * s.sh + (s.r - 1) * s.dh + 1;
        if (rt > 4096) continue;
        // Residue classes of filter rows and their zero-padded block sequences.
        int ncls = T > 1 ? static_cast<int>(s.sh) : 1;
        int nblocks = 0;
        for (int rho = 0; rho < sgb::RW_MAX_CLASSES; ++rho) {
            int k = 0;
            if (rho < ncls) k = T > 1 ? (rho < s.r ? static_cast<int>(cdiv(s.r - rho, s.sh)) : 0) : static_cast<int>(s.r);
            o->cls_k[rho] = k;
            o->cls_base[rho] = nblocks;
            if (k > 0) nblocks += k + 2 * (T - 1);
        }
        const bool reuse = rt > T * s.sh;
        const int new_rows = reuse ? static_cast<int>(T * s.sh) : static_cast<int>(rt);
        // Ring: one tile's window plus two tiles of look-ahead, fewer when shared memory is short.
        // The weight is copied in through an area of its own in one pass when
        // shared memory allows, else through the epilogue staging area in passes.
        const int64_t w_all = (s.k * crs_bytes + 32 + 127) / 128 * 128;
        for (int64_t slots = rt + 2 * new_rows; slots >= rt; --slots) {
            sgb::RowWinLayout lay = sgb::rowwin_layout(bn, o->nch, nblocks, o->seg_elems, static_cast<int>(slots),
                                                       static_cast<int>(rt), o->raw_bytes, static_cast<int>(w_all));
            int64_t wtmp = s.k;
            if (w_all > kSmemLimit || lay.total > kSmemLimit) {
                lay = sgb::rowwin_layout(bn, o->nch, nblocks, o->seg_elems, static_cast<int>(slots),
                                         static_cast<int>(rt), o->raw_bytes, 0);
                wtmp = (4 * sgb::RW_EPI_SLOT_BYTES - 32) / crs_bytes;
            }
            if (lay.total > kSmemLimit) continue;
            if (wtmp < 1) break;
            o->T = T;
            o->rt = static_cast<int>(rt);
            o->new_rows = new_rows;
            o->reuse = reuse ? 1 : 0;
            o->ncls = ncls;
            o->nblocks = nblocks;
            o->row_slots = static_cast<int>(slots);
            o->wtmp_filters = static_cast<int>(wtmp < 256 ? wtmp : 256);
            o->pblocks = static_cast<int>(cdiv(s.p, T));
            o->tiles = static_cast<int>(s.n * o->qblocks * o->pblocks);
            uint32_t cols = 32;
            while (cols < static_cast<uint32_t>(2 * T * bn)) cols <<= 1;
            o->tmem_cols = cols;
            o->lay = lay;
            return true;
        }
    }
    return false;
}

// ------------------------------------------------------------------ heuristic
// ------------------------------------------------------------------ halo loader (stride 1)
// Each image is a grid of virtual pixels with the padded row pitch wv = W + 2*pw;
// a tile is 128 consecutive virtual pixels of one image and, per 64-channel
// chunk, one tiled TMA box of hr whole padded input rows holds every filter
// tap's operand (the kernel header describes the layout).
struct HaloGeom {
    int64_t m_tiles;
    int wv, vp, tpi, hr, halo_bytes;
    int taps;  // CTA-pair halo loader: filter taps per pipeline stage (0 otherwise)
};  // no padding bytes: the tensor-map cache compares keys bytewise

// Halo geometry for output-channel tile width bn, or false when the shape does
// not allow the halo loader: stride 1, C % 64 == 0, a padded row of at most 256
// pixels (a TMA box dimension), and the ring plus two halo buffers within the
// per-block shared memory.
bool halo_geometry(const Shape& s, int bn, HaloGeom* g)
{
    if (s.g != 1 || s.sh != 1 || s.sw != 1 || s.c % BK != 0) return false;
    const int64_t wv = s.w + 2 * s.pw;
    if (wv > 256 || s.p < 1) return false;
    const int64_t vp = s.p * wv;
    // Highest halo row any tap of any tile reads: the tile may start up to wv - 1
    // pixels into its first padded row.
    const int64_t max_row = (wv - 1) + (s.r - 1) * s.dh * wv + (s.s - 1) * s.dw + (kMinTileM - 1);
    const int64_t hr = max_row / wv + 1;
    if (hr > 256) return false;
    const int64_t halo_bytes = (hr * wv * 128 + 1023) / 1024 * 1024;
    int fixed;
    if (bn == 64) fixed = sgb::conv2d_tc_smem_bytes<128, 64, sgb::LOADER_HALO>(0);
    else if (bn == 128) fixed = sgb::conv2d_tc_smem_bytes<128, 128, sgb::LOADER_HALO>(0);
    else if (bn == 256) fixed = sgb::conv2d_tc_smem_bytes<128, 256, sgb::LOADER_HALO>(0);
    else return false;
    if (fixed + 2 * halo_bytes > sgb::kMaxSmemBytes) return false;
    const int64_t tpi = cdiv(vp, kMinTileM);
    if (s.n * tpi > 2147483647ll / 1024) return false;
    g->wv = static_cast<int>(wv);
    g->vp = static_cast<int>(vp);
    g->tpi = static_cast<int>(tpi);
    g->hr = static_cast<int>(hr);
    g->halo_bytes = static_cast<int>(halo_bytes);
    g->m_tiles = s.n * tpi;
    g->taps = 0;
    return true;
}

struct Plan {
    int block_m;
    int block_n;
    int splits;  // classic split-K factor, or 0 for stream-K
    int loader;
    int m_tiles, n_tiles, num_kb;  // num_kb: pipeline stages per tile (two k-blocks each for the box loader)
    int grid;         // CTAs launched
    long long units;  // (tile, stage) work units
    BoxGeom box;      // box loader only
    HaloGeom halo;    // halo loader only
    int kbs;          // CTA-pair loaders: 64-wide k-blocks (filter taps for the halo loader) per pipeline stage
    int unit_offset;  // CTA-pair loaders only: rotation of the pairs' unit ranges
};

// Semaphores the workspace holds: one per tile of the smallest tiles any plan
// uses (128-pixel rows of M, or the box loader's 128-pixel rectangles, by
// 64 output channels).
int64_t semaphore_capacity(const Shape& s)
{
    int64_t m_tiles = cdiv(s.m, kMinTileM);
    BoxGeom g;
    if (box_geometry(s, 128, &g) && g.m_tiles > m_tiles) m_tiles = g.m_tiles;
    HaloGeom h;
    if (halo_geometry(s, 64, &h) && h.m_tiles > m_tiles) m_tiles = h.m_tiles;
    // CTA-pair halo loader: one semaphore per 128-pixel row-block of every image.
    if (s.sh == 1 && s.sw == 1 && s.w + 2 * s.pw <= 256 && s.p >= 1) {
        const int64_t rb = s.n * cdiv(s.p * (s.w + 2 * s.pw), kMinTileM);
        if (rb > m_tiles) m_tiles = rb;
    }
    return m_tiles * s.g * cdiv(s.kg, 64);
}


constexpr int kMinUnitsPerCta = 4;     // no split gets fewer k-blocks than this
constexpr int kMaxSplitsPerTile = 6;   // longest serial in-place reduction chain the heuristic builds

// ------------------------------------------------------------------ direct kernel (groups of few channels)
// C/groups == K/groups in {1, 2, 4, 8, 16} with groups > 1: the implicit GEMM would
// fill CG of each 64-wide column block, so a CUDA-core kernel takes these shapes.
int direct_chunk(int64_t cg) { return cg == 16 ? 16 : 8; }   // channels per thread (DirectCfg::CH)
int direct_px(int64_t cg) { return cg == 16 ? 2 : 4; }       // output pixels per thread (DirectCfg::PX)

// Threads of the direct kernel: one per (image, output row, block of PX pixels, channel chunk).
int64_t direct_items(const Shape& s)
{
    return s.n * s.p * cdiv(s.q, direct_px(s.cg)) * (s.c / direct_chunk(s.cg));
}

bool direct_eligible(const Shape& s)
{
    if (s.g < 2 || s.cg != s.kg) return false;
    if (s.cg != 1 && s.cg != 2 && s.cg != 4 && s.cg != 8 && s.cg != 16) return false;
    if (s.c % direct_chunk(s.cg) != 0) return false;  // whole 16-byte chunks of whole groups
    if (direct_items(s) > 2147483647ll) return false;
    return sgb::conv2d_direct_smem_bytes((int)s.k, (int)s.r, (int)s.s, (int)s.cg) <= kSmemDirectLimit;
}

// CTAs of the direct kernel: as many per SM as shared memory and the thread limit
// allow (each stages every group weight), enough to cover the items once.
int64_t direct_grid(const Shape& s)
{
    const long long smem = sgb::conv2d_direct_smem_bytes((int)s.k, (int)s.r, (int)s.s, (int)s.cg);
    const long long nsm = sm_count_current() > 0 ? sm_count_current() : 1;
    long long per_sm = smem > 0 ? kSmemDirectLimit / smem : 8;
    if (per_sm > 2048 / sgb::DIRECT_THREADS) per_sm = 2048 / sgb::DIRECT_THREADS;
    if (per_sm < 1) per_sm = 1;
    long long grid = cdiv(direct_items(s), sgb::DIRECT_THREADS);
    if (grid > nsm * per_sm) grid = nsm * per_sm;
    return grid < 1 ? 1 : grid;
}

// Nothing forced but what every path accepts (wait bound, reduction, test hooks).
bool nothing_forced(const conv2d_algo* a)
{
    return !a || (a->loader == CONV2D_LOADER_AUTO && a->splits == 0 && a->grid == 0 && a->block_n == 0 &&
                  a->block_m == 0);
}

// whole_tiles: where the heuristic would divide many tiles stream-K style over
// the SMs, give every CTA whole tiles instead.  A fused epilogue (bf16 output,
// activation) asks for it: its cut tiles take a detour through an fp32 buffer.
// ------------------------------------------------------------------ CTA-pair plans
bool plan_cuts_tiles(const Plan& p);

// The CTA-pair kernel (conv2d_pair.cuh): 256-pixel tiles on clusters of two
// CTAs, TMA im2col loads of 128 pixels per CTA, 16-byte vector stores.
// The im2col pair kernel: C/groups % 64 == 0 (im2col boxes inside one group), K/groups % 4 == 0
// (16-byte stores inside one group's columns); the halo pair kernel adds its own
// geometry conditions (halo_pair_geometry).
bool pair_eligible(const Shape& s) { return tma_im2col_eligible(s) && s.kg % 4 == 0; }

int pair_max_resident(int bn, int kbs, bool fused)
{
    if (kbs == 1) {
        if (bn == 64) return sgb::conv2d_pair_max_resident<64, 1>(fused);
        if (bn == 128) return sgb::conv2d_pair_max_resident<128, 1>(fused);
        if (bn == 256) return sgb::conv2d_pair_max_resident<256, 1>(fused);
    } else {
        if (bn == 64) return sgb::conv2d_pair_max_resident<64, 2>(fused);
        if (bn == 128) return sgb::conv2d_pair_max_resident<128, 2>(fused);
        if (bn == 256) return sgb::conv2d_pair_max_resident<256, 2>(fused);
    }
    return 0;
}

cudaError_t launch_pair(int bn, int kbs, const CUtensorMap& a, const CUtensorMap& b, const sgb::ConvKernelParams& kp,
                        int pairs, cudaStream_t st)
{
    if (kbs == 1) {
        if (bn == 64) return sgb::launch_conv2d_pair<64, 1>(a, b, kp, pairs, st);
        if (bn == 128) return sgb::launch_conv2d_pair<128, 1>(a, b, kp, pairs, st);
        if (bn == 256) return sgb::launch_conv2d_pair<256, 1>(a, b, kp, pairs, st);
    } else {
        if (bn == 64) return sgb::launch_conv2d_pair<64, 2>(a, b, kp, pairs, st);
        if (bn == 128) return sgb::launch_conv2d_pair<128, 2>(a, b, kp, pairs, st);
        if (bn == 256) return sgb::launch_conv2d_pair<256, 2>(a, b, kp, pairs, st);
    }
    return cudaErrorInvalidValue;
}

// Stream-K over every resident pair when the reduction gives each pair at least
// this many two-k-block stages (the cut tiles' in-place adds are then a small
// share of the work); otherwise whole tiles.
constexpr int64_t kPairStreamKStages = 8;
constexpr int64_t PAIR_KBS_NORM = 2;  // units count stages of kbs k-blocks; the threshold counts pairs of k-blocks
constexpr int64_t PAIR_M_SLACK = 512;  // pixel indices up to one tile past M are decoded

// Rotation of the pairs' unit ranges (see PairWalker): the offset d, 0 < d <
// stages, for which no range [floor(c*U/G) + d, ...) starts on a tile boundary
// (a multiple of `stages`), searched outward from half a range; 0 when the plan
// cuts no tile or no offset works.
int64_t choose_unit_offset(int64_t units, int64_t grid, int64_t stages)
{
    if (grid <= 1 || stages <= 1 || (units % grid == 0 && (units / grid) % stages == 0)) return 0;
    auto ok = [&](int64_t d) {
        for (int64_t c = 0; c < grid; ++c)
            if ((c * units / grid + d) % stages == 0) return false;
        return true;
    };
    const int64_t mid = units / grid / 2 < stages ? units / grid / 2 : stages / 2;
    for (int64_t step = 0; step < stages; ++step) {
        if (mid + step >= 1 && mid + step < stages && ok(mid + step)) return mid + step;
        if (mid - step >= 1 && mid - step < stages && ok(mid - step)) return mid - step;
    }
    return 0;
}

int choose_pair_plan(const Shape& s, const conv2d_algo* force, Plan* plan, bool whole_tiles)
{
    if (!pair_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    if (force && force->block_m != 0 && force->block_m != sgb::PAIR_TILE_M) return CONV2D_ERR_UNSUPPORTED;
    int bn = force && force->block_n ? force->block_n : (s.kg <= 64 ? 64 : (s.kg <= 128 ? 128 : 256));
    if (bn != 64 && bn != 128 && bn != 256) return CONV2D_ERR_INVALID;
    // Stage depth: two k-blocks per stage (three 64 KB stages at block_n = 256, one
    // producer thread per operand): 1.5 TMA operations per k-block against 2 with one
    // k-block per stage, and the SM's TMA unit completes about one operation per
    // ~0.17 us, so the deeper stages measured faster.  A measurement hook forces one.
    const int dbg = force ? force->debug_flags : 0;
    const int kbs = (dbg & CONV2D_DEBUG_PAIR_KB1) ? 1 : 2;
    const int64_t m_tiles = cdiv(s.m, sgb::PAIR_TILE_M);
    const int64_t n_tiles = s.g * cdiv(s.kg, bn);  // column blocks never straddle a group
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t stages = cdiv(s.crs / BK, kbs);
    const int64_t units = tiles * stages;
    const int64_t resident = pair_max_resident(bn, kbs, whole_tiles);
    if (resident <= 0) return CONV2D_ERR_CUDA;
    const int64_t fsplits = force ? force->splits : 0;
    const int64_t fgrid = force ? force->grid : 0;
    if (fsplits < 0 || fgrid < 0 || (fsplits > 0 && fgrid > 0)) return CONV2D_ERR_INVALID;
    int64_t grid;
    if (fsplits > 0) {
        if (fsplits > stages) return CONV2D_ERR_UNSUPPORTED;  // every split needs at least one stage
        grid = tiles * fsplits;
    } else if (fgrid > 0) {
        if (fgrid > units) return CONV2D_ERR_UNSUPPORTED;
        grid = fgrid;
    } else if (!whole_tiles && units * kbs >= kPairStreamKStages * PAIR_KBS_NORM * resident) {
        grid = resident;
    } else {
        // Whole tiles: the smallest even share of at least tiles/resident tiles per pair.
        const int64_t per = cdiv(tiles, resident);
        grid = tiles;
        for (int64_t d = per; d <= 2 * per; ++d)
            if (tiles % d == 0) {
                grid = tiles / d;
                break;
            }
    }
    // The kernel splits the work with 32-bit arithmetic (FastDiv, n < 2^31).
    const int64_t offset = choose_unit_offset(units, grid, stages);
    if ((units + offset + 1) * (grid + 1) >= (int64_t(1) << 31) || s.m >= (int64_t(1) << 31) - PAIR_M_SLACK)
        return CONV2D_ERR_UNSUPPORTED;
    plan->block_m = sgb::PAIR_TILE_M;
    plan->block_n = bn;
    plan->splits = static_cast<int>(fsplits);
    plan->loader = CONV2D_LOADER_TMA_PAIR;
    plan->m_tiles = static_cast<int>(m_tiles);
    plan->n_tiles = static_cast<int>(n_tiles);
    plan->num_kb = static_cast<int>(stages);
    plan->grid = static_cast<int>(grid);
    plan->units = units;
    plan->box = BoxGeom{};
    plan->halo = HaloGeom{};
    plan->kbs = kbs;
    plan->unit_offset = static_cast<int>(offset);
    if (plan_cuts_tiles(*plan)) {
        // A later split waits for an earlier one: every pair must be resident at once.
        if (grid > resident) return CONV2D_ERR_UNSUPPORTED;
        // bf16 output cannot carry partial sums (and ReLU needs the whole sum).
        if (whole_tiles) return CONV2D_ERR_UNSUPPORTED;
    }
    return CONV2D_OK;
}

// Shared memory of the CTA-pair halo kernel for tile width bn, taps per stage
// and halo buffer size (0 for a combination that is not instantiated).
int pair_halo_smem(int bn, int taps, int halo_bytes)
{
    if (taps == 3) {
        if (bn == 64) return sgb::conv2d_pair_halo_smem_bytes<64, 3>(halo_bytes);
        if (bn == 128) return sgb::conv2d_pair_halo_smem_bytes<128, 3>(halo_bytes);
        return 0;
    }
    if (taps != 2) return 0;
    if (bn == 64) return sgb::conv2d_pair_halo_smem_bytes<64, 2>(halo_bytes);
    if (bn == 128) return sgb::conv2d_pair_halo_smem_bytes<128, 2>(halo_bytes);
    if (bn == 256) return sgb::conv2d_pair_halo_smem_bytes<256, 2>(halo_bytes);
    return 0;
}

// The CTA-pair halo loader: geometry (row pitch, row-blocks, halo rows and
// bytes, taps per stage) for tile width bn, or false when the shape does not
// allow it.  Stages hold three taps where the ring still fits beside the two
// halo buffers (64- and 128-wide tiles), else two.  Groups need Cg, the chunked
// reduction of one group, to be whole 64-channel chunks.
bool halo_pair_geometry(const Shape& s, int bn, HaloGeom* g)
{
    if (s.sh != 1 || s.sw != 1 || s.cg % BK != 0 || s.kg % 4 != 0 || s.p < 1) return false;
    const int64_t wv = s.w + 2 * s.pw;
    if (wv > 256) return false;
    const int64_t vp = s.p * wv;
    const int64_t max_row = (wv - 1) + (s.r - 1) * s.dh * wv + (s.s - 1) * s.dw + (sgb::PAIR_ROWS - 1);
    const int64_t hr = max_row / wv + 1;
    if (hr > 256) return false;
    const int64_t halo_bytes = (hr * wv * 128 + 1023) / 1024 * 1024;
    if (bn != 64 && bn != 128 && bn != 256) return false;
    int taps = bn == 256 ? 2 : 3;
    if (pair_halo_smem(bn, taps, static_cast<int>(halo_bytes)) > sgb::kMaxSmemBytes) taps = 2;
    if (pair_halo_smem(bn, taps, static_cast<int>(halo_bytes)) > sgb::kMaxSmemBytes) return false;
    const int64_t tpi = cdiv(vp, sgb::PAIR_ROWS);
    if (s.n * tpi > 2147483647ll / 1024) return false;
    g->wv = static_cast<int>(wv);
    g->vp = static_cast<int>(vp);
    g->tpi = static_cast<int>(tpi);
    g->hr = static_cast<int>(hr);
    g->halo_bytes = static_cast<int>(halo_bytes);
    g->m_tiles = cdiv(s.n, 2) * tpi;  // a tile is one row-block of two images
    g->taps = taps;
    return true;
}

int pair_halo_max_resident(int bn, int taps, bool fused, int halo_bytes)
{
    const int smem = pair_halo_smem(bn, taps, halo_bytes);
    if (smem <= 0) return 0;
    if (taps == 3) {
        if (bn == 64) return sgb::conv2d_pair_halo_max_resident<64, 3>(fused, smem);
        if (bn == 128) return sgb::conv2d_pair_halo_max_resident<128, 3>(fused, smem);
        return 0;
    }
    if (bn == 64) return sgb::conv2d_pair_halo_max_resident<64, 2>(fused, smem);
    if (bn == 128) return sgb::conv2d_pair_halo_max_resident<128, 2>(fused, smem);
    if (bn == 256) return sgb::conv2d_pair_halo_max_resident<256, 2>(fused, smem);
    return 0;
}

cudaError_t launch_pair_halo(int bn, int taps, const CUtensorMap& a, const CUtensorMap& b,
                             const sgb::ConvKernelParams& kp, int pairs, cudaStream_t stream)
{
    if (taps == 3) {
        if (bn == 64) return sgb::launch_conv2d_pair_halo<64, 3>(a, b, kp, pairs, stream);
        if (bn == 128) return sgb::launch_conv2d_pair_halo<128, 3>(a, b, kp, pairs, stream);
        return cudaErrorInvalidValue;
    }
    if (bn == 64) return sgb::launch_conv2d_pair_halo<64, 2>(a, b, kp, pairs, stream);
    if (bn == 128) return sgb::launch_conv2d_pair_halo<128, 2>(a, b, kp, pairs, stream);
    if (bn == 256) return sgb::launch_conv2d_pair_halo<256, 2>(a, b, kp, pairs, stream);
    return cudaErrorInvalidValue;
}

int choose_pair_halo_plan(const Shape& s, const conv2d_algo* force, Plan* plan, bool whole_tiles)
{
    if (force && force->block_m != 0 && force->block_m != sgb::PAIR_TILE_M) return CONV2D_ERR_UNSUPPORTED;
    int bn = force && force->block_n ? force->block_n : (s.kg <= 64 ? 64 : (s.kg <= 128 ? 128 : 256));
    if (bn != 64 && bn != 128 && bn != 256) return CONV2D_ERR_INVALID;
    HaloGeom g;
    if (!halo_pair_geometry(s, bn, &g)) return CONV2D_ERR_UNSUPPORTED;
    const int64_t m_tiles = g.m_tiles;
    const int64_t n_tiles = s.g * cdiv(s.kg, bn);  // column blocks within each group
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t stages = (s.cg / BK) * cdiv(s.r * s.s, g.taps);  // chunk-major
    const int64_t units = tiles * stages;
    const int64_t resident = pair_halo_max_resident(bn, g.taps, whole_tiles, g.halo_bytes);
    if (resident <= 0) return CONV2D_ERR_CUDA;
    const int64_t fsplits = force ? force->splits : 0;
    const int64_t fgrid = force ? force->grid : 0;
    if (fsplits < 0 || fgrid < 0 || (fsplits > 0 && fgrid > 0)) return CONV2D_ERR_INVALID;
    int64_t grid;
    if (fsplits > 0) {
        if (fsplits > stages) return CONV2D_ERR_UNSUPPORTED;
        grid = tiles * fsplits;
    } else if (fgrid > 0) {
        if (fgrid > units) return CONV2D_ERR_UNSUPPORTED;
        grid = fgrid;
    } else if (!whole_tiles && units * 2 >= kPairStreamKStages * PAIR_KBS_NORM * resident) {
        grid = resident;
    } else {
        const int64_t per = cdiv(tiles, resident);
        grid = tiles;
        for (int64_t d = per; d <= 2 * per; ++d)
            if (tiles % d == 0) {
                grid = tiles / d;
                break;
            }
    }
    const int64_t offset = choose_unit_offset(units, grid, stages);
    if ((units + offset + 1) * (grid + 1) >= (int64_t(1) << 31)) return CONV2D_ERR_UNSUPPORTED;
    plan->block_m = sgb::PAIR_TILE_M;
    plan->block_n = bn;
    plan->splits = static_cast<int>(fsplits);
    plan->loader = CONV2D_LOADER_PAIR_HALO;
    plan->unit_offset = static_cast<int>(offset);
    plan->m_tiles = static_cast<int>(m_tiles);
    plan->n_tiles = static_cast<int>(n_tiles);
    plan->num_kb = static_cast<int>(stages);
    plan->grid = static_cast<int>(grid);
    plan->units = units;
    plan->box = BoxGeom{};
    plan->halo = g;
    plan->kbs = g.taps;
    if (plan_cuts_tiles(*plan)) {
        if (grid > resident) return CONV2D_ERR_UNSUPPORTED;
        if (whole_tiles) return CONV2D_ERR_UNSUPPORTED;
    }
    return CONV2D_OK;
}

// The heuristic's CTA-pair choices (loader AUTO with no shape field forced), in
// the two regimes where the pair kernels measured faster than the single-CTA
// kernel on GB300; anything else returns CONV2D_ERR_UNSUPPORTED and the
// single-CTA planner decides.
//  - Few output tiles and a long reduction (split-K): 256-pixel pair tiles, each
//    tile cut into an equal number of splits so that tiles x splits fills the
//    resident pairs (every pair computes one segment and reduces it once), each
//    split at least 8 stages long; only when the 256-row tiles waste at most 35%
//    of their rows and the epilogue is not fused (a fused epilogue needs whole
//    tiles).
//  - Whole-tile stride-1 ungrouped layers with at least 128 input channels whose halo
//    tiles fill at least 70% of the resident pairs' waves and whose
//    virtual pixels (padded row pitch, image pairs) exceed the output pixels by
//    at most 20%: the halo loader, whole tiles (a single wave of 256-wide tiles
//    as two 128-wide halves per pair).
//  - Otherwise, where the pair tiles cover at least half the resident pairs
//    (and waste at most 35% of their rows): the im2col pair loader.  Grouped
//    layers stay on it: with 64-wide group tiles the halo kernel's MMAs and stage
//    handshakes (35-40 ns per 256x64x16 MMA) set the same pace as the im2col
//    kernel's activation loads, and its virtual pixels add 14% on a 28x28 layer.
int choose_auto_pair(const Shape& s, const conv2d_algo* force, Plan* plan, bool whole_tiles)
{
    if (!pair_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    conv2d_algo f;
    std::memset(&f, 0, sizeof(f));
    if (force) f = *force;
    const int bn = s.kg <= 64 ? 64 : (s.kg <= 128 ? 128 : 256);
    const int64_t col_blocks = s.g * cdiv(s.kg, bn);
    if (!whole_tiles) {
        const int64_t m_tiles = cdiv(s.m, sgb::PAIR_TILE_M);
        const int64_t tiles = m_tiles * col_blocks;
        const int64_t stages = cdiv(s.crs / BK, 2);
        const int64_t res = pair_max_resident(bn, 2, false);
        if (res > 0 && tiles * 2 <= res && stages >= 16 && m_tiles * sgb::PAIR_TILE_M * 20 <= s.m * 27) {
            int64_t splits = res / tiles;
            if (splits > stages / 8) splits = stages / 8;
            if (splits >= 2) {
                f.loader = CONV2D_LOADER_TMA_PAIR;
                f.block_n = bn;
                f.splits = static_cast<int32_t>(splits);
                if (choose_pair_plan(s, &f, plan, false) == CONV2D_OK) return CONV2D_OK;
            }
        }
    }
    HaloGeom g;
    if (s.g == 1 && s.c >= 128 && halo_pair_geometry(s, bn, &g)) {
        const int64_t tiles = g.m_tiles * col_blocks;
        const int64_t res = pair_halo_max_resident(bn, g.taps, whole_tiles, g.halo_bytes);
        const int64_t virt = cdiv(s.n, 2) * 2 * static_cast<int64_t>(g.tpi) * sgb::PAIR_ROWS;
        if (res > 0) {
            const int64_t waves = cdiv(tiles, res);
            if (tiles * 10 >= waves * res * 7 && virt * 5 <= s.m * 6) {
                f.loader = CONV2D_LOADER_PAIR_HALO;
                f.block_n = bn;
                f.splits = 0;
                f.grid = 0;
                // One 256-wide tile per pair in a single wave: two 128-wide halves instead, which
                // the planner gives to the same pair one after the other, so that the first
                // half's epilogue overlaps the second half's main loop and the exposed tail
                // halves (28 x 28 layer: 16.88 against 17.04 us per launch).
                HaloGeom g2;
                if (bn == 256 && tiles <= res && halo_pair_geometry(s, 128, &g2) &&
                    pair_halo_max_resident(128, g2.taps, whole_tiles, g2.halo_bytes) >= tiles)
                    f.block_n = 128;
                if (choose_pair_halo_plan(s, &f, plan, true) == CONV2D_OK) return CONV2D_OK;
            }
        }
    }
    // Otherwise the im2col pair kernel with its own schedule, where its 256-row tiles
    // cover at least half the resident pairs and waste at most 35% of their rows.
    const int64_t m_tiles = cdiv(s.m, sgb::PAIR_TILE_M);
    const int64_t res = pair_max_resident(bn, 2, whole_tiles);
    if (res > 0 && m_tiles * col_blocks * 2 >= res && m_tiles * sgb::PAIR_TILE_M * 20 <= s.m * 27) {
        f.loader = CONV2D_LOADER_TMA_PAIR;
        f.block_n = bn;
        f.splits = 0;
        f.grid = 0;
        if (choose_pair_plan(s, &f, plan, whole_tiles) == CONV2D_OK) return CONV2D_OK;
    }
    return CONV2D_ERR_UNSUPPORTED;
}

int choose_plan(const Shape& s, const conv2d_algo* force, Plan* plan, bool whole_tiles = false)
{
    const int sms = sm_count_current();
    if (!force || (force->loader == CONV2D_LOADER_AUTO && force->block_m == 0 && force->block_n == 0 &&
                   force->splits == 0 && force->grid == 0)) {
        if (choose_auto_pair(s, force, plan, whole_tiles) == CONV2D_OK) return CONV2D_OK;
    }
    // Loader.
    int loader = force ? force->loader : 0;
    RowWinCfg rw;
    if (loader == CONV2D_LOADER_AUTO) {
        // The halo loader (CONV2D_LOADER_HALO) moves fewer bytes and issues fewer
        // TMA operations, but measured slower than the im2col loader on every
        // stride-1 benchmark shape (its per-stage weight loads see a longer ring
        // round trip), so the heuristic does not pick it; callers may force it.
        if (tma_im2col_eligible(s)) loader = CONV2D_LOADER_TMA_IM2COL;
        else if (s.cg % 8 == 0) loader = CONV2D_LOADER_CPASYNC;
        else if (rowwin_config(s, force ? force->block_n : 0, &rw)) loader = CONV2D_LOADER_ROW_WINDOW;
        else loader = CONV2D_LOADER_SCALAR;
    } else if (loader == CONV2D_LOADER_ROW_WINDOW) {
        if (!rowwin_config(s, force->block_n, &rw)) return CONV2D_ERR_UNSUPPORTED;
    } else if (loader == CONV2D_LOADER_TMA_IM2COL) {
        if (!tma_im2col_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    } else if (loader == CONV2D_LOADER_CPASYNC) {
        if (s.cg % 8 != 0) return CONV2D_ERR_UNSUPPORTED;
    } else if (loader == CONV2D_LOADER_HYBRID) {
        if (!tma_im2col_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    } else if (loader == CONV2D_LOADER_TMA_BOX) {
        BoxGeom g;
        if (!box_geometry(s, 128, &g) && !box_geometry(s, 256, &g)) return CONV2D_ERR_UNSUPPORTED;
    } else if (loader == CONV2D_LOADER_HALO) {
        HaloGeom g;
        if (!halo_geometry(s, 64, &g)) return CONV2D_ERR_UNSUPPORTED;
    } else if (loader == CONV2D_LOADER_TMA_PAIR) {
        return choose_pair_plan(s, force, plan, whole_tiles);
    } else if (loader == CONV2D_LOADER_PAIR_HALO) {
        return choose_pair_halo_plan(s, force, plan, whole_tiles);
    } else if (loader != CONV2D_LOADER_SCALAR) {
        return CONV2D_ERR_INVALID;
    }
    if (loader == CONV2D_LOADER_ROW_WINDOW) {
        // One tile = up to 128 pixels of one output row, all channels; never split.
        if (force && (force->splits > 1 || (force->block_m != 0 && force->block_m != 128) || force->grid < 0))
            return CONV2D_ERR_UNSUPPORTED;
        int64_t grid = force && force->grid > 0 ? force->grid : (rw.tiles < sms ? rw.tiles : (sms > 0 ? sms : 1));
        if (grid > rw.tiles) return CONV2D_ERR_UNSUPPORTED;
        plan->block_m = sgb::RW_TILE_M;
        plan->block_n = rw.bn;
        plan->splits = 0;
        plan->loader = loader;
        plan->m_tiles = rw.tiles;
        plan->n_tiles = 1;
        plan->num_kb = 1;
        plan->grid = static_cast<int>(grid);
        plan->units = rw.tiles;
        return CONV2D_OK;
    }
    int bm = force ? force->block_m : 0;
    if (bm == 0) {
        // 256-pixel tiles halve the im2col operations per MMA (the TMA unit's cost
        // is per operation); worth it when the output channels are few (<= 128,
        // so the MMA per k-block is short) and the tiles still cover the SMs.
        bm = 128;
        const int64_t bn_guess = (force && force->block_n) ? force->block_n : (s.kg <= 64 ? 64 : (s.kg <= 128 ? 128 : 256));
        const int64_t cover = (sms > 0 ? sms : 1) * 4;
        BoxGeom g256;
        if (loader == CONV2D_LOADER_TMA_IM2COL && bn_guess <= 128 && (!force || force->splits == 0) &&
            cdiv(s.m, 256) * s.g * cdiv(s.kg, bn_guess) * 5 >= cover)
            bm = 256;
        if (loader == CONV2D_LOADER_TMA_BOX && bn_guess <= 128 && (!force || force->splits == 0) &&
            box_geometry(s, 256, &g256) && g256.px * 4 >= 256 * 3 && g256.m_tiles * cdiv(s.k, bn_guess) * 5 >= cover)
            bm = 256;
        BoxGeom g128;
        if (loader == CONV2D_LOADER_TMA_BOX && bm == 128 && !box_geometry(s, 128, &g128)) bm = 256;
    }
    if (bm != 128 && bm != 256) return CONV2D_ERR_INVALID;
    if (bm == 256 && loader != CONV2D_LOADER_TMA_IM2COL && loader != CONV2D_LOADER_TMA_BOX)
        return CONV2D_ERR_UNSUPPORTED;
    BoxGeom geom{};
    if (loader == CONV2D_LOADER_TMA_BOX && !box_geometry(s, bm, &geom)) return CONV2D_ERR_UNSUPPORTED;
    HaloGeom hgeom{};
    if (loader == CONV2D_LOADER_HALO && !halo_geometry(s, 64, &hgeom)) return CONV2D_ERR_UNSUPPORTED;
    const int64_t m_tiles = loader == CONV2D_LOADER_TMA_BOX ? geom.m_tiles
                            : loader == CONV2D_LOADER_HALO  ? hgeom.m_tiles
                                                            : cdiv(s.m, bm);
    const int64_t num_kb = loader == CONV2D_LOADER_TMA_BOX ? s.crs / (kBoxChunks * BK) : cdiv(s.crs, BK);
    const int64_t forced_splits = force ? force->splits : 0;
    const int64_t forced_grid = force ? force->grid : 0;
    if (forced_splits < 0 || forced_grid < 0 || (forced_splits > 0 && forced_grid > 0)) return CONV2D_ERR_INVALID;
    const int64_t nsm = sms > 0 ? sms : 1;
    // Tile width: as wide as the output channels allow (one A tile feeds more
    // MMAs); narrower when that leaves so few tiles that a long reduction would
    // need more than kMaxSplitsPerTile in-place turns per tile.
    int bn = force ? force->block_n : 0;
    if (bn == 0) {
        bn = s.kg <= 64 ? 64 : (s.kg <= 128 ? 128 : 256);
        while (bn > 64 && forced_splits == 0 && forced_grid == 0) {
            const int64_t tiles = m_tiles * s.g * cdiv(s.kg, bn);
            if (tiles * 2 > nsm || num_kb < 8 || nsm / tiles <= kMaxSplitsPerTile) break;
            bn /= 2;
        }
    }
    if (bn != 64 && bn != 128 && bn != 256) return CONV2D_ERR_INVALID;
    if (loader == CONV2D_LOADER_TMA_BOX && bm == 256 && bn > 128) return CONV2D_ERR_UNSUPPORTED;
    if (loader == CONV2D_LOADER_HALO) {
        // The widest tile whose ring and halo buffers fit the shared memory.
        while (!halo_geometry(s, bn, &hgeom)) {
            if (bn == 64 || (force && force->block_n)) return CONV2D_ERR_UNSUPPORTED;
            bn /= 2;
        }
    }
    // Column blocks never straddle a group: ntpg blocks per group.
    const int64_t n_tiles = s.g * cdiv(s.kg, bn);
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t units = tiles * num_kb;
    int64_t splits = forced_splits;
    int64_t grid = forced_grid;
    if (splits == 0 && grid == 0 && whole_tiles && tiles >= nsm) {
        // Each CTA takes whole tiles: the smallest whole-tile share per CTA that
        // fits the SMs in one wave and divides the tiles evenly, else one tile per CTA.
        grid = tiles;
        const int64_t per_cta = cdiv(tiles, nsm);
        for (int64_t d = per_cta; d <= 2 * per_cta; ++d)
            if (tiles % d == 0) {
                grid = tiles / d;
                break;
            }
    } else if (splits == 0 && grid == 0) {
        if (tiles >= nsm) {
            // Persistent: every SM takes the same number of whole tiles where that
            // divides out, otherwise an even share of (tile, k-block) units.
            const int64_t per_cta = cdiv(tiles, nsm);
            grid = cdiv(tiles, per_cta);
        } else if (tiles * 2 <= nsm && num_kb >= 8) {
            // Few tiles, long reduction: classic split-K (the "small M*N, large
            // C*R*S" regime), every split keeping at least four k-blocks.
            splits = nsm / tiles;
            if (splits > kMaxSplitsPerTile) splits = kMaxSplitsPerTile;
            if (splits > num_kb / kMinUnitsPerCta) splits = num_kb / kMinUnitsPerCta;
            if (splits < 1) splits = 1;
        } else {
            grid = tiles;  // one tile per CTA: cutting tiles costs more than the idle SMs
        }
    }
    if (splits > 0) {
        if (splits > num_kb) return CONV2D_ERR_UNSUPPORTED;  // every split needs at least one k-block
        grid = tiles * splits;
    } else if (grid > units) {
        return CONV2D_ERR_UNSUPPORTED;  // every CTA needs at least one unit
    }
    if (grid > 2147483647ll) return CONV2D_ERR_UNSUPPORTED;
    // A plan that cuts tiles needs one semaphore per tile.
    if (num_kb > 1 && ((units % grid) != 0 || (units / grid) % num_kb != 0) && tiles > semaphore_capacity(s))
        return CONV2D_ERR_UNSUPPORTED;
    plan->box = geom;
    plan->halo = hgeom;
    plan->block_m = bm;
    plan->block_n = bn;
    plan->splits = static_cast<int>(splits);
    plan->loader = loader;
    plan->m_tiles = static_cast<int>(m_tiles);
    plan->n_tiles = static_cast<int>(n_tiles);
    plan->num_kb = static_cast<int>(num_kb);
    plan->grid = static_cast<int>(grid);
    plan->units = units;
    return CONV2D_OK;
}

// CTA b takes units [b*units/grid, (b+1)*units/grid): a tile is cut when a
// boundary falls inside its num_kb units.  With one unit per tile no boundary
// can; otherwise equal shares that are whole multiples of num_kb cut nothing,
// and every other division is treated as cutting (it may spare some tiles).
bool plan_cuts_tiles(const Plan& p)
{
    if (p.num_kb <= 1) return false;
    return (p.units % p.grid) != 0 || (p.units / p.grid) % p.num_kb != 0;
}

size_t workspace_bytes_for(const Shape& s)
{
    // Enough semaphores for the narrowest tile width.
    return kStatusBytes + static_cast<size_t>(semaphore_capacity(s)) * sizeof(uint32_t);
}

// Where the fused epilogue's fp32 partial-sum buffer starts in the workspace.
size_t part_offset(const Shape& s) { return (workspace_bytes_for(s) + 255) & ~size_t(255); }

size_t round256(size_t v) { return (v + 255) & ~size_t(255); }

// Workspace one call needs: status and semaphores, plus under a fused epilogue
// an fp32 [M][K] partial-sum buffer when the plan cuts tiles.
size_t workspace_bytes_for_plan(const Shape& s, const Plan& plan, bool fused)
{
    if (fused && plan_cuts_tiles(plan)) return part_offset(s) + static_cast<size_t>(s.m * s.k) * sizeof(float);
    return workspace_bytes_for(s);
}

// ------------------------------------------------------------------ descriptors
int encode_maps(const Shape& s, const Plan& plan, const void* x, const void* w, CUtensorMap* tm_a, CUtensorMap* tm_b)
{
    std::memset(tm_a, 0, sizeof(*tm_a));
    std::memset(tm_b, 0, sizeof(*tm_b));
    if (!load_encoders()) return CONV2D_ERR_CUDA;
    if (plan.loader == CONV2D_LOADER_PAIR_HALO) {
        // A: x as {C, W, H, N}; a box is one 64-channel chunk of hr whole padded rows (wv columns
        // from -pad_w), landing pixel-major in 128-byte rows.  B: w as {64, K, Cg/64, R*S}; a box
        // is block_n/2 weight rows of one chunk at kbs consecutive taps (a tap past R*S reads zeros).
        const HaloGeom& g = plan.halo;
        const cuuint64_t dims[4] = {(cuuint64_t)s.c, (cuuint64_t)s.w, (cuuint64_t)s.h, (cuuint64_t)s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.w * s.c * 2),
                                       (cuuint64_t)(s.h * s.w * s.c * 2)};
        const cuuint32_t box[4] = {(cuuint32_t)BK, (cuuint32_t)g.wv, (cuuint32_t)g.hr, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult rc = g_encode_tiled(tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
        const cuuint64_t wd[4] = {(cuuint64_t)BK, (cuuint64_t)s.k, (cuuint64_t)(s.cg / BK), (cuuint64_t)(s.r * s.s)};
        const cuuint64_t ws[3] = {(cuuint64_t)(s.crs * 2), (cuuint64_t)(BK * 2), (cuuint64_t)(s.cg * 2)};
        const cuuint32_t wb[4] = {(cuuint32_t)BK, (cuuint32_t)(plan.block_n / 2), 1, (cuuint32_t)plan.kbs};
        const cuuint32_t we[4] = {1, 1, 1, 1};
        rc = g_encode_tiled(tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(w), wd, ws, wb, we,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
        return CONV2D_OK;
    }
    if (plan.loader == CONV2D_LOADER_TMA_PAIR) {
        // A: each CTA's 128 pixels x 64 channels per im2col load (window origins as for the
        // one-CTA loader).  B: w viewed as {64, K, C*R*S/64}; a box is block_n/2 weight rows x
        // two consecutive k-blocks, landing k-block-major (a k-block past the end reads zeros).
        const cuuint64_t dims[4] = {(cuuint64_t)s.c, (cuuint64_t)s.w, (cuuint64_t)s.h, (cuuint64_t)s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.w * s.c * 2),
                                       (cuuint64_t)(s.h * s.w * s.c * 2)};
        const int lower[2] = {(int)-s.pw, (int)-s.ph};
        const int upper[2] = {(int)(s.pw - (s.s - 1) * s.dw), (int)(s.ph - (s.r - 1) * s.dh)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)s.sw, (cuuint32_t)s.sh, 1};
        CUresult rc = g_encode_im2col(tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                                      strides, lower, upper, BK, static_cast<cuuint32_t>(sgb::PAIR_ROWS), estr,
                                      CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                      CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
        const cuuint64_t wd[3] = {(cuuint64_t)BK, (cuuint64_t)s.k, (cuuint64_t)(s.crs / BK)};
        const cuuint64_t ws[2] = {(cuuint64_t)(s.crs * 2), (cuuint64_t)(BK * 2)};
        const cuuint32_t wb[3] = {(cuuint32_t)BK, (cuuint32_t)(plan.block_n / 2), (cuuint32_t)plan.kbs};
        const cuuint32_t we[3] = {1, 1, 1};
        rc = g_encode_tiled(tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), wd, ws, wb, we,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
        return CONV2D_OK;
    }
    if (plan.loader == CONV2D_LOADER_TMA_IM2COL || plan.loader == CONV2D_LOADER_HYBRID) {
        const cuuint64_t dims[4] = {(cuuint64_t)s.c, (cuuint64_t)s.w, (cuuint64_t)s.h, (cuuint64_t)s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.w * s.c * 2),
                                       (cuuint64_t)(s.h * s.w * s.c * 2)};
        // Bounding box of window origins: lower corner -pad; upper corner measured
        // from the last element, pad - (filter-1)*dilation.  Order {W, H}.
        const int lower[2] = {(int)-s.pw, (int)-s.ph};
        const int upper[2] = {(int)(s.pw - (s.s - 1) * s.dw), (int)(s.ph - (s.r - 1) * s.dh)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)s.sw, (cuuint32_t)s.sh, 1};
        CUresult rc = g_encode_im2col(tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims,
                                      strides, lower, upper, BK, static_cast<cuuint32_t>(plan.block_m), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
    }
    if (plan.loader == CONV2D_LOADER_HALO) {
        // x as {C, W, H, N}; a box is one 64-channel chunk of hr whole padded
        // rows (wv columns from -pad_w), landing pixel-major in 128-byte rows.
        const HaloGeom& g = plan.halo;
        const cuuint64_t dims[4] = {(cuuint64_t)s.c, (cuuint64_t)s.w, (cuuint64_t)s.h, (cuuint64_t)s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.w * s.c * 2),
                                       (cuuint64_t)(s.h * s.w * s.c * 2)};
        const cuuint32_t box[4] = {(cuuint32_t)BK, (cuuint32_t)g.wv, (cuuint32_t)g.hr, 1};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        CUresult rc = g_encode_tiled(tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides,
                                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
    }
    if (plan.loader == CONV2D_LOADER_TMA_BOX) {
        // x as {64 channels, W, H, N, C/64}: a box is KC chunks of a bn_img x bh x bw pixel rectangle
        // (traversal strides sh, sw), landing chunk-major; w as {64, K, C*R*S/64}: KC k-blocks of BN rows.
        const BoxGeom& g = plan.box;
        const cuuint64_t xd[5] = {(cuuint64_t)BK, (cuuint64_t)s.w, (cuuint64_t)s.h, (cuuint64_t)s.n,
                                  (cuuint64_t)(s.c / BK)};
        const cuuint64_t xs[4] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.w * s.c * 2),
                                  (cuuint64_t)(s.h * s.w * s.c * 2), (cuuint64_t)(BK * 2)};
        const cuuint32_t xb[5] = {(cuuint32_t)BK, (cuuint32_t)(g.bw * s.sw), (cuuint32_t)(g.bh * s.sh),
                                  (cuuint32_t)g.bn_img, (cuuint32_t)kBoxChunks};
        const cuuint32_t xe[5] = {1, (cuuint32_t)s.sw, (cuuint32_t)s.sh, 1, 1};
        CUresult rc = g_encode_tiled(tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(x), xd, xs, xb, xe,
                                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
        const cuuint64_t wd[3] = {(cuuint64_t)BK, (cuuint64_t)s.k, (cuuint64_t)(s.crs / BK)};
        const cuuint64_t ws[2] = {(cuuint64_t)(s.crs * 2), (cuuint64_t)(BK * 2)};
        const cuuint32_t wb[3] = {(cuuint32_t)BK, (cuuint32_t)plan.block_n, (cuuint32_t)kBoxChunks};
        const cuuint32_t we[3] = {1, 1, 1};
        rc = g_encode_tiled(tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), wd, ws, wb, we,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
        return CONV2D_OK;
    }
    if (plan.loader != CONV2D_LOADER_SCALAR) {
        const cuuint64_t dims[2] = {(cuuint64_t)s.crs, (cuuint64_t)s.k};
        const cuuint64_t strides[1] = {(cuuint64_t)(s.crs * 2)};
        const cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)plan.block_n};
        const cuuint32_t estr[2] = {1, 1};
        CUresult rc = g_encode_tiled(tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(w), dims, strides,
                                     box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
    }
    return CONV2D_OK;
}

// ------------------------------------------------------------------ tensor-map cache
// Encoding a tensor map is host work on every call (a driver call per map).
// Repeated calls on the same problem and the same buffers -- a serving loop,
// an eager training step -- reuse the maps encoded the first time: a small
// cache keyed on everything a map depends on (the shape, the loader and tile
// geometry of the plan, the two base pointers and the device).  A changed
// pointer, shape or plan is a different key and is encoded afresh.
struct MapKey {
    Shape shape;
    int loader, block_m, block_n, kbs;
    BoxGeom box;
    HaloGeom halo;
    const void* x;
    const void* w;
    int device;
};

struct MapEntry {
    MapKey key;
    CUtensorMap a, b;
    bool used;
};

constexpr int kMapCacheEntries = 32;
std::mutex g_map_mutex;
MapEntry g_map_cache[kMapCacheEntries];
int g_map_next = 0;  // round-robin replacement
unsigned long long g_map_hits = 0, g_map_misses = 0;

MapKey make_map_key(const Shape& s, const Plan& plan, const void* x, const void* w, int device)
{
    MapKey k;
    std::memset(&k, 0, sizeof(k));  // padding bytes take part in the comparison
    k.shape = s;
    k.loader = plan.loader;
    k.block_m = plan.block_m;
    k.block_n = plan.block_n;
    if (plan.loader == CONV2D_LOADER_TMA_PAIR) k.kbs = plan.kbs;
    if (plan.loader == CONV2D_LOADER_TMA_BOX) k.box = plan.box;
    if (plan.loader == CONV2D_LOADER_HALO || plan.loader == CONV2D_LOADER_PAIR_HALO) k.halo = plan.halo;
    k.x = x;
    k.w = w;
    k.device = device;
    return k;
}

// y as a 2-D fp32 tensor {K, M} with row pitch ldy, boxes of 32 columns x 64
// rows in the 128-byte swizzle (the CTA-pair epilogue's TMA stores), cached by
// (pointer, sizes, device) like the operand maps.
struct YMapEntry {
    const void* y;
    int64_t m, k, ldy;
    int device;
    CUtensorMap map;
    bool used;
};
constexpr int kYMapEntries = 32;
YMapEntry g_ymap_cache[kYMapEntries];
int g_ymap_next = 0;

int encode_y_map_cached(float* y, int64_t m, int64_t k, int64_t ldy, CUtensorMap* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (m < 1 || k < 1 || (ldy * 4) % 16 != 0) return CONV2D_ERR_UNSUPPORTED;
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (const YMapEntry& e : g_ymap_cache)
            if (e.used && e.y == y && e.m == m && e.k == k && e.ldy == ldy && e.device == dev) {
                *out = e.map;
                ++g_map_hits;
                return CONV2D_OK;
            }
    }
    if (!load_encoders()) return CONV2D_ERR_CUDA;
    std::memset(out, 0, sizeof(*out));
    const cuuint64_t dims[2] = {(cuuint64_t)k, (cuuint64_t)m};
    const cuuint64_t strides[1] = {(cuuint64_t)(ldy * 4)};
    const cuuint32_t box[2] = {32, (cuuint32_t)sgb::EPI_BOX_ROWS};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult rc = g_encode_tiled(out, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, y, dims, strides, box, estr,
                                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                                       CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (rc != CUDA_SUCCESS) return CONV2D_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    YMapEntry& e = g_ymap_cache[g_ymap_next];
    g_ymap_next = (g_ymap_next + 1) % kYMapEntries;
    e.y = y;
    e.m = m;
    e.k = k;
    e.ldy = ldy;
    e.device = dev;
    e.map = *out;
    e.used = true;
    ++g_map_misses;
    return CONV2D_OK;
}

// CONV2D_NO_MAP_CACHE=1 in the environment encodes every call's maps afresh
// (a measurement switch: the cache's effect on host time per call).
bool map_cache_enabled()
{
    static const bool on = [] {
        const char* v = std::getenv("CONV2D_NO_MAP_CACHE");
        return !(v && v[0] == '1');
    }();
    return on;
}

int encode_maps_cached(const Shape& s, const Plan& plan, const void* x, const void* w, CUtensorMap* tm_a,
                       CUtensorMap* tm_b)
{
    if (!map_cache_enabled()) return encode_maps(s, plan, x, w, tm_a, tm_b);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CONV2D_ERR_CUDA;
    const MapKey key = make_map_key(s, plan, x, w, dev);
    {
        std::lock_guard<std::mutex> lock(g_map_mutex);
        for (const MapEntry& e : g_map_cache)
            if (e.used && std::memcmp(&e.key, &key, sizeof(key)) == 0) {
                *tm_a = e.a;
                *tm_b = e.b;
                ++g_map_hits;
                return CONV2D_OK;
            }
    }
    const int rc = encode_maps(s, plan, x, w, tm_a, tm_b);
    if (rc != CONV2D_OK) return rc;
    std::lock_guard<std::mutex> lock(g_map_mutex);
    MapEntry& e = g_map_cache[g_map_next];
    g_map_next = (g_map_next + 1) % kMapCacheEntries;
    e.key = key;
    e.a = *tm_a;
    e.b = *tm_b;
    e.used = true;
    ++g_map_misses;
    return CONV2D_OK;
}

cudaError_t dispatch(int bm, int bn, int loader, const CUtensorMap& a, const CUtensorMap& b,
                     const sgb::ConvKernelParams& kp, int grid, cudaStream_t st)
{
    using namespace sgb;
    if (loader == CONV2D_LOADER_HALO) {
        if (bm != 128) return cudaErrorInvalidValue;
        if (bn == 64) return launch_conv2d_tc<128, 64, LOADER_HALO>(a, b, kp, grid, st);
        if (bn == 128) return launch_conv2d_tc<128, 128, LOADER_HALO>(a, b, kp, grid, st);
        if (bn == 256) return launch_conv2d_tc<128, 256, LOADER_HALO>(a, b, kp, grid, st);
        return cudaErrorInvalidValue;
    }
    if (loader == CONV2D_LOADER_TMA_BOX) {
        if (bm == 256) {
            if (bn == 64) return launch_conv2d_tc<256, 64, LOADER_BOX>(a, b, kp, grid, st);
            if (bn == 128) return launch_conv2d_tc<256, 128, LOADER_BOX>(a, b, kp, grid, st);
            return cudaErrorInvalidValue;
        }
        if (bn == 64) return launch_conv2d_tc<128, 64, LOADER_BOX>(a, b, kp, grid, st);
        if (bn == 128) return launch_conv2d_tc<128, 128, LOADER_BOX>(a, b, kp, grid, st);
        if (bn == 256) return launch_conv2d_tc<128, 256, LOADER_BOX>(a, b, kp, grid, st);
        return cudaErrorInvalidValue;
    }
#define SGB_CASE(BN_)                                                                                          \
    if (bn == BN_) {                                                                                           \
        if (bm == 256) return launch_conv2d_tc<256, BN_, LOADER_TMA>(a, b, kp, grid, st);                 \
        if (loader == CONV2D_LOADER_TMA_IM2COL) return launch_conv2d_tc<128, BN_, LOADER_TMA>(a, b, kp, grid, st); \
        if (loader == CONV2D_LOADER_CPASYNC) return launch_conv2d_tc<128, BN_, LOADER_CPASYNC>(a, b, kp, grid, st); \
        if (loader == CONV2D_LOADER_HYBRID) return launch_conv2d_tc<128, BN_, LOADER_HYBRID>(a, b, kp, grid, st); \
        return launch_conv2d_tc<128, BN_, LOADER_SCALAR>(a, b, kp, grid, st);                               \
    }
    SGB_CASE(64)
    SGB_CASE(128)
    SGB_CASE(256)
#undef SGB_CASE
    return cudaErrorInvalidValue;
}

bool log_enabled()
{
    static const bool on = [] {
        const char* v = std::getenv("CONV2D_LOG");
        return v && v[0] == '1';
    }();
    return on;
}

int run_direct(const Shape& s, const void* x, const void* w, const float* bias, float* y, cudaStream_t stream,
               const conv2d_algo* algo, bool relu, bool out_bf16)
{
    sgb::DirectParams dp{};
    dp.x = static_cast<const uint16_t*>(x);
    dp.w = static_cast<const uint16_t*>(w);
    dp.bias = bias;
    dp.y = y;
    dp.N = (int)s.n; dp.H = (int)s.h; dp.W = (int)s.w; dp.C = (int)s.c;
    dp.K = (int)s.k; dp.R = (int)s.r; dp.S = (int)s.s; dp.P = (int)s.p; dp.Q = (int)s.q;
    dp.sh = (int)s.sh; dp.sw = (int)s.sw; dp.ph = (int)s.ph; dp.pw = (int)s.pw; dp.dh = (int)s.dh; dp.dw = (int)s.dw;
    dp.G = (int)s.g;
    dp.relu = relu ? 1 : 0;
    dp.out_bf16 = out_bf16 ? 1 : 0;
    dp.nchunk = (int)(s.c / direct_chunk(s.cg));
    dp.qblocks = (int)cdiv(s.q, direct_px(s.cg));
    dp.items = (int)direct_items(s);
    const long long smem = sgb::conv2d_direct_smem_bytes(dp.K, dp.R, dp.S, (int)s.cg);
    long long grid = direct_grid(s);
    if (algo && algo->grid > 0) grid = algo->grid;
    if (grid < 1 || grid > 2147483647ll) return CONV2D_ERR_UNSUPPORTED;
    if (log_enabled())
        std::fprintf(stderr, "[conv2d] M=%lld K=%lld groups=%lld -> direct CG=%lld grid=%lld smem=%lld\n",
                     (long long)s.m, (long long)s.k, (long long)s.g, (long long)s.cg, grid, smem);
    cudaError_t err;
    switch (s.cg) {
        case 1: err = sgb::launch_conv2d_direct<1>(dp, (int)grid, stream); break;
        case 2: err = sgb::launch_conv2d_direct<2>(dp, (int)grid, stream); break;
        case 4: err = sgb::launch_conv2d_direct<4>(dp, (int)grid, stream); break;
        case 8: err = sgb::launch_conv2d_direct<8>(dp, (int)grid, stream); break;
        default: err = sgb::launch_conv2d_direct<16>(dp, (int)grid, stream); break;
    }
    if (err != cudaSuccess) return CONV2D_ERR_CUDA;
    g_last_launches = 1;
    return CONV2D_OK;
}

// Block-diagonal grouped tiles: groups of cg = 8, 16 or 32 channels (cg input and
// cg output channels each) merged 64 / cg at a time into groups of 64, the
// weight expanded to [K][R][S][64] with zeros outside each output channel's own
// group (launch_expand_blockdiag).  The tensor cores then do 64 / cg times the
// multiplications, but through TMA im2col boxes and 128 x 64 MMAs instead of
// CUDA-core FMAs.
bool blockdiag_eligible(const Shape& s)
{
    if (s.g < 2 || s.cg != s.kg || (s.cg != 8 && s.cg != 16 && s.cg != 32)) return false;
    const int64_t f = 64 / s.cg;
    return s.g % f == 0;
}

Shape blockdiag_shape(const Shape& s)
{
    Shape t = s;
    const int64_t f = 64 / s.cg;
    t.g = s.g / f;
    t.cg = 64;
    t.kg = 64;
    t.crs = t.r * t.s * t.cg;
    return t;
}

size_t blockdiag_weight_bytes(const Shape& s) { return static_cast<size_t>(s.k * s.r * s.s * 64) * 2; }

// Launches one planned forward convolution (encodes the maps, fills the kernel
// parameters, dispatches on the loader).
int run_plan(const Shape& s, const Plan& plan, const void* x, const void* w, const float* bias, float* y,
             void* workspace, size_t workspace_bytes, cudaStream_t stream, const conv2d_algo* algo, bool relu,
             bool out_bf16)
{
    int rc = CONV2D_OK;
    const bool fused = relu || out_bf16;
    const bool have_ws = workspace && workspace_bytes >= workspace_bytes_for(s);
    // Any tile cut between CTAs needs the semaphores (and, under a fused
    // epilogue, the partial-sum buffer).
    const bool cuts_tiles = plan_cuts_tiles(plan);
    if (cuts_tiles && (!workspace || workspace_bytes < workspace_bytes_for_plan(s, plan, fused)))
        return CONV2D_ERR_WORKSPACE;
    if (workspace && !have_ws) return CONV2D_ERR_WORKSPACE;
    const bool vec_store = (s.k % 4) == 0 && (s.kg % 4) == 0;  // 16-byte vector writes inside one group's columns
    if (plan.loader == CONV2D_LOADER_ROW_WINDOW) {
        RowWinCfg rw;
        if (!rowwin_config(s, plan.block_n, &rw)) return CONV2D_ERR_UNSUPPORTED;
        sgb::RowWinParams rp{};
        rp.x = static_cast<const uint16_t*>(x);
        rp.w = static_cast<const uint16_t*>(w);
        rp.bias = bias;
        rp.y = y;
        rp.status = have_ws ? static_cast<uint32_t*>(workspace) : nullptr;
        rp.N = (int)s.n; rp.H = (int)s.h; rp.W = (int)s.w; rp.C = (int)s.c;
        rp.K = (int)s.k; rp.R = (int)s.r; rp.S = (int)s.s; rp.P = (int)s.p; rp.Q = (int)s.q;
        rp.sh = (int)s.sh; rp.sw = (int)s.sw; rp.ph = (int)s.ph; rp.pw = (int)s.pw; rp.dh = (int)s.dh;
        rp.cp_log2 = rw.cp_log2;
        rp.nch = rw.nch;
        rp.seg_elems = rw.seg_elems;
        rp.raw_bytes = rw.raw_bytes;
        rp.T = rw.T;
        rp.rt = rw.rt;
        rp.new_rows = rw.new_rows;
        rp.reuse = rw.reuse;
        rp.ncls = rw.ncls;
        for (int i = 0; i < sgb::RW_MAX_CLASSES; ++i) {
            rp.cls_k[i] = rw.cls_k[i];
            rp.cls_base[i] = rw.cls_base[i];
        }
        rp.nblocks = rw.nblocks;
        rp.row_slots = rw.row_slots;
        rp.wtmp_filters = rw.wtmp_filters;
        rp.qblocks = rw.qblocks;
        rp.pblocks = rw.pblocks;
        rp.tiles = rw.tiles;
        rp.grid = plan.grid;
        rp.tmem_cols = rw.tmem_cols;
        rp.vec_store = vec_store ? 1 : 0;
        rp.relu = relu ? 1 : 0;
        rp.out_bf16 = out_bf16 ? 1 : 0;
        rp.x_bytes = s.n * s.h * s.w * s.c * 2;
        rp.w_bytes = s.k * s.crs * 2;
        rp.off_rows = rw.lay.off_rows;
        rp.off_raw = rw.lay.off_raw;
        rp.off_wtmp = rw.lay.off_wtmp;
        rp.off_epi = rw.lay.off_epi;
        rp.off_bar = rw.lay.off_bar;
        rp.off_tab = rw.lay.off_tab;
        rp.wait_limit_ns =
            (algo && algo->wait_limit_ns > 0) ? (unsigned long long)algo->wait_limit_ns : kDefaultWaitNs;
        rp.trace = nullptr;
#ifdef SGB_TRACE_ENABLED
        rp.trace = g_trace;
#endif
        if (log_enabled())
            std::fprintf(stderr,
                         "[conv2d] M=%lld K=%lld CRS=%lld -> row window BN=%d T=%d rt=%d tiles=%d grid=%d slots=%d "
                         "nch=%d blocks=%d reuse=%d smem=%d\n",
                         (long long)s.m, (long long)s.k, (long long)s.crs, rw.bn, rw.T, rw.rt, rw.tiles, plan.grid,
                         rw.row_slots, rw.nch, rw.nblocks, rw.reuse, rw.lay.total);
        cudaError_t err;
        const bool pdl = sgb::pdl_enabled();
        if (rw.bn == 64) err = sgb::launch_conv2d_rowwin<64>(rp, rw.lay.total, pdl, stream);
        else if (rw.bn == 128) err = sgb::launch_conv2d_rowwin<128>(rp, rw.lay.total, pdl, stream);
        else err = sgb::launch_conv2d_rowwin<256>(rp, rw.lay.total, pdl, stream);
        if (err != cudaSuccess) return CONV2D_ERR_CUDA;
        g_last_launches = 1;
        return CONV2D_OK;
    }

    CUtensorMap tm_a, tm_b;
    rc = encode_maps_cached(s, plan, x, w, &tm_a, &tm_b);
    if (rc != CONV2D_OK) return rc;

    sgb::ConvKernelParams kp{};
    kp.x = static_cast<const uint16_t*>(x);
    kp.w = static_cast<const uint16_t*>(w);
    kp.bias = bias;
    kp.y = y;
    kp.ldy = (int)s.k;
    kp.status = have_ws ? static_cast<uint32_t*>(workspace) : nullptr;
    kp.sems = have_ws ? reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kStatusBytes) : nullptr;
    kp.N = (int)s.n; kp.H = (int)s.h; kp.W = (int)s.w; kp.C = (int)s.c;
    kp.K = (int)s.k; kp.R = (int)s.r; kp.S = (int)s.s; kp.P = (int)s.p; kp.Q = (int)s.q;
    kp.sh = (int)s.sh; kp.sw = (int)s.sw; kp.ph = (int)s.ph; kp.pw = (int)s.pw; kp.dh = (int)s.dh; kp.dw = (int)s.dw;
    kp.M = (int)s.m;
    kp.CRS = (int)s.crs;
    kp.G = (int)s.g;
    kp.Cg = (int)s.cg;
    kp.Kg = (int)s.kg;
    kp.ntpg = (int)(plan.n_tiles / s.g);
    kp.num_kb = plan.num_kb;
    kp.m_tiles = plan.m_tiles;
    kp.n_tiles = plan.n_tiles;
    kp.grid = plan.grid;
    kp.units = plan.units;
    kp.vec_store = vec_store ? 1 : 0;
    kp.relu = relu ? 1 : 0;
    kp.out_bf16 = out_bf16 ? 1 : 0;
    kp.part = fused && cuts_tiles ? reinterpret_cast<float*>(static_cast<char*>(workspace) + part_offset(s)) : nullptr;
    kp.bw = plan.box.bw;
    kp.bh = plan.box.bh;
    kp.bn_img = plan.box.bn_img;
    kp.px = plan.box.px;
    kp.q_blocks = plan.box.q_blocks;
    kp.p_blocks = plan.box.p_blocks;
    kp.wv = plan.halo.wv;
    kp.vp = plan.halo.vp;
    kp.tpi = plan.halo.tpi;
    kp.halo_rows = plan.halo.hr;
    kp.halo_bytes = plan.loader == CONV2D_LOADER_HALO ? plan.halo.halo_bytes : 0;
    kp.halo_tx = plan.halo.hr * plan.halo.wv * 128;
    kp.debug_flags = algo ? algo->debug_flags : 0;
    kp.reduce_concurrent = (algo && algo->reduction == CONV2D_REDUCTION_ORDERED) ? 0 : 1;
    kp.wait_limit_ns = (algo && algo->wait_limit_ns > 0) ? (unsigned long long)algo->wait_limit_ns : kDefaultWaitNs;
    kp.trace = nullptr;
#ifdef SGB_TRACE_ENABLED
    kp.trace = g_trace;
#endif
    if (plan.loader == CONV2D_LOADER_PAIR_HALO) {
        kp.wv = plan.halo.wv;
        kp.vp = plan.halo.vp;
        kp.tpi = plan.halo.tpi;
        kp.halo_rows = plan.halo.hr;
        kp.halo_bytes = plan.halo.halo_bytes;
        kp.halo_tx = plan.halo.hr * plan.halo.wv * 128;
        kp.fd_tpi = sgb::FastDiv(static_cast<uint32_t>(plan.halo.tpi));
        kp.fd_wv = sgb::FastDiv(static_cast<uint32_t>(plan.halo.wv));
        kp.fd_tapst = sgb::FastDiv(static_cast<uint32_t>(cdiv(s.r * s.s, plan.kbs)));
    }
    if (plan.loader == CONV2D_LOADER_TMA_PAIR || plan.loader == CONV2D_LOADER_PAIR_HALO) {
        // fp32 output through the TMA unit: a measurement hook (16-byte aligned y).
        // Per-thread vector stores measured faster on GB300 (the boxes' staging
        // handshakes cost more than the shared-memory reads they save).
        kp.tma_y = 0;
        if (!out_bf16 && (reinterpret_cast<uintptr_t>(y) & 15u) == 0 && (kp.debug_flags & CONV2D_DEBUG_TMA_STORE) &&
            encode_y_map_cached(y, s.m, s.k, kp.ldy, &kp.tm_y) == CONV2D_OK)
            kp.tma_y = 1;
        kp.unit_offset = plan.unit_offset;
        kp.fd_grid = sgb::FastDiv(static_cast<uint32_t>(plan.grid));
        kp.fd_units = sgb::FastDiv(static_cast<uint32_t>(plan.units));
        kp.fd_nkb = sgb::FastDiv(static_cast<uint32_t>(plan.num_kb));
        kp.fd_ntiles = sgb::FastDiv(static_cast<uint32_t>(plan.n_tiles));
        kp.fd_pq = sgb::FastDiv(static_cast<uint32_t>(s.p * s.q));
        kp.fd_q = sgb::FastDiv(static_cast<uint32_t>(s.q));
        kp.fd_c = sgb::FastDiv(static_cast<uint32_t>(s.cg));
        kp.fd_s = sgb::FastDiv(static_cast<uint32_t>(s.s));
    }

    const int64_t grid = plan.grid;
    if (log_enabled())
        std::fprintf(stderr, "[conv2d] M=%lld K=%lld CRS=%lld -> BM=%d BN=%d splits=%d loader=%d grid=%lld vec_store=%d\n",
                     (long long)s.m, (long long)s.k, (long long)s.crs, plan.block_m, plan.block_n, plan.splits, plan.loader,
                     (long long)grid, (int)vec_store);
    cudaError_t err;
    if (plan.loader == CONV2D_LOADER_TMA_PAIR)
        err = launch_pair(plan.block_n, plan.kbs, tm_a, tm_b, kp, (int)grid, stream);
    else if (plan.loader == CONV2D_LOADER_PAIR_HALO)
        err = launch_pair_halo(plan.block_n, plan.kbs, tm_a, tm_b, kp, (int)grid, stream);
    else
        err = dispatch(plan.block_m, plan.block_n, plan.loader, tm_a, tm_b, kp, (int)grid, stream);
    if (err != cudaSuccess) return CONV2D_ERR_CUDA;
    g_last_launches = 1;
    return CONV2D_OK;
}

int run_conv(const conv2d_params* params, const void* x, const void* w, const float* bias, float* y,
             void* workspace, size_t workspace_bytes, cudaStream_t stream, const conv2d_algo* algo,
             const conv2d_epilogue* epi = nullptr)
{
    g_last_launches = 0;
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (s.m == 0 || s.k == 0) return CONV2D_OK;  // empty batch or no filters: nothing to compute
    if (!x || !w || !y) return CONV2D_ERR_INVALID;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || (bias && !aligned16(bias)) ||
        (workspace && !aligned16(workspace)))
        return CONV2D_ERR_ALIGNMENT;
    if (algo && (algo->splits < 0 || algo->block_n < 0 || algo->block_m < 0 || algo->grid < 0 ||
                 algo->wait_limit_ns < 0 || algo->reduction < CONV2D_REDUCTION_AUTO ||
                 algo->reduction > CONV2D_REDUCTION_CONCURRENT))
        return CONV2D_ERR_INVALID;
    if (epi && (epi->activation < CONV2D_ACT_NONE || epi->activation > CONV2D_ACT_RELU ||
                epi->out_dtype < CONV2D_OUT_F32 || epi->out_dtype > CONV2D_OUT_BF16))
        return CONV2D_ERR_INVALID;
    const bool relu = epi && epi->activation == CONV2D_ACT_RELU;
    const bool out_bf16 = epi && epi->out_dtype == CONV2D_OUT_BF16;
    const bool fused = relu || out_bf16;
    const bool force_direct = algo && algo->loader == CONV2D_LOADER_DIRECT;
    // Block-diagonal grouped tiles (before the direct kernel, which they beat):
    // groups of cg = 8, 16 or 32 channels merged 64 / cg at a time into 64-channel
    // groups, on a weight expanded into the workspace with zeros off the diagonal
    // blocks; the rest is the grouped implicit GEMM.  Needs the room in the workspace
    // (else the direct kernel or the plain grouped path runs).
    const bool force_bd = algo && algo->loader == CONV2D_LOADER_BLOCKDIAG;
    if (force_bd && (!blockdiag_eligible(s) || algo->splits || algo->grid || algo->block_n || algo->block_m))
        return CONV2D_ERR_UNSUPPORTED;
    if (force_bd || (!force_direct && nothing_forced(algo) && blockdiag_eligible(s))) {
        const Shape t = blockdiag_shape(s);
        conv2d_algo tf;
        std::memset(&tf, 0, sizeof(tf));
        if (algo) {  // keep the caller's waits, hooks and reduction mode
            tf.wait_limit_ns = algo->wait_limit_ns;
            tf.debug_flags = algo->debug_flags;
            tf.reduction = algo->reduction;
        }
        Plan tplan;
        if (choose_plan(t, &tf, &tplan, fused) == CONV2D_OK) {
            const size_t off = round256(workspace_bytes_for_plan(t, tplan, fused));
            if (force_bd && !(workspace && workspace_bytes >= off + blockdiag_weight_bytes(s)))
                return CONV2D_ERR_WORKSPACE;
            if (workspace && workspace_bytes >= off + blockdiag_weight_bytes(s)) {
                uint16_t* wb = reinterpret_cast<uint16_t*>(static_cast<char*>(workspace) + off);
                if (sgb::launch_expand_blockdiag(static_cast<const uint16_t*>(w), wb, (int)s.k, (int)(s.r * s.s),
                                                 (int)s.cg, stream) != cudaSuccess)
                    return CONV2D_ERR_CUDA;
                rc = run_plan(t, tplan, x, wb, bias, y, workspace, workspace_bytes, stream, &tf, relu, out_bf16);
                if (rc != CONV2D_OK) return rc;
                // The workspace is zero at rest (a later call's semaphores or partial-sum
                // buffer may lie where the expanded weight was): clear it in stream order.
                if (cudaMemsetAsync(wb, 0, blockdiag_weight_bytes(s), stream) != cudaSuccess) return CONV2D_ERR_CUDA;
                g_last_launches = 2;  // the expansion and the convolution
                return CONV2D_OK;
            }
        }
    }
    if (force_direct || (nothing_forced(algo) && direct_eligible(s))) {
        if (!direct_eligible(s) || (algo && (algo->splits > 1 || algo->block_m != 0)))
            return CONV2D_ERR_UNSUPPORTED;
        return run_direct(s, x, w, bias, y, stream, algo, relu, out_bf16);
    }
    Plan plan;
    rc = choose_plan(s, algo, &plan, fused);
    if (rc != CONV2D_OK) return rc;
    return run_plan(s, plan, x, w, bias, y, workspace, workspace_bytes, stream, algo, relu, out_bf16);
}


// ------------------------------------------------------------------ weight gradient
// dw[k][(r*S + s)*C + c] = sum over output pixels l of dy[l][k] * im2col(x)[l][(r, s, c)]:
// GEMM rows are output channels (128 per tile), columns are (tap, channel block)
// pairs inside one tap, and the reduction runs over the N*P*Q output pixels in
// 64-pixel k-blocks.  The kernel is the forward kernel's pipeline with the
// LOADER_WGRAD loads: dy by tiled TMA, x by 64-pixel im2col TMA boxes.
bool wgrad_eligible(const Shape& s) { return s.g == 1 && s.c % BK == 0 && s.k % 8 == 0; }

int64_t wgrad_sem_capacity(const Shape& s) { return cdiv(s.k, 128) * s.r * s.s * cdiv(s.c, 64); }

size_t wgrad_workspace_bytes_for(const Shape& s)
{
    return kStatusBytes + static_cast<size_t>(wgrad_sem_capacity(s)) * sizeof(uint32_t);
}

struct WgradPlan {
    int block_n, splits, grid, m_tiles, n_tiles, ntpt, num_kb;
    int64_t units;
};

int choose_wgrad_plan(const Shape& s, const conv2d_algo* force, WgradPlan* pl)
{
    const int64_t nsm = sm_count_current() > 0 ? sm_count_current() : 1;
    if (force && force->block_m != 0 && force->block_m != 128) return CONV2D_ERR_UNSUPPORTED;
    if (force && force->loader != CONV2D_LOADER_AUTO && force->loader != CONV2D_LOADER_TMA_IM2COL)
        return CONV2D_ERR_UNSUPPORTED;
    // The widest column block the channels fill, so that each 64-pixel stage's dy tile
    // feeds the most MMA work (measured: 256 beats 128 by 8-25% where C allows it),
    // unless that leaves fewer than 16 tiles to share the reduction (a 1x1 layer with
    // C = 256 and K = 512 measured 8% slower at 256 wide).
    int bn = (force && force->block_n) ? force->block_n : (s.c % 256 == 0 ? 256 : s.c % 128 == 0 ? 128 : 64);
    if (!(force && force->block_n) && bn == 256 && cdiv(s.k, 128) * s.r * s.s * (s.c / 256) < 16) bn = 128;
    if (bn != 64 && bn != 128 && bn != 256) return CONV2D_ERR_INVALID;
    const int64_t m_tiles = cdiv(s.k, 128);
    const int64_t ntpt = cdiv(s.c, bn);
    const int64_t n_tiles = s.r * s.s * ntpt;
    const int64_t tiles = m_tiles * n_tiles;
    const int64_t num_kb = cdiv(s.m, BK);
    const int64_t units = tiles * num_kb;
    int64_t splits = force ? force->splits : 0;
    int64_t grid = force ? force->grid : 0;
    if (splits < 0 || grid < 0 || (splits > 0 && grid > 0)) return CONV2D_ERR_INVALID;
    if (splits == 0 && grid == 0) {
        if (tiles >= nsm) {
            const int64_t per_cta = cdiv(tiles, nsm);
            grid = cdiv(tiles, per_cta);
        } else {
            // Few tiles, a long reduction over the output pixels: every SM takes an
            // even share of the (tile, k-block) units, at least kMinUnitsPerCta.
            grid = units / kMinUnitsPerCta < nsm ? units / kMinUnitsPerCta : nsm;
            if (grid < tiles) grid = tiles;
        }
    }
    if (splits > 0) {
        if (splits > num_kb) return CONV2D_ERR_UNSUPPORTED;
        grid = tiles * splits;
    } else if (grid > units) {
        return CONV2D_ERR_UNSUPPORTED;
    }
    if (grid > 2147483647ll || units > (int64_t(1) << 62)) return CONV2D_ERR_UNSUPPORTED;
    pl->block_n = bn;
    pl->splits = static_cast<int>(splits);
    pl->grid = static_cast<int>(grid);
    pl->m_tiles = static_cast<int>(m_tiles);
    pl->n_tiles = static_cast<int>(n_tiles);
    pl->ntpt = static_cast<int>(ntpt);
    pl->num_kb = static_cast<int>(num_kb);
    pl->units = units;
    return CONV2D_OK;
}

bool wgrad_cuts_tiles(const WgradPlan& p)
{
    if (p.num_kb <= 1) return false;
    return (p.units % p.grid) != 0 || (p.units / p.grid) % p.num_kb != 0;
}

// ------------------------------------------------------------------ data gradient (stride 1)
// dx = conv(dy, w') with w'[c][r][s][k] = w[k][R-1-r][S-1-s][c], stride 1, the same
// dilation and padding dil*(R-1) - pad: a forward convolution of the output
// gradient, whose weight operand the kernel reads from w itself (LOADER_DGRAD).
// The data gradient runs as a forward convolution of dy (channels K) that
// produces dx (channels C), one launch per output phase.  At stride 1 there is
// one phase: dx[h] = sum_r dy[h + ph - r*dh] w[r], a stride-1 convolution of dy
// with the flipped filter.  At stride sh the rows h = a + sh*i of phase a
// (0 <= a < sh) receive only the taps r with a + ph - r*dh divisible by sh:
// r = r0 + m*u (m = sh / gcd(sh, dh)), and then
//     dx[a + sh*i] = sum_u dy[i + c - u*d'] w[r0 + m*u],   c = (a + ph - r0*dh) / sh,
// with d' = dh / gcd(sh, dh): a stride-1 convolution of dy over the phase's
// R' taps at dilation d' (the sub-pixel decomposition); columns likewise.  A
// phase with no tap is all zero.
struct DgradAxis {
    int r0, m, taps, dil, pad;  // first tap, tap step, tap count, dilation d', forward-form padding d'(R'-1) - c
    int64_t out;                // phase output extent ceil((H - a) / sh)
};

int64_t gcd64(int64_t a, int64_t b) { return b == 0 ? a : gcd64(b, a % b); }

// Phase `a` along one axis of extent h (stride st, padding pad, dilation dil,
// kernel ker).  false when the phase has no pixel; taps == 0 for no tap.
bool dgrad_axis(int64_t a, int64_t h, int64_t st, int64_t pad, int64_t dil, int64_t ker, DgradAxis* ax)
{
    if (a >= h) return false;
    ax->out = (h - a + st - 1) / st;
    const int64_t g = gcd64(st, dil);
    ax->m = static_cast<int>(st / g);
    ax->dil = static_cast<int>(dil / g);
    ax->taps = 0;
    ax->r0 = 0;
    ax->pad = 0;
    int64_t r0 = -1;
    for (int64_t r = 0; r < ker; ++r)
        if (((a + pad - r * dil) % st + st) % st == 0) {
            r0 = r;
            break;
        }
    if (r0 < 0) return true;
    ax->r0 = static_cast<int>(r0);
    ax->taps = static_cast<int>((ker - 1 - r0) / ax->m + 1);
    const int64_t c = (a + pad - r0 * dil) / st;  // exact
    ax->pad = static_cast<int>(static_cast<int64_t>(ax->dil) * (ax->taps - 1) - c);
    return true;
}

bool dgrad_eligible(const Shape& s)
{
    if (s.g != 1 || s.k % BK != 0 || s.c % 8 != 0) return false;
    // Every phase's forward-form padding d'(R'-1) - c must be >= 0 (the im2col
    // box's lower corner at or below 0), as ph <= dh*(R-1) is at stride 1.
    for (int64_t a = 0; a < s.sh; ++a) {
        DgradAxis ax;
        if (dgrad_axis(a, s.h, s.sh, s.ph, s.dh, s.r, &ax) && ax.taps > 0 && ax.pad < 0) return false;
    }
    for (int64_t b = 0; b < s.sw; ++b) {
        DgradAxis ax;
        if (dgrad_axis(b, s.w, s.sw, s.pw, s.dw, s.s, &ax) && ax.taps > 0 && ax.pad < 0) return false;
    }
    return true;
}

// The forward problem of one phase: input dy [N][P][Q][K], output the phase's
// [N][out_h][out_w][C] pixels, R' x S' taps at dilations d'.
Shape dgrad_phase_shape(const Shape& s, const DgradAxis& ah, const DgradAxis& aw)
{
    Shape t = s;
    t.h = s.p; t.w = s.q; t.c = s.k; t.k = s.c;
    t.r = ah.taps; t.s = aw.taps;
    t.sh = 1; t.sw = 1;
    t.dh = ah.dil; t.dw = aw.dil;
    t.ph = ah.pad; t.pw = aw.pad;
    t.g = 1; t.cg = t.c; t.kg = t.k;
    t.p = ah.out; t.q = aw.out;
    t.m = s.n * t.p * t.q;
    t.crs = t.c * t.r * t.s;
    return t;
}

// The whole-gradient forward problem (stride 1), used to size the workspace: every
// phase has at most its output pixels and so needs at most its semaphores.
Shape dgrad_forward_shape(const Shape& s)
{
    Shape t = s;
    t.h = s.p; t.w = s.q; t.c = s.k; t.k = s.c;
    t.sh = 1; t.sw = 1;
    t.ph = s.dh * (s.r - 1) - s.ph;
    t.pw = s.dw * (s.s - 1) - s.pw;
    t.g = 1; t.cg = t.c; t.kg = t.k;
    t.p = s.h; t.q = s.w;
    t.m = s.n * s.h * s.w;
    t.crs = t.c * t.r * t.s;
    return t;
}

int dgrad_plan(const Shape& t, const conv2d_algo* algo, Plan* plan)
{
    if (algo && algo->loader != CONV2D_LOADER_AUTO && algo->loader != CONV2D_LOADER_TMA_IM2COL)
        return CONV2D_ERR_UNSUPPORTED;
    if (algo && algo->block_m != 0 && algo->block_m != 128) return CONV2D_ERR_UNSUPPORTED;
    conv2d_algo f{};
    if (algo) f = *algo;
    f.loader = CONV2D_LOADER_TMA_IM2COL;
    f.block_m = 128;
    return choose_plan(t, &f, plan);
}

// One launch: phase (a, b) with axes ah, aw (stride 1: a = b = 0, the whole dx).
int launch_dgrad_phase(const Shape& s, const DgradAxis& ah, const DgradAxis& aw, int64_t a, int64_t b, const void* dy,
                       const void* w, float* dx, void* workspace, size_t workspace_bytes, cudaStream_t stream,
                       const conv2d_algo* algo)
{
    const Shape t = dgrad_phase_shape(s, ah, aw);
    Plan plan;
    int rc = dgrad_plan(t, algo, &plan);
    if (rc != CONV2D_OK) return rc;
    const bool have_ws = workspace && workspace_bytes >= workspace_bytes_for(t);
    if (plan_cuts_tiles(plan) && !have_ws) return CONV2D_ERR_WORKSPACE;

    CUtensorMap tm_a, tm_b;
    std::memset(&tm_a, 0, sizeof(tm_a));
    std::memset(&tm_b, 0, sizeof(tm_b));
    {   // dy through an im2col map whose window origins run over the phase's t.p x t.q
        // output pixels: lower corner -pad, upper corner (out - in) - pad per axis.
        const cuuint64_t dims[4] = {(cuuint64_t)t.c, (cuuint64_t)t.w, (cuuint64_t)t.h, (cuuint64_t)t.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(t.c * 2), (cuuint64_t)(t.w * t.c * 2),
                                       (cuuint64_t)(t.h * t.w * t.c * 2)};
        const int lower[2] = {(int)-t.pw, (int)-t.ph};
        const int upper[2] = {(int)(t.q - t.w - t.pw), (int)(t.p - t.h - t.ph)};
        const cuuint32_t estr[4] = {1, 1, 1, 1};
        if (g_encode_im2col(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(dy), dims, strides, lower,
                            upper, BK, static_cast<cuuint32_t>(plan.block_m), estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }
    {   // w as {C, R*S, K}: boxes of 64 channels x one tap x 64 filters (rows), 128-byte swizzle
        const cuuint64_t dims[3] = {(cuuint64_t)s.c, (cuuint64_t)(s.r * s.s), (cuuint64_t)s.k};
        const cuuint64_t strides[2] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.r * s.s * s.c * 2)};
        const cuuint32_t box[3] = {64, 1, (cuuint32_t)BK};
        const cuuint32_t estr[3] = {1, 1, 1};
        if (g_encode_tiled(&tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(w), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }

    sgb::ConvKernelParams kp{};
    kp.x = static_cast<const uint16_t*>(dy);
    kp.w = static_cast<const uint16_t*>(w);
    kp.bias = nullptr;
    kp.y = dx;
    kp.ldy = (int)t.k;
    kp.status = have_ws ? static_cast<uint32_t*>(workspace) : nullptr;
    kp.sems = have_ws ? reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kStatusBytes) : nullptr;
    kp.N = (int)t.n; kp.H = (int)t.h; kp.W = (int)t.w; kp.C = (int)t.c;
    kp.K = (int)t.k; kp.R = (int)t.r; kp.S = (int)t.s; kp.P = (int)t.p; kp.Q = (int)t.q;
    kp.sh = 1; kp.sw = 1; kp.ph = (int)t.ph; kp.pw = (int)t.pw; kp.dh = (int)t.dh; kp.dw = (int)t.dw;
    kp.M = (int)t.m;
    kp.CRS = (int)t.crs;
    kp.G = 1;
    kp.Cg = (int)t.c;
    kp.Kg = (int)t.k;
    kp.ntpg = plan.n_tiles;
    kp.num_kb = plan.num_kb;
    kp.m_tiles = plan.m_tiles;
    kp.n_tiles = plan.n_tiles;
    kp.grid = plan.grid;
    kp.units = plan.units;
    kp.vec_store = (t.k % 4) == 0 ? 1 : 0;
    kp.debug_flags = algo ? algo->debug_flags : 0;
    kp.reduce_concurrent = (algo && algo->reduction == CONV2D_REDUCTION_ORDERED) ? 0 : 1;
    kp.wait_limit_ns = (algo && algo->wait_limit_ns > 0) ? (unsigned long long)algo->wait_limit_ns : kDefaultWaitNs;
    kp.dg_r0 = ah.r0; kp.dg_rm = ah.m; kp.dg_s0 = aw.r0; kp.dg_sm = aw.m; kp.dg_S = (int)s.s;
    kp.dg_phase = (s.sh > 1 || s.sw > 1) ? 1 : 0;
    kp.dg_H = (int)s.h; kp.dg_W = (int)s.w; kp.dg_a = (int)a; kp.dg_b = (int)b;
    kp.dg_sh = (int)s.sh; kp.dg_sw = (int)s.sw;
    kp.trace = nullptr;
#ifdef SGB_TRACE_ENABLED
    kp.trace = g_trace;
#endif
    if (log_enabled())
        std::fprintf(stderr, "[conv2d dgrad] phase (%lld,%lld) M=%lld C=%lld KRS=%lld -> BN=%d splits=%d grid=%d\n",
                     (long long)a, (long long)b, (long long)t.m, (long long)t.k, (long long)t.crs, plan.block_n,
                     plan.splits, plan.grid);
    cudaError_t err;
    if (plan.block_n == 64) err = sgb::launch_conv2d_tc<128, 64, sgb::LOADER_DGRAD>(tm_a, tm_b, kp, plan.grid, stream);
    else if (plan.block_n == 128) err = sgb::launch_conv2d_tc<128, 128, sgb::LOADER_DGRAD>(tm_a, tm_b, kp, plan.grid, stream);
    else err = sgb::launch_conv2d_tc<128, 256, sgb::LOADER_DGRAD>(tm_a, tm_b, kp, plan.grid, stream);
    if (err != cudaSuccess) return CONV2D_ERR_CUDA;
    ++g_last_launches;
    return CONV2D_OK;
}

int run_dgrad(const conv2d_params* params, const void* dy, const void* w, float* dx, void* workspace,
              size_t workspace_bytes, cudaStream_t stream, const conv2d_algo* algo)
{
    g_last_launches = 0;
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (s.n == 0 || s.c == 0) return CONV2D_OK;  // empty input gradient
    if (!dx || (s.k > 0 && (!dy || !w))) return CONV2D_ERR_INVALID;
    if (!aligned16(dx) || (dy && !aligned16(dy)) || (w && !aligned16(w)) || (workspace && !aligned16(workspace)))
        return CONV2D_ERR_ALIGNMENT;
    if (algo && (algo->splits < 0 || algo->block_n < 0 || algo->block_m < 0 || algo->grid < 0 ||
                 algo->wait_limit_ns < 0 || algo->reduction < CONV2D_REDUCTION_AUTO ||
                 algo->reduction > CONV2D_REDUCTION_CONCURRENT))
        return CONV2D_ERR_INVALID;
    const size_t dx_bytes = static_cast<size_t>(s.n * s.h * s.w * s.c) * sizeof(float);
    if (s.k == 0) {  // no filters: the gradient is zero
        if (cudaMemsetAsync(dx, 0, dx_bytes, stream) != cudaSuccess) return CONV2D_ERR_CUDA;
        return CONV2D_OK;
    }
    if (!dgrad_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    const Shape full = dgrad_forward_shape(s);
    if (workspace && workspace_bytes < workspace_bytes_for(full)) return CONV2D_ERR_WORKSPACE;
    if (!load_encoders()) return CONV2D_ERR_CUDA;
    // Phases with no tap contribute nothing: dx starts at zero when there is one.
    bool empty_phase = false;
    for (int64_t a = 0; a < s.sh; ++a)
        for (int64_t b = 0; b < s.sw; ++b) {
            DgradAxis ah, aw;
            if (!dgrad_axis(a, s.h, s.sh, s.ph, s.dh, s.r, &ah) || !dgrad_axis(b, s.w, s.sw, s.pw, s.dw, s.s, &aw))
                continue;
            if (ah.taps == 0 || aw.taps == 0) empty_phase = true;
        }
    if (empty_phase && cudaMemsetAsync(dx, 0, dx_bytes, stream) != cudaSuccess) return CONV2D_ERR_CUDA;
    int launches = 0;
    for (int64_t a = 0; a < s.sh; ++a)
        for (int64_t b = 0; b < s.sw; ++b) {
            DgradAxis ah, aw;
            if (!dgrad_axis(a, s.h, s.sh, s.ph, s.dh, s.r, &ah) || !dgrad_axis(b, s.w, s.sw, s.pw, s.dw, s.s, &aw))
                continue;
            if (ah.taps == 0 || aw.taps == 0) continue;
            rc = launch_dgrad_phase(s, ah, aw, a, b, dy, w, dx, workspace, workspace_bytes, stream, algo);
            if (rc != CONV2D_OK) return rc;
            ++launches;
        }
    g_last_launches = launches;
    return CONV2D_OK;
}

int run_wgrad(const conv2d_params* params, const void* x, const void* dy, float* dw, void* workspace,
              size_t workspace_bytes, cudaStream_t stream, const conv2d_algo* algo)
{
    g_last_launches = 0;
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (s.k == 0) return CONV2D_OK;  // no filters: nothing to write
    if (!dw || (s.m > 0 && (!x || !dy))) return CONV2D_ERR_INVALID;
    if (!aligned16(dw) || (x && !aligned16(x)) || (dy && !aligned16(dy)) || (workspace && !aligned16(workspace)))
        return CONV2D_ERR_ALIGNMENT;
    if (algo && (algo->splits < 0 || algo->block_n < 0 || algo->block_m < 0 || algo->grid < 0 ||
                 algo->wait_limit_ns < 0 || algo->reduction < CONV2D_REDUCTION_AUTO ||
                 algo->reduction > CONV2D_REDUCTION_CONCURRENT))
        return CONV2D_ERR_INVALID;
    if (!wgrad_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    if (s.m == 0) {  // empty batch: the gradient is zero
        if (cudaMemsetAsync(dw, 0, static_cast<size_t>(s.k * s.crs) * sizeof(float), stream) != cudaSuccess)
            return CONV2D_ERR_CUDA;
        return CONV2D_OK;
    }
    WgradPlan plan;
    rc = choose_wgrad_plan(s, algo, &plan);
    if (rc != CONV2D_OK) return rc;
    const bool have_ws = workspace && workspace_bytes >= wgrad_workspace_bytes_for(s);
    const bool cuts = wgrad_cuts_tiles(plan);
    if (cuts && !have_ws) return CONV2D_ERR_WORKSPACE;
    if (workspace && !have_ws) return CONV2D_ERR_WORKSPACE;
    if (!load_encoders()) return CONV2D_ERR_CUDA;

    CUtensorMap tm_a, tm_b;
    std::memset(&tm_a, 0, sizeof(tm_a));
    std::memset(&tm_b, 0, sizeof(tm_b));
    {   // dy as [N*P*Q][K]: boxes of 64 channels x 64 output pixels, 128-byte swizzle
        const cuuint64_t dims[2] = {(cuuint64_t)s.k, (cuuint64_t)s.m};
        const cuuint64_t strides[1] = {(cuuint64_t)(s.k * 2)};
        const cuuint32_t box[2] = {64, (cuuint32_t)BK};
        const cuuint32_t estr[2] = {1, 1};
        if (g_encode_tiled(&tm_a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(dy), dims, strides, box,
                           estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }
    {   // x as im2col boxes of 64 output pixels x 64 channels (the forward map with 64-pixel columns)
        const cuuint64_t dims[4] = {(cuuint64_t)s.c, (cuuint64_t)s.w, (cuuint64_t)s.h, (cuuint64_t)s.n};
        const cuuint64_t strides[3] = {(cuuint64_t)(s.c * 2), (cuuint64_t)(s.w * s.c * 2),
                                       (cuuint64_t)(s.h * s.w * s.c * 2)};
        const int lower[2] = {(int)-s.pw, (int)-s.ph};
        const int upper[2] = {(int)(s.pw - (s.s - 1) * s.dw), (int)(s.ph - (s.r - 1) * s.dh)};
        const cuuint32_t estr[4] = {1, (cuuint32_t)s.sw, (cuuint32_t)s.sh, 1};
        if (g_encode_im2col(&tm_b, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, lower,
                            upper, BK, BK, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return CONV2D_ERR_CUDA;
    }

    sgb::ConvKernelParams kp{};
    kp.x = static_cast<const uint16_t*>(x);
    kp.w = nullptr;
    kp.bias = nullptr;
    kp.y = dw;
    kp.ldy = static_cast<int>(s.crs);
    kp.status = have_ws ? static_cast<uint32_t*>(workspace) : nullptr;
    kp.sems = have_ws ? reinterpret_cast<uint32_t*>(static_cast<char*>(workspace) + kStatusBytes) : nullptr;
    kp.N = (int)s.n; kp.H = (int)s.h; kp.W = (int)s.w; kp.C = (int)s.c;
    kp.K = (int)s.k; kp.R = (int)s.r; kp.S = (int)s.s; kp.P = (int)s.p; kp.Q = (int)s.q;
    kp.sh = (int)s.sh; kp.sw = (int)s.sw; kp.ph = (int)s.ph; kp.pw = (int)s.pw; kp.dh = (int)s.dh; kp.dw = (int)s.dw;
    kp.M = (int)s.k;        // GEMM rows: output channels
    kp.CRS = (int)s.m;      // reduction length: output pixels
    kp.G = (int)(s.r * s.s);  // column blocks never straddle a tap: R*S "groups" of C columns
    kp.Cg = (int)s.c;
    kp.Kg = (int)s.c;
    kp.ntpg = plan.ntpt;
    kp.num_kb = plan.num_kb;
    kp.m_tiles = plan.m_tiles;
    kp.n_tiles = plan.n_tiles;
    kp.grid = plan.grid;
    kp.units = plan.units;
    kp.vec_store = 1;  // C % 64 == 0: every row and column block is 16-byte aligned
    kp.debug_flags = algo ? algo->debug_flags : 0;
    kp.reduce_concurrent = (algo && algo->reduction == CONV2D_REDUCTION_ORDERED) ? 0 : 1;
    kp.wait_limit_ns = (algo && algo->wait_limit_ns > 0) ? (unsigned long long)algo->wait_limit_ns : kDefaultWaitNs;
    kp.trace = nullptr;
#ifdef SGB_TRACE_ENABLED
    kp.trace = g_trace;
#endif
    if (log_enabled())
        std::fprintf(stderr, "[conv2d wgrad] K=%lld RSC=%lld NPQ=%lld -> BN=%d splits=%d grid=%d kb=%d tiles=%d\n",
                     (long long)s.k, (long long)s.crs, (long long)s.m, plan.block_n, plan.splits, plan.grid,
                     plan.num_kb, plan.m_tiles * plan.n_tiles);
    cudaError_t err;
    if (plan.block_n == 64) err = sgb::launch_conv2d_tc<128, 64, sgb::LOADER_WGRAD>(tm_a, tm_b, kp, plan.grid, stream);
    else if (plan.block_n == 128) err = sgb::launch_conv2d_tc<128, 128, sgb::LOADER_WGRAD>(tm_a, tm_b, kp, plan.grid, stream);
    else err = sgb::launch_conv2d_tc<128, 256, sgb::LOADER_WGRAD>(tm_a, tm_b, kp, plan.grid, stream);
    if (err != cudaSuccess) return CONV2D_ERR_CUDA;
    g_last_launches = 1;
    return CONV2D_OK;
}


}  // namespace

namespace sgb {
// The smallest workspace a plain forward call can run with (no block-diagonal
// weight: grouped layers then take the direct kernel or the plain grouped path).
size_t fwd_workspace_bytes_min(const conv2d_params* params)
{
    Shape s;
    if (make_shape(params, &s) != CONV2D_OK) return 0;
    return workspace_bytes_for(s);
}
}  // namespace sgb

extern "C" {

int conv2d_fwd_output_shape(const conv2d_params* params, int64_t* p, int64_t* q)
{
    Shape s;
    const int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (p) *p = s.p;
    if (q) *q = s.q;
    return CONV2D_OK;
}

size_t conv2d_fwd_workspace_bytes(const conv2d_params* params)
{
    Shape s;
    if (make_shape(params, &s) != CONV2D_OK) return 0;
    size_t need = workspace_bytes_for(s);
    if (blockdiag_eligible(s)) {  // room for the block-diagonal weight after the semaphores
        const size_t bd = round256(workspace_bytes_for(blockdiag_shape(s))) + blockdiag_weight_bytes(s);
        if (bd > need) need = bd;
    }
    return need;
}


int conv2d_fwd_ex(const conv2d_params* params, const void* x_dev, const void* w_dev, const float* bias_dev,
                  float* y_dev, void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream,
                  const conv2d_algo* algo)
{
    return run_conv(params, x_dev, w_dev, bias_dev, y_dev, workspace_dev, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream), algo);
}

int conv2d_fwd_epi(const conv2d_params* params, const void* x_dev, const void* w_dev, const float* bias_dev,
                   void* y_dev, void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream,
                   const conv2d_algo* algo, const conv2d_epilogue* epi)
{
    return run_conv(params, x_dev, w_dev, bias_dev, static_cast<float*>(y_dev), workspace_dev, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream), algo, epi);
}

int conv2d_fwd(const conv2d_params* params, const void* x_dev, const void* w_dev, const float* bias_dev,
               float* y_dev, void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream)
{
    return run_conv(params, x_dev, w_dev, bias_dev, y_dev, workspace_dev, workspace_bytes,
                    reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int conv2d_fwd_query_algo_epi(const conv2d_params* params, const conv2d_epilogue* epi, conv2d_algo* out)
{
    if (!out) return CONV2D_ERR_INVALID;
    if (epi && (epi->activation < CONV2D_ACT_NONE || epi->activation > CONV2D_ACT_RELU ||
                epi->out_dtype < CONV2D_OUT_F32 || epi->out_dtype > CONV2D_OUT_BF16))
        return CONV2D_ERR_INVALID;
    const bool fused = epi && (epi->activation != CONV2D_ACT_NONE || epi->out_dtype != CONV2D_OUT_F32);
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (blockdiag_eligible(s)) {  // with the workspace conv2d_fwd(_epi)_workspace_bytes asks for
        Plan tplan;
        if (choose_plan(blockdiag_shape(s), nullptr, &tplan, fused) == CONV2D_OK) {
            std::memset(out, 0, sizeof(*out));
            out->loader = CONV2D_LOADER_BLOCKDIAG;
            return CONV2D_OK;
        }
    }
    if (direct_eligible(s)) {
        std::memset(out, 0, sizeof(*out));
        out->loader = CONV2D_LOADER_DIRECT;
        out->grid = static_cast<int32_t>(direct_grid(s));
        return CONV2D_OK;
    }
    Plan plan;
    rc = choose_plan(s, nullptr, &plan, fused);
    if (rc != CONV2D_OK) return rc;
    std::memset(out, 0, sizeof(*out));
    out->block_m = plan.block_m;
    out->block_n = plan.block_n;
    out->splits = plan.splits;
    out->loader = plan.loader;
    out->grid = plan.grid;
    const bool cuts = plan_cuts_tiles(plan);
    out->reduction = cuts ? CONV2D_REDUCTION_CONCURRENT : CONV2D_REDUCTION_AUTO;
    return CONV2D_OK;
}

size_t conv2d_fwd_epi_workspace_bytes(const conv2d_params* params, const conv2d_algo* algo,
                                      const conv2d_epilogue* epi)
{
    Shape s;
    if (make_shape(params, &s) != CONV2D_OK) return 0;
    const bool fused = epi && (epi->activation != CONV2D_ACT_NONE || epi->out_dtype != CONV2D_OUT_F32);
    if (!fused) return conv2d_fwd_workspace_bytes(params);
    Plan plan;
    size_t need = workspace_bytes_for(s);
    if (s.m > 0 && s.k > 0 && choose_plan(s, algo, &plan, true) == CONV2D_OK) need = workspace_bytes_for_plan(s, plan, true);
    if (s.m > 0 && s.k > 0 && blockdiag_eligible(s) && (nothing_forced(algo) || algo->loader == CONV2D_LOADER_BLOCKDIAG)) {
        const Shape t = blockdiag_shape(s);
        Plan tplan;
        if (choose_plan(t, nullptr, &tplan, true) == CONV2D_OK) {
            const size_t bd = round256(workspace_bytes_for_plan(t, tplan, true)) + blockdiag_weight_bytes(s);
            if (bd > need) need = bd;
        }
    }
    return need;
}

int conv2d_fwd_query_algo(const conv2d_params* params, conv2d_algo* out)
{
    return conv2d_fwd_query_algo_epi(params, nullptr, out);
}

size_t conv2d_bwd_data_workspace_bytes(const conv2d_params* params)
{
    Shape s;
    if (make_shape(params, &s) != CONV2D_OK) return 0;
    return workspace_bytes_for(dgrad_forward_shape(s));
}

int conv2d_bwd_data(const conv2d_params* params, const void* dy_dev, const void* w_dev, float* dx_dev,
                    void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream, const conv2d_algo* algo)
{
    return run_dgrad(params, dy_dev, w_dev, dx_dev, workspace_dev, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream), algo);
}

int conv2d_bwd_data_query_algo(const conv2d_params* params, conv2d_algo* out)
{
    if (!out) return CONV2D_ERR_INVALID;
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (!dgrad_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    // The plan of the first phase with taps (stride 1: the only one).
    Shape t = dgrad_forward_shape(s);
    bool found = false;
    for (int64_t a = 0; a < s.sh && !found; ++a)
        for (int64_t b = 0; b < s.sw && !found; ++b) {
            DgradAxis ah, aw;
            if (dgrad_axis(a, s.h, s.sh, s.ph, s.dh, s.r, &ah) && dgrad_axis(b, s.w, s.sw, s.pw, s.dw, s.s, &aw) &&
                ah.taps > 0 && aw.taps > 0) {
                t = dgrad_phase_shape(s, ah, aw);
                found = true;
            }
        }
    Plan plan;
    rc = dgrad_plan(t, nullptr, &plan);
    if (rc != CONV2D_OK) return rc;
    std::memset(out, 0, sizeof(*out));
    out->block_m = plan.block_m;
    out->block_n = plan.block_n;
    out->splits = plan.splits;
    out->loader = plan.loader;
    out->grid = plan.grid;
    out->reduction = plan_cuts_tiles(plan) ? CONV2D_REDUCTION_CONCURRENT : CONV2D_REDUCTION_AUTO;
    return CONV2D_OK;
}

size_t conv2d_bwd_weight_workspace_bytes(const conv2d_params* params)
{
    Shape s;
    if (make_shape(params, &s) != CONV2D_OK) return 0;
    return wgrad_workspace_bytes_for(s);
}

int conv2d_bwd_weight(const conv2d_params* params, const void* x_dev, const void* dy_dev, float* dw_dev,
                      void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream, const conv2d_algo* algo)
{
    return run_wgrad(params, x_dev, dy_dev, dw_dev, workspace_dev, workspace_bytes,
                     reinterpret_cast<cudaStream_t>(stream), algo);
}

int conv2d_bwd_weight_query_algo(const conv2d_params* params, conv2d_algo* out)
{
    if (!out) return CONV2D_ERR_INVALID;
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (!wgrad_eligible(s)) return CONV2D_ERR_UNSUPPORTED;
    WgradPlan plan;
    rc = choose_wgrad_plan(s, nullptr, &plan);
    if (rc != CONV2D_OK) return rc;
    std::memset(out, 0, sizeof(*out));
    out->block_m = 128;
    out->block_n = plan.block_n;
    out->splits = plan.splits;
    out->loader = CONV2D_LOADER_TMA_IM2COL;
    out->grid = plan.grid;
    out->reduction = wgrad_cuts_tiles(plan) ? CONV2D_REDUCTION_CONCURRENT : CONV2D_REDUCTION_AUTO;
    return CONV2D_OK;
}

int conv2d_fwd_status(void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream)
{
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (!workspace_dev) return CONV2D_OK;
    if (workspace_bytes < sizeof(uint32_t)) return CONV2D_ERR_WORKSPACE;
    uint32_t status = 0;
    if (cudaMemcpy(&status, workspace_dev, sizeof(status), cudaMemcpyDeviceToHost) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    if (status == 0) return CONV2D_OK;
    if (cudaMemset(workspace_dev, 0, workspace_bytes) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess) return CONV2D_ERR_CUDA;
    return status == CONV2D_ERR_TIMEOUT ? CONV2D_ERR_TIMEOUT : CONV2D_ERR_CUDA;
}

size_t conv2d_fwd_host_staging_bytes(const conv2d_params* params)
{
    Shape s;
    if (make_shape(params, &s) != CONV2D_OK) return 0;
    return round256(s.n * s.h * s.w * s.c * 2) + round256(s.k * s.crs * 2) + round256(s.k * 4) +
           round256(s.m * s.k * 4) + round256(workspace_bytes_for(s));
}

int conv2d_fwd_host(const conv2d_params* params, const void* x_host, const void* w_host, const float* bias_host,
                    float* y_host, void* staging_dev, size_t staging_bytes, conv2d_stream_t stream)
{
    g_last_launches = 0;
    Shape s;
    int rc = make_shape(params, &s);
    if (rc != CONV2D_OK) return rc;
    if (s.m == 0 || s.k == 0) return CONV2D_OK;
    if (!x_host || !w_host || !y_host || !staging_dev) return CONV2D_ERR_INVALID;
    if (staging_bytes < conv2d_fwd_host_staging_bytes(params)) return CONV2D_ERR_WORKSPACE;
    if (!aligned16(staging_dev)) return CONV2D_ERR_ALIGNMENT;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* base = static_cast<char*>(staging_dev);
    const size_t xb = s.n * s.h * s.w * s.c * 2, wb = s.k * s.crs * 2, bb = s.k * 4, yb = s.m * s.k * 4;
    char* xd = base;
    char* wd = xd + round256(xb);
    char* bd = wd + round256(wb);
    char* yd = bd + round256(bb);
    char* ws = yd + round256(yb);
    if (cudaMemcpyAsync(xd, x_host, xb, cudaMemcpyHostToDevice, st) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (cudaMemcpyAsync(wd, w_host, wb, cudaMemcpyHostToDevice, st) != cudaSuccess) return CONV2D_ERR_CUDA;
    if (bias_host && cudaMemcpyAsync(bd, bias_host, bb, cudaMemcpyHostToDevice, st) != cudaSuccess)
        return CONV2D_ERR_CUDA;
    rc = run_conv(params, xd, wd, bias_host ? reinterpret_cast<float*>(bd) : nullptr, reinterpret_cast<float*>(yd),
                  ws, workspace_bytes_for(s), st, nullptr);
    if (rc != CONV2D_OK) return rc;
    if (cudaMemcpyAsync(y_host, yd, yb, cudaMemcpyDeviceToHost, st) != cudaSuccess) return CONV2D_ERR_CUDA;
    return CONV2D_OK;
}

int conv2d_last_launch_count(void) { return g_last_launches; }

void conv2d_tensor_map_cache_stats(unsigned long long* hits, unsigned long long* misses)
{
    std::lock_guard<std::mutex> lock(g_map_mutex);
    if (hits) *hits = g_map_hits;
    if (misses) *misses = g_map_misses;
}

#ifdef SGB_TRACE_ENABLED
// Profiling builds only: device buffer of grid x 16 timestamps that later launches fill.
void conv2d_debug_set_trace(void* trace_dev) { g_trace = static_cast<unsigned long long*>(trace_dev); }
#endif

const char* conv2d_strerror(int status)
{
    switch (status) {
        case CONV2D_OK: return "ok";
        case CONV2D_ERR_INVALID: return "invalid argument (sizes, options or pointers)";
        case CONV2D_ERR_UNSUPPORTED: return "unsupported (sizes beyond 32-bit indexing, or a forced algo that cannot run)";
        case CONV2D_ERR_ALIGNMENT: return "device pointer not 16-byte aligned";
        case CONV2D_ERR_WORKSPACE: return "workspace missing or too small";
        case CONV2D_ERR_CUDA: return "CUDA runtime or driver error";
        case CONV2D_ERR_TIMEOUT: return "a device-side wait ran out (workspace reset)";
        case CONV2D_ERR_SCRATCH_LIMIT:
            return "problem needs more workspace than the no-allocation entry point's static scratch array holds";
        default: return "unknown status";
    }
}

}  // extern "C"
