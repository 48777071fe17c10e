/*
 * conv2d.h -- C ABI of the GB300 (sm_103a) implicit-GEMM 2-D convolution forward.
 *
 * The operation: y = conv2d(x, w) + bias, computed as an implicit GEMM
 *   M = N*P*Q output pixels, GEMM-N = K output channels, reduction over C*R*S,
 * with the im2col operand formed on the fly in the loader and never written to
 * memory.  Sources for the definition and its pieces:
 *   - the convolution itself and its NHWC/KRSC layouts: docs.rs burn-cubecl 0.20.0,
 *     burn_cubecl/kernel/conv/base.rs, conv_forward / conv_forward_nhwc (input and
 *     weight both permuted NCHW->NHWC, i.e. weight [K][R][S][C]);
 *   - "The bias added to each channel": the same page, conv_forward's doc comment;
 *   - implicit GEMM as the conv algorithm: burn PR #2287 "Introduce autotuning to
 *     conv2d and conv_transpose2d ..." (Changes) and burn PR #2545 "[Optimization]
 *     Implicit gemm rewrite" (Changes);
 *   - split-K with an in-place, serialised reduction on a per-tile semaphore, the
 *     fp32 output doubling as the work buffer: NVIDIA/Fuser issue #1316 "Split-K
 *     matmul is slow even for few partitions" (Eliminating the workspace, and the
 *     comment on aliasing the output buffer).
 *
 * Math (cross-correlation, zero padding):
 *   y[n][p][q][k] = bias[k] + sum_{r,s,c} x[n][p*sh-ph+r*dh][q*sw-pw+s*dw][g*Cg + c] * w[k][r][s][c]
 *   with G = groups, Cg = C/G, Kg = K/G, g = k / Kg and c over 0 .. Cg-1: the
 *   channels split into G equal consecutive groups, each output channel summing
 *   over its own group's input channels (burn's ConvOptions carry `groups`; its
 *   implicit GEMM sends G != 1 to the direct strategy, burn-cubecl base.rs
 *   conv_forward_nhwc).  G = 1 is the ordinary convolution.
 *   P = floor((H + 2*ph - dh*(R-1) - 1)/sh) + 1,  Q likewise.
 * Inputs are bf16, products are exact in fp32, accumulation is fp32 (tensor
 * cores, TMEM), the output is fp32.
 *
 * Conventions for every entry point:
 *   - Status is returned as an int (conv2d_status); nothing throws across the ABI.
 *   - Pointers named *_dev are device pointers owned by the caller; pointers
 *     named *_host are host pointers owned by the caller.  The library never
 *     frees or retains them beyond the call.
 *   - Tensors are dense and contiguous: x is [N][H][W][C] bf16, w is
 *     [K][R][S][C/groups] bf16, bias is [K] fp32, y is [N][P][Q][K] fp32.
 *   - Device pointers must be 16-byte aligned, or the call returns
 *     CONV2D_ERR_ALIGNMENT.
 *   - Device work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and the call returns without waiting for it.
 *   - Nothing is allocated on the device by these calls.
 */
#ifndef SPLIT_GEMM_GB300_CONV2D_H
#define SPLIT_GEMM_GB300_CONV2D_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; declared here so that this header needs no CUDA headers. */
typedef struct CUstream_st* conv2d_stream_t;

/* Problem description.  Options follow burn's ConvOptions (stride, padding,
 * dilation, groups); padding is symmetric (pad_h rows above and below). */
typedef struct {
    int64_t n, h, w, c;  /* input  NHWC */
    int64_t k, r, s;     /* weight KRSC: k output channels, r x s filter */
    int32_t stride_h, stride_w;
    int32_t pad_h, pad_w;
    int32_t dil_h, dil_w;
    int32_t groups;      /* >= 1, dividing both c and k (CONV2D_ERR_INVALID otherwise) */
} conv2d_params;

typedef enum {
    CONV2D_OK = 0,
    CONV2D_ERR_INVALID = 1,     /* bad sizes/options, NULL pointer, empty window */
    CONV2D_ERR_UNSUPPORTED = 2, /* sizes beyond 32-bit index range, or a forced algo that cannot run */
    CONV2D_ERR_ALIGNMENT = 3,   /* a device pointer is not 16-byte aligned */
    CONV2D_ERR_WORKSPACE = 4,   /* workspace missing or smaller than conv2d_fwd_workspace_bytes() */
    CONV2D_ERR_CUDA = 5,        /* a CUDA runtime/driver call failed */
    CONV2D_ERR_TIMEOUT = 6,     /* a device-side wait ran out (reported by conv2d_fwd_status) */
    CONV2D_ERR_SCRATCH_LIMIT = 7 /* conv2d_fwd_noalloc: problem needs more than CONV2D_NOALLOC_SCRATCH_BYTES */
} conv2d_status;

/* Loader kinds for the im2col (activation) operand. */
typedef enum {
    CONV2D_LOADER_AUTO = 0,
    CONV2D_LOADER_TMA_IM2COL = 1, /* TMA im2col-mode descriptor; needs C/groups % 64 == 0 */
    CONV2D_LOADER_CPASYNC = 2,    /* 16-byte cp.async gather; needs C/groups % 8 == 0 */
    CONV2D_LOADER_SCALAR = 3,     /* element gather; any C (also gathers the weight) */
    CONV2D_LOADER_HYBRID = 4,     /* TMA im2col and cp.async gather on alternate k-blocks; needs C/groups % 64 == 0 */
    CONV2D_LOADER_ROW_WINDOW = 5, /* few channels: staged input rows read in place by the MMA as overlapping
                                     16-byte-pitch windows; needs groups == 1, dil_w == 1, stride_w in {1,2,4,8},
                                     C <= 8 / stride_w, K <= 256 (one tile of output channels), no split */
    CONV2D_LOADER_TMA_BOX = 6,    /* tiles are rectangles of output pixels; each tiled TMA box carries two
                                     64-channel chunks of one filter tap (and a 3-D box two weight k-blocks);
                                     needs groups == 1, C % 128 == 0, strides <= 8, and block_n <= 128
                                     with 256-pixel tiles */
    CONV2D_LOADER_HALO = 7,       /* stride 1 only: a tile is 128 consecutive pixels of an image seen with the
                                     padded row pitch W + 2*pad_w (pixels past Q are computed and discarded);
                                     per 64-channel chunk one tiled TMA box of whole padded input rows serves
                                     every filter tap, which the MMA reads in place at the tap's row offset.
                                     Needs groups == 1, C % 64 == 0, W + 2*pad_w <= 256, 128-pixel tiles, and the two halo
                                     buffers plus the weight ring within shared memory (block_n is narrowed
                                     to fit unless forced) */
    CONV2D_LOADER_DIRECT = 8,     /* not an implicit GEMM: a CUDA-core direct convolution for groups of few
                                     channels, one thread per (output pixel, group) in fp32 FMAs, the group
                                     weights in shared memory.  Needs groups > 1, C/groups == K/groups in
                                     {1, 2, 4, 8, 16} (depthwise: 1), C % 8 == 0, and the weights
                                     (K*R*S*C/groups fp32) within shared memory.  The heuristic takes it for such shapes when nothing else
                                     is forced; block_n, block_m and splits do not apply */
    CONV2D_LOADER_TMA_PAIR = 9,   /* TMA im2col loads on clusters of two CTAs: a tile is 256 output pixels x
                                     block_n (64/128/256) channels computed by 2-CTA tensor-core MMAs
                                     (each CTA loads 128 pixel rows and half the weight rows), two 64-wide
                                     k-blocks per pipeline stage.  Needs groups == 1, C % 64 == 0,
                                     K % 4 == 0; block_m is 256 (or 0); grid counts CTA pairs; a fused
                                     epilogue runs on whole tiles only.  The heuristic takes it for such
                                     shapes when nothing else is forced */
    CONV2D_LOADER_PAIR_HALO = 10, /* stride 1 on clusters of two CTAs: each CTA holds 128 consecutive pixels of
                                     one image seen with the padded row pitch W + 2*pad_w (pixels past Q are
                                     computed and discarded), the pair the same pixels of two images; per
                                     64-channel chunk one tiled TMA box of whole padded input rows serves every
                                     filter tap, read in place by 2-CTA tensor-core MMAs, and the weights of
                                     two or three taps come in one box per stage.  Needs stride 1,
                                     C/groups % 64 == 0, K/groups % 4 == 0 (a column block lies in one group),
                                     W + 2*pad_w <= 256 and the two halo buffers within shared memory; block_m
                                     is 256 (or 0); grid counts CTA pairs.  The heuristic takes it for
                                     ungrouped layers only */
    CONV2D_LOADER_BLOCKDIAG = 11  /* grouped convolution with C/groups == K/groups = cg in {8, 16, 32} and groups a
                                     multiple of 64/cg: 64/cg groups merged into one 64-channel group whose weight
                                     is block-diagonal (zeros outside each output channel's own group), expanded
                                     into the workspace by a first launch (K*R*S*64 bf16 after the semaphores;
                                     conv2d_fwd_workspace_bytes includes it), then the grouped implicit GEMM on
                                     TMA im2col boxes.  The heuristic's choice for such layers when the
                                     workspace has room (else the direct kernel); forcing it needs the room.
                                     Only reported by the query functions or forced: no other field may be set
                                     with it */
} conv2d_loader;

/* Kernel configuration.  All-zero fields mean "let the heuristic choose".
 * Work is split stream-K style: the (tile, k-block) units are divided evenly
 * over `grid` CTAs, and a tile cut between CTAs is reduced in place in y, the
 * CTAs taking turns on a per-tile semaphore.  `splits` = S forces classic
 * split-K instead (grid = tiles * S, every tile cut into S equal parts). */
typedef struct {
    int32_t block_n;   /* output channels per CTA tile: 64, 128 or 256 */
    int32_t splits;    /* classic split-K factor S >= 1; 0 = stream-K */
    int32_t loader;    /* conv2d_loader */
    int32_t grid;      /* CTAs for stream-K (1 .. tiles * k-blocks); 0 = heuristic */
    int32_t debug_flags;      /* test hook, 0 in normal use; see CONV2D_DEBUG_* */
    int32_t block_m;          /* output pixels per CTA tile: 128, or 256 (TMA im2col and TMA box loaders) */
    int64_t wait_limit_ns;    /* bound on every device-side wait; 0 = default (1 s) */
    int32_t reduction;        /* conv2d_reduction: how the splits of a cut tile meet in y */
} conv2d_algo;

/* In-place reduction of a tile cut between CTAs.  Either way split 0 stores
 * first (with the bias) and the only memory besides y is one semaphore per tile. */
typedef enum {
    CONV2D_REDUCTION_AUTO = 0,       /* the heuristic's choice (concurrent) */
    CONV2D_REDUCTION_ORDERED = 1,    /* later splits add in k-order, one at a time: bitwise reproducible */
    CONV2D_REDUCTION_CONCURRENT = 2  /* later splits add as they finish (fp32 atomic adds in L2): results
                                        may differ between runs in the last bits, within the fp32
                                        summation bound */
} conv2d_reduction;

/* Test hook: split 0 of every tile skips its semaphore signal, so later splits'
 * bounded waits run out and the call reports CONV2D_ERR_TIMEOUT. */
#define CONV2D_DEBUG_SKIP_SIGNAL 1
/* Measurement hooks of the CTA-pair loader (CONV2D_LOADER_TMA_PAIR): force one
 * or two 64-wide k-blocks per pipeline stage instead of the heuristic's choice. */
#define CONV2D_DEBUG_PAIR_KB1 2
#define CONV2D_DEBUG_PAIR_KB2 4
/* Measurement hook of the CTA-pair loaders: write fp32 y through TMA stores
 * and TMA reductions of staged 64-row boxes instead of per-thread vector
 * stores (measured slower on GB300, so not the default). */
#define CONV2D_DEBUG_TMA_STORE 8

/* Output extents P and Q (pure host computation).  Returns CONV2D_OK or
 * CONV2D_ERR_INVALID (bad options, or the filter window does not fit). */
int conv2d_fwd_output_shape(const conv2d_params* params, int64_t* p, int64_t* q);

/* Bytes of device workspace conv2d_fwd needs for these params with any
 * algorithm: a status word plus one semaphore per output tile.  The workspace
 * must be zero-filled before its first use; the kernels leave it zeroed after
 * every successful call (the last split of a tile resets its semaphore). */
size_t conv2d_fwd_workspace_bytes(const conv2d_params* params);

/* The forward convolution.  x_dev, w_dev, y_dev: device tensors as above;
 * bias_dev: [K] fp32 or NULL.  y is fully overwritten (its prior contents are
 * ignored, also under split-K).  workspace_dev/workspace_bytes: see
 * conv2d_fwd_workspace_bytes (may be NULL/0 only if the chosen split factor is 1).
 * The algorithm is chosen by the host heuristic (conv2d_fwd_query_algo). */
int conv2d_fwd(const conv2d_params* params, const void* x_dev, const void* w_dev,
               const float* bias_dev, float* y_dev, void* workspace_dev,
               size_t workspace_bytes, conv2d_stream_t stream);

/* As conv2d_fwd with a forced configuration (any zero field is chosen by the
 * heuristic).  Returns CONV2D_ERR_UNSUPPORTED if the forced configuration
 * cannot run these params (e.g. the TMA loader with C % 64 != 0). */
int conv2d_fwd_ex(const conv2d_params* params, const void* x_dev, const void* w_dev,
                  const float* bias_dev, float* y_dev, void* workspace_dev,
                  size_t workspace_bytes, conv2d_stream_t stream, const conv2d_algo* algo);

/* What the heuristic picks for these params (tile width, split factor, loader),
 * without launching anything.  Needs no device pointers; uses the current
 * device's SM count. */
int conv2d_fwd_query_algo(const conv2d_params* params, conv2d_algo* out);

/* Synchronises `stream`, then reads the workspace's device status word.
 * Returns CONV2D_OK, CONV2D_ERR_TIMEOUT if a device-side wait ran out during a
 * call that used this workspace, or CONV2D_ERR_CUDA.  After a timeout it zeroes
 * the whole workspace (status and semaphores) so that it can be used again; the
 * output of the failed call is undefined. */
int conv2d_fwd_status(void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream);

/* Bytes of device staging memory conv2d_fwd_host needs: room for x, w, bias,
 * y and the workspace, each 256-byte aligned. */
size_t conv2d_fwd_host_staging_bytes(const conv2d_params* params);

/* End-to-end call for callers whose tensors live in host memory: enqueues on
 * `stream` the host->device copies of x_host, w_host and bias_host (NULL for no
 * bias), the convolution, and the device->host copy of y into y_host.  The
 * caller provides `staging_dev` (conv2d_fwd_host_staging_bytes bytes of device
 * memory that the library partitions; its workspace part must be zero before
 * the first call and stays zero afterwards).  Host buffers should be pinned for
 * the copies to be asynchronous; y_host is valid after the stream synchronises. */
int conv2d_fwd_host(const conv2d_params* params, const void* x_host, const void* w_host,
                    const float* bias_host, float* y_host, void* staging_dev,
                    size_t staging_bytes, conv2d_stream_t stream);

/* Number of kernel launches the last successful conv2d_fwd* call on this host
 * thread enqueued (1 for every algorithm; 0 before any call and for empty problems). */
int conv2d_last_launch_count(void);

/* Tensor-map cache of the forward entry points (conv2d_fwd, conv2d_fwd_ex,
 * conv2d_fwd_epi, conv2d_fwd_host, conv2d_fwd_noalloc).  The TMA descriptors a
 * call needs are encoded on the host; a small process-wide cache (32 entries,
 * replaced in turn) keyed on the problem (params), the plan's loader and tile
 * geometry, the x and w pointers and the current device reuses them on
 * repeated calls, so a call on buffers seen before skips the driver's encoding.
 * The pages have no counterpart (burn's conv_forward has no descriptors to
 * encode); it removes per-call host cost of this boundary.  Any change of
 * pointer, shape or plan encodes afresh.  This reports how many lookups
 * found an entry (hits) and how many encoded (misses) since the library was
 * loaded; either pointer may be NULL.  Thread-safe. */
void conv2d_tensor_map_cache_stats(unsigned long long* hits, unsigned long long* misses);

/* Fused epilogue.  After the bias, the epilogue may apply an activation and
 * may store y in bf16 instead of fp32:
 *   y[n][p][q][k] = round_out(act(acc + bias[k]))
 * with act = identity or ReLU (max(v, 0), applied to the fp32 value) and
 * round_out = identity (fp32 y) or fp32 -> bf16 round to nearest even.
 * A bf16 output cannot hold the partial sums of a tile cut between CTAs (the
 * in-place reduction needs the fp32 accumulator type in y; NVIDIA/Fuser issue
 * #1316 "Split-K matmul is slow even for few partitions", the comment on
 * aliasing the output as the reduction work buffer, notes the same for a
 * half-precision output), and ReLU needs the finished sum.  So under a fused
 * epilogue the splits of a cut tile add their partial sums into a separate
 * fp32 [M][K] buffer in the workspace (atomic adds in L2, no waiting), and the
 * CTA that arrives last at the tile's counter reads the complete sum back, adds
 * the bias, applies the activation, converts, stores y and zeroes its part of
 * the buffer again.  The heuristic still splits few-tile, long-reduction
 * problems (classic split-K); where it would cut tiles stream-K style over many
 * tiles it gives each CTA whole tiles instead.  conv2d_fwd_epi_workspace_bytes
 * gives the workspace a fused call needs. */
typedef enum {
    CONV2D_ACT_NONE = 0,
    CONV2D_ACT_RELU = 1
} conv2d_activation;

typedef enum {
    CONV2D_OUT_F32 = 0,   /* y is float[N][P][Q][K] */
    CONV2D_OUT_BF16 = 1   /* y is bf16 (uint16 bit patterns) [N][P][Q][K] */
} conv2d_out_dtype;

typedef struct {
    int32_t activation;  /* conv2d_activation */
    int32_t out_dtype;   /* conv2d_out_dtype */
} conv2d_epilogue;

/* conv2d_fwd_ex with a fused epilogue.  y_dev points to N*P*Q*K values of the
 * type `epi->out_dtype` names (16-byte aligned, caller-owned, fully
 * overwritten).  algo may be NULL (heuristic); epi may be NULL, which is the
 * plain fp32 epilogue and then this call is conv2d_fwd_ex itself.  Returns
 * CONV2D_ERR_INVALID for an unknown activation or output type, and
 * CONV2D_ERR_WORKSPACE when the plan cuts tiles and the workspace is smaller
 * than conv2d_fwd_epi_workspace_bytes(params, algo, epi).  The workspace
 * follows the rules of conv2d_fwd's (zero before first use; left zero by every
 * successful call, partial-sum buffer included). */
int conv2d_fwd_epi(const conv2d_params* params, const void* x_dev, const void* w_dev,
                   const float* bias_dev, void* y_dev, void* workspace_dev,
                   size_t workspace_bytes, conv2d_stream_t stream, const conv2d_algo* algo,
                   const conv2d_epilogue* epi);

/* Bytes of workspace conv2d_fwd_epi needs with this configuration (algo NULL:
 * the heuristic's) and epilogue: conv2d_fwd_workspace_bytes, plus
 * 256-byte-aligned room for an fp32 [M][K] partial-sum buffer when a fused
 * epilogue's plan cuts tiles.  Uses the current device's SM count, as the
 * heuristic does; 0 for invalid params. */
size_t conv2d_fwd_epi_workspace_bytes(const conv2d_params* params, const conv2d_algo* algo,
                                      const conv2d_epilogue* epi);

/* What the heuristic picks for conv2d_fwd_epi with this epilogue (NULL: as
 * conv2d_fwd_query_algo).  A fused epilogue's plan gives every tile to one CTA. */
int conv2d_fwd_query_algo_epi(const conv2d_params* params, const conv2d_epilogue* epi, conv2d_algo* out);

/* Weight gradient: the backward pass of the convolution with regard to the
 * weight (docs.rs burn-cubecl 0.20.0, burn_cubecl/kernel/conv/base.rs,
 * conv_weight_backward: the input feature map and the output gradient, both
 * NHWC, give a weight gradient of the weight's shape in KRSC order):
 *
 *   dw[k][r][s][c] = sum_{n,p,q} dy[n][p][q][k] * x[n][p*sh - ph + r*dh][q*sw - pw + s*dw][c]
 *
 * out-of-image positions contributing zero.  params describe the forward
 * convolution (x [N][H][W][C], weight [K][R][S][C]); x_dev: bf16 NHWC input;
 * dy_dev: bf16 [N][P][Q][K] output gradient; dw_dev: fp32 [K][R][S][C], fully
 * overwritten (zero for an empty batch).  Computed as an implicit GEMM on the
 * forward kernel's pipeline: rows are output channels, columns (tap, channel)
 * pairs, the reduction runs over the N*P*Q output pixels (split over CTAs and
 * reduced in place in dw like a split forward tile; the workspace follows the
 * rules of conv2d_fwd's).  Supported: groups == 1, C % 64 == 0 (im2col TMA
 * boxes of 64 channels) and K % 8 == 0 (16-byte rows of dy); otherwise
 * CONV2D_ERR_UNSUPPORTED.  algo may be NULL; block_n 64/128/256 is the channel
 * width of a column block, splits/grid/reduction as for conv2d_fwd_ex;
 * block_m must be 0 or 128 and loader 0 or CONV2D_LOADER_TMA_IM2COL. */
size_t conv2d_bwd_weight_workspace_bytes(const conv2d_params* params);

int conv2d_bwd_weight(const conv2d_params* params, const void* x_dev, const void* dy_dev, float* dw_dev,
                      void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream,
                      const conv2d_algo* algo);

/* What the heuristic picks for conv2d_bwd_weight (no launch; current device's SM count). */
int conv2d_bwd_weight_query_algo(const conv2d_params* params, conv2d_algo* out);

/* Data gradient: the backward pass of the convolution with regard to the input
 * (docs.rs burn-cubecl 0.20.0, burn_cubecl/kernel/conv/base.rs,
 * conv_data_backward: output gradient and weights, NHWC / KRSC, give an input
 * gradient NHWC):
 *
 *   dx[n][h][w][c] = sum_{r,s,k} dy[n][p][q][k] * w[k][r][s][c]
 *       over the taps with h + ph - r*dh = p*sh, w + pw - s*dw = q*sw, 0 <= p < P, 0 <= q < Q.
 *
 * It is also conv_transpose2d: conv_transpose2d of an input [N][Hi][Wi][Cin]
 * with weights [Cin][R][S][Cout] (stride st, padding p, dilation d, output
 * padding op < st) is this call with params {n = N, h = (Hi-1)*st - 2p +
 * d(R-1) + 1 + op, w likewise, c = Cout, k = Cin, r = R, s = S, stride st,
 * pad p, dil d} and dy = the input.
 * params describe the forward convolution (x [N][H][W][C], weight
 * [K][R][S][C]); dy_dev: bf16 [N][P][Q][K]; w_dev: bf16 [K][R][S][C]; dx_dev:
 * fp32 [N][H][W][C], fully overwritten.  Computed as forward convolutions of
 * dy with the flipped, transposed weight w'[c][r][s][k] = w[k][R-1-r][S-1-s][c],
 * which the kernel reads from w directly (no transformed copy): at stride 1
 * one launch with padding dil*(R-1) - pad; at stride (sh, sw) one launch per
 * output phase (a, b), 0 <= a < sh, 0 <= b < sw (the sub-pixel decomposition):
 * the rows h = a + sh*i receive only the taps r with a + ph - r*dh divisible
 * by sh, which are every (sh / gcd(sh, dh))-th tap, and form a stride-1
 * convolution of dy at dilation dh / gcd(sh, dh); a phase that no tap reaches
 * is zero (dx is cleared first when there is one).  Supported: groups == 1,
 * K % 64 == 0 (im2col TMA boxes of dy), C % 8 == 0, and every phase's padding
 * d'(R'-1) - c >= 0 (at stride 1: pad <= dil*(R-1)); otherwise
 * CONV2D_ERR_UNSUPPORTED.  algo as for conv2d_fwd_ex (block_m 0/128, loader 0
 * or CONV2D_LOADER_TMA_IM2COL), applied to every phase. */
size_t conv2d_bwd_data_workspace_bytes(const conv2d_params* params);

int conv2d_bwd_data(const conv2d_params* params, const void* dy_dev, const void* w_dev, float* dx_dev,
                    void* workspace_dev, size_t workspace_bytes, conv2d_stream_t stream,
                    const conv2d_algo* algo);

/* What the heuristic picks for conv2d_bwd_data (no launch; current device's SM count). */
int conv2d_bwd_data_query_algo(const conv2d_params* params, conv2d_algo* out);

/* Size of the library's built-in device scratch array used by conv2d_fwd_noalloc. */
#define CONV2D_NOALLOC_SCRATCH_BYTES 65536

/* The pages have no counterpart to this entry point.  It is conv2d_fwd for
 * callers that cannot allocate device memory, so cannot pass a workspace: for
 * example plugins whose host framework owns every device allocation, deployments
 * that forbid allocation after start-up, or latency-critical loops that must not
 * call cudaMalloc/cudaFree because those can synchronise the device.  It takes
 * the same inputs and outputs as conv2d_fwd (caller-owned device memory) and
 * allocates nothing; the workspace is a static device array of
 * CONV2D_NOALLOC_SCRATCH_BYTES bytes inside the library, which every GPU that
 * loads the library keeps until the process exits.
 *   - Problems whose conv2d_fwd_workspace_bytes() exceeds that size are rejected
 *     with CONV2D_ERR_SCRATCH_LIMIT before anything is enqueued (65536 bytes
 *     cover 16320 output tiles of 128 pixels x 64 channels).
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress, with the device current); make that first
 *     call before any stream capture.  The address is kept for the life of the
 *     process: after cudaDeviceReset (or anything else that destroys the
 *     device's primary context) it no longer names the array, so do not call
 *     this entry point again on that device in the same process.
 *   - Every call clears the part of the array it uses (cudaMemsetAsync on
 *     `stream`) and then enqueues the kernel.  All calls on one device share
 *     that device's copy of the array, and it keeps the previous call's
 *     contents, so calls that can overlap on the GPU (for example on two
 *     streams) race with each other: serialise them.
 *   - Device-side timeouts are not reported here (the status word is cleared by
 *     the next call); use conv2d_fwd + conv2d_fwd_status where that matters. */
int conv2d_fwd_noalloc(const conv2d_params* params, const void* x_dev, const void* w_dev,
                       const float* bias_dev, float* y_dev, conv2d_stream_t stream);

/* A static, human-readable message for a conv2d_status value. */
const char* conv2d_strerror(int status);

#ifdef __cplusplus
}
#endif

#endif /* SPLIT_GEMM_GB300_CONV2D_H */
