/*
 * lmoe -- forward pass of a LatentMoE layer (route to the top 16 of 896
 * experts, SwiGLU experts on MXFP4 weights, weighted combine) as a C ABI over
 * hand-written CUDA kernels for sm_103a (GB300).
 *
 * Sources (page title, section) that define the operations:
 *  [MoE]  "SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section "MoE 稀疏激活：
 *         896 专家中选 16 的 104B 激活逻辑": the router scores every token
 *         against all 896 experts (token embeddings x router weights), keeps
 *         the 16 best, and only those experts compute; their outputs are
 *         summed with weights.
 *  [MX]   same page, section "MXFP4 原生支持": 4-bit values sharing one scale
 *         per block of 32 (or 64) elements; dequantisation fused into the GEMM.
 *  [L1]   "从Kimi K3到MiniMax-H3：国产大模型竞争进入“推理系统战”", section 二,
 *         first layer: 4-bit weights meet higher-precision activations and
 *         accumulation; section 一: 896 experts, 16 active, routing and
 *         expert compute in a 3584-wide latent space (LatentMoE), gated FFN.
 *  [EP]   "Kimi K3 Day-0 适配剖析", section 四: dispatch tokens to experts
 *         (index computation, buffer planning, bucketing), expert compute,
 *         combine the results back by weight; section 三: weights converted
 *         to the hardware's form at load time, layer by layer.
 *
 * Readings where the pages are silent (the same in the CPU oracle):
 *  - block size 32, E8M0 scales, shared exponent floor(log2 amax) - emax
 *    (emax 2 for e2m1, 8 for e4m3), elements rounded to nearest even and
 *    saturated (6 for e2m1, 448 for e4m3);
 *  - gate weights: softmax over the 16 selected logits;
 *  - top-16 order: larger logit first, equal logits by smaller expert id;
 *  - the gated activation is SiLU (SwiGLU);
 *  - activations entering each expert GEMM (the latent x and the gated
 *    product h) are MXFP8 (e4m3 + E8M0 per 32), accumulation is fp32.
 *
 * Conventions for every call:
 *  - Array pointers are DEVICE pointers owned by the caller, 16-byte aligned
 *    (MXFP4 weight codes: 32-byte aligned).  Structs (lmoe_dims,
 *    lmoe_expert_weights) are host pointers read during the call.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls only
 *    enqueue work; LMOE_OK means "enqueued".
 *  - Argument errors are reported synchronously before anything is enqueued
 *    and leave every output untouched.  Launch failures return LMOE_ERR_CUDA.
 *  - Errors found by kernels (an expert id out of range, a bounded wait that
 *    ran out) are recorded in a status word at the start of the workspace;
 *    read it with lmoe_last_device_status.
 *  - No call allocates device memory; scratch comes from the caller's
 *    workspace (size from the matching *_workspace_size query).
 *  - Bit layouts:
 *      bf16 tensors are passed as uint16_t bit patterns;
 *      MXFP4 canonical: codes[r][K/2] (element 2i in the low nibble of byte
 *        i), scales[r][K/32] (E8M0);
 *      MXFP4 tensor-core layout (LMOE_LAYOUT_TC, the form lmoe_expert_ffn
 *        reads): each matrix of `rows` x K is stored with K padded to
 *        Kp = roundup(K, 128) (padding codes 0); scales are grouped in
 *        512-byte atoms, one per 128 rows x 128 columns: atom (rt, kc) of
 *        matrix m starts at ((m * RT + rt) * KC + kc) * 512 with
 *        RT = ceil(rows/128), KC = Kp/128, and holds the scale of row
 *        rt*128 + 32*j + i, column block kc*4 + b at byte 16*i + 4*j + b
 *        (rows and blocks beyond the matrix hold 0);
 *      MXFP8: codes[r][K] (e4m3), scales[r][K/32] (E8M0).
 */
#ifndef LMOE_H
#define LMOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    LMOE_OK = 0,
    LMOE_ERR_INVALID_ARG = -1,  /* bad size, null or misaligned pointer       */
    LMOE_ERR_UNSUPPORTED = -2,  /* valid request this build does not handle   */
    LMOE_ERR_WORKSPACE = -3,    /* workspace missing or too small             */
    LMOE_ERR_CUDA = -4,         /* a CUDA runtime/driver call or launch failed */
    LMOE_ERR_DEVICE_CHECK = -5, /* a kernel found bad input (status word)     */
    LMOE_ERR_TIMEOUT = -6       /* a kernel's bounded wait ran out            */
} lmoe_status;

/* Activation format of the expert GEMMs' inputs (x and h).  MXFP8: e4m3 +
 * E8M0 per 32.  MXFP4 (the full-FP4 variant: e2m1 + E8M0 per 32, the
 * weights' rule): taken by lmoe_forward on the small-batch path only
 * (lmoe_set_small_batch_pairs); elsewhere it returns LMOE_ERR_UNSUPPORTED,
 * as the tensor-core kernels for FP4 activations are not built.  Its
 * numerics are a different layer: about 20% relative RMS away from the
 * MXFP8 layer on decode-shaped tokens. */
typedef enum { LMOE_ACT_MXFP8 = 1, LMOE_ACT_MXFP4 = 2 } lmoe_act_fmt;
typedef enum { LMOE_LAYOUT_CANONICAL = 0, LMOE_LAYOUT_TC = 1 } lmoe_layout;

/* Layer shape: T tokens, latent width d, E experts, top-k, expert
 * intermediate width I, activation format.
 * Limits: T >= 0, d % 128 == 0, I % 32 == 0, 1 <= k <= min(E, 32),
 * 1 <= E <= 2048, act == LMOE_ACT_MXFP8. */
typedef struct {
    int32_t T, d, E, k, I;
    int32_t act;
} lmoe_dims;

/* The expert bank: for every expert e, gate and up [I][d] and down [d][I]
 * MXFP4 matrices, stacked over e (matrix index m = e).  `layout` says which
 * byte layout the six arrays use (see above). */
typedef struct {
    const uint8_t *gate_q, *gate_s;
    const uint8_t *up_q, *up_s;
    const uint8_t *down_q, *down_s;
    int32_t layout;
} lmoe_expert_weights;

/* ---- load-time conversion ([MX], [EP] section 三) ------------------------ */

/* Bytes of the codes (return value) and scales (*scale_bytes) of `nmat`
 * stacked MXFP4 matrices of rows x K in the given layout; 0 on bad sizes. */
size_t lmoe_mxfp4_bytes(int64_t nmat, int32_t rows, int32_t K, int32_t layout, size_t *scale_bytes);

/* Quantise nmat stacked fp32 matrices w[nmat][rows][K] to MXFP4 codes q and
 * scales s in `layout`.  K % 32 == 0.  Each block of 32 along K: scale byte
 * clamp(floor(log2 amax) - 2 + 127, 0, 254) (0 for an all-zero block),
 * element code = e2m1 round-to-nearest-even of w / 2^(byte-127), saturated
 * at 6, sign kept. */
lmoe_status lmoe_quant_mxfp4(const float *w, int64_t nmat, int32_t rows, int32_t K, uint8_t *q, uint8_t *s,
                             int32_t layout, void *stream);

/* Load-time conversion of an MXFP4 checkpoint ([EP] section 三: the checkpoint
 * is converted to the hardware's form layer by layer as it loads): nmat
 * stacked matrices of rows x K (K % 32 == 0) in LMOE_LAYOUT_CANONICAL (codes
 * q[nmat][rows][K/2], 16-byte aligned; scales s[nmat][rows][K/32]) rewritten
 * in LMOE_LAYOUT_TC into q_tc / s_tc (sizes from lmoe_mxfp4_bytes; q_tc
 * 32-byte, s_tc 16-byte aligned).  A byte rearrangement, not a
 * re-quantisation: every code and scale byte keeps its value, padding codes
 * and padding scale bytes are written as 0.  The canonical arrays can be a
 * staging buffer that the caller refills group by group of matrices (e.g.
 * one layer or one chunk of experts at a time), so the checkpoint never
 * takes more device memory in canonical form than one group.  Source and
 * destination must not overlap. */
lmoe_status lmoe_repack_mxfp4(const uint8_t *q, const uint8_t *s, int64_t nmat, int32_t rows, int32_t K, uint8_t *q_tc,
                              uint8_t *s_tc, void *stream);

/* Distribution of the E8M0 block scales ([MX] section "精度与速度的平衡":
 * the per-expert-block scale factors are logged to watch the quantisation):
 * hist[m][v] (uint32, [nmat][256], overwritten) = how many of matrix m's
 * rows x K/32 blocks have scale byte v (the block's values were divided by
 * 2^(v - 127)), read from scales s in the given layout (padding of the
 * tensor-core layout is not counted). */
lmoe_status lmoe_mxfp4_scale_histogram(const uint8_t *s, int64_t nmat, int32_t rows, int32_t K, int32_t layout,
                                       uint32_t *hist, void *stream);

/* ---- stages -------------------------------------------------------------- */

/* MXFP8 quantisation of bf16 rows x[rows][K] (K % 32 == 0): per block of
 * 32, scale byte clamp(floor(log2 amax) - 8 + 127, 0, 254), codes = e4m3
 * round-to-nearest-even of x / 2^(byte-127), saturated at 448. */
lmoe_status lmoe_quant_mxfp8(const uint16_t *x_bf16, int64_t rows, int32_t K, uint8_t *q, uint8_t *s, void *stream);

/* Router weights in the form the router GEMM reads (load-time conversion, as
 * for the expert weights): the fp32 weights Wr [E][d] written as three bf16
 * planes Wr3 [3][E][d] (hi = bf16(Wr), mid = bf16(Wr - hi), lo = bf16(Wr -
 * hi - mid), each rounded to nearest even) whose sum is Wr exactly (24
 * significand bits).  d % 64 == 0.  Wr3 must hold
 * lmoe_router_prepared_bytes(E, d) bytes (0 for invalid sizes). */
size_t lmoe_router_prepared_bytes(int32_t E, int32_t d);
lmoe_status lmoe_prepare_router(const float *Wr, int32_t E, int32_t d, uint16_t *Wr3, void *stream);

/* Router [MoE]: logits[t][e] = fp32(sum_c x[t][c] * Wr[e][c]) (+ bias[e]),
 * accumulated in fp32 on the tensor cores: each bf16 x times each bf16 plane
 * of Wr is exact in fp32 and the three planes accumulate into one sum.
 * x bf16 [T][d], Wr3 the prepared router weights (lmoe_prepare_router), bias
 * fp32 [E] or NULL (the skewed workload's popularity bias); then the top-k of
 * each row (larger logit first, ties by smaller id) into topk_idx[T][k] and
 * the softmax over those k logits into topk_w[T][k].  logits [T][E] is a
 * required output. */
lmoe_status lmoe_route(const uint16_t *x_bf16, const uint16_t *Wr3, const float *bias, const lmoe_dims *dims,
                       float *logits, int32_t *topk_idx, float *topk_w, void *workspace, size_t ws_bytes,
                       void *stream);

/* Scratch bytes lmoe_route needs for these dims (split-K partial sums). */
size_t lmoe_route_workspace_size(const lmoe_dims *dims);

/* The top-k + softmax half of lmoe_route on given fp32 logits [T][E]. */
lmoe_status lmoe_topk_from_logits(const float *logits, const lmoe_dims *dims, int32_t *topk_idx, float *topk_w,
                                  void *stream);

/* Scratch bytes lmoe_permute needs for these dims. */
size_t lmoe_permute_workspace_size(const lmoe_dims *dims);

/* Dispatch metadata [EP]: stable counting sort of the pairs p = t*k + j by
 * expert topk_idx[p]: counts[E], offsets[E+1] (exclusive prefix sum),
 * perm[T*k] (pairs of expert 0, then expert 1, ..., each in ascending p),
 * inv[p] = position of p in perm.  An id outside [0, E) is skipped and
 * recorded as LMOE_ERR_DEVICE_CHECK in the workspace status word. */
lmoe_status lmoe_permute(const int32_t *topk_idx, const lmoe_dims *dims, int32_t *counts, int32_t *offsets,
                         int32_t *perm, int32_t *inv, void *workspace, size_t ws_bytes, void *stream);

/* lmoe_permute for callers that can neither pass a workspace nor let the
 * library allocate (no counterpart on the pages: this is a deployment aid).
 * Such callers include plugin code running inside another runtime's memory
 * pool and serving loops whose device memory is fixed at start-up.  The
 * block histograms live in a fixed device array inside the library, sized
 * for at most LMOE_PERMUTE_NOALLOC_MAX_PAIRS = T*k pairs and 2048 experts
 * (about 1 MB, held on every device that loads the library until the process
 * exits).  Larger inputs are rejected with LMOE_ERR_INVALID_ARG before any
 * work is enqueued.  Outputs and their meaning are those of lmoe_permute.
 * `device_status` (nullable, a device int32) receives the device-side check
 * result (LMOE_OK or LMOE_ERR_DEVICE_CHECK).  The first call on a device
 * looks up the array's device address (the first call after a device reset
 * looks it up again, in the new context); make it before any stream capture.
 * All calls share the array, so calls that overlap on the GPU race: the
 * caller serialises them.  Nothing is allocated. */
#define LMOE_PERMUTE_NOALLOC_MAX_PAIRS 524288
lmoe_status lmoe_permute_noalloc(const int32_t *topk_idx, const lmoe_dims *dims, int32_t *counts, int32_t *offsets,
                                 int32_t *perm, int32_t *inv, int32_t *device_status, void *stream);

/* Scratch bytes lmoe_expert_ffn needs for these dims. */
size_t lmoe_expert_ffn_workspace_size(const lmoe_dims *dims);

/* Expert compute [MoE], [MX], [L1]: for every position q of perm (pair
 * p = perm[q], token t = p / k, expert e, gate weight w = topk_w[p]):
 *   g = Wg[e] x^_t, u = Wu[e] x^_t (fp32 accumulation),
 *   h^ = MXFP8(silu(g) * u) along I,
 *   yp[q][:] = w * (Wd[e] h^),
 * x^_t the MXFP8 activation (xq[T][d] codes, xs[T][d/32] scales, as made by
 * lmoe_quant_mxfp8), weights in LMOE_LAYOUT_TC, offsets/perm from
 * lmoe_permute, yp fp32 [T*k][d] in permuted order. */
lmoe_status lmoe_expert_ffn(const uint8_t *xq, const uint8_t *xs, const lmoe_expert_weights *W,
                            const int32_t *offsets, const int32_t *perm, const float *topk_w, const lmoe_dims *dims,
                            float *yp, void *workspace, size_t ws_bytes, void *stream);

/* Combine [EP]: y[t][c] = bf16( sum_{j=0..k-1} yp[inv[t*k+j]][c] ), summed
 * in fp32 in slot order, rounded to nearest even. */
lmoe_status lmoe_combine(const float *yp, const int32_t *inv, const lmoe_dims *dims, uint16_t *y_bf16, void *stream);

/* ---- whole layer ----------------------------------------------------------- */

/* Scratch bytes lmoe_forward needs for these dims (and the current
 * small-batch setting below). */
size_t lmoe_workspace_size(const lmoe_dims *dims);

/* Small batches ([L1] section 二, second layer: batch-1 decode): a batch of
 * at most `max_pairs` pairs T*k (and at most 8 tokens, 256 pairs) runs
 * lmoe_forward as three weight-streaming kernels (routing with top-k and the
 * pair lists; gate/up with SwiGLU and MXFP8 of h, on warp-level tensor-core
 * products; down with the gate weights and the combine) instead of the
 * tensor-core path.  Same contract and roundings; the k terms of a token are
 * summed in a fixed order (deterministic), but not strictly slot by slot.  It
 * is also the path of the MXFP4-activation variant (LMOE_ACT_MXFP4).  The
 * default is 0: every batch takes the tensor-core path, which with its fused
 * expert kernel measures faster at batch 1 too (45.6 against 58.9 us per
 * step, L2 flushed).  Process-wide setting, not thread-safe; the workspace
 * size of a batch depends on it.  lmoe_small_batch_pairs() reads it. */
#define LMOE_SMALL_BATCH_PAIRS_DEFAULT 0
lmoe_status lmoe_set_small_batch_pairs(int32_t max_pairs);
int32_t lmoe_small_batch_pairs(void);

/* route -> permute -> MXFP8 activations -> expert FFN -> combine, all on
 * `stream` (up to 64 tokens the routing kernel does the permute as well).
 * Wr3: prepared router weights (lmoe_prepare_router).  y bf16 [T][d].
 * Optional outputs (NULL to skip): topk_idx [T][k], topk_w [T][k],
 * logits [T][E]. */
lmoe_status lmoe_forward(const uint16_t *x_bf16, const uint16_t *Wr3, const float *bias, const lmoe_expert_weights *W,
                         const lmoe_dims *dims, uint16_t *y_bf16, int32_t *topk_idx, float *topk_w, float *logits,
                         void *workspace, size_t ws_bytes, void *stream);

/* ---- full block around the layer ([L1] section 一: LatentMoE compresses the
 * hidden state to the latent space, routes and computes experts there) ---- */

/* out[r][n] = bf16( sum_c x[r][c] * W[n][c] ), x bf16 [rows][K], W bf16 [N][K],
 * fp32 accumulation on the tensor cores, round to nearest even.
 * K % 64 == 0, N % 16 == 0. */
lmoe_status lmoe_linear_bf16(const uint16_t *x, const uint16_t *W, int64_t rows, int32_t K, int32_t N, uint16_t *out,
                             void *stream);

/* Scratch bytes lmoe_forward_block needs for these dims and hidden width. */
size_t lmoe_block_workspace_size(const lmoe_dims *dims, int32_t hidden);

/* lat = bf16(x_h W_in^T) [T][d]; y = lmoe_forward(lat) [T][d];
 * out = bf16(y W_out^T) [T][hidden].  x_h bf16 [T][hidden], W_in bf16
 * [d][hidden], W_out bf16 [hidden][d]; hidden % 64 == 0.  Optional outputs
 * (NULL to skip): lat and y (bf16 [T][d]), topk_idx, topk_w, logits. */
lmoe_status lmoe_forward_block(const uint16_t *x_h, const uint16_t *W_in, const uint16_t *Wr3, const float *bias,
                               const lmoe_expert_weights *W, const uint16_t *W_out, const lmoe_dims *dims,
                               int32_t hidden, uint16_t *out, uint16_t *lat, uint16_t *y, int32_t *topk_idx,
                               float *topk_w, float *logits, void *workspace, size_t ws_bytes, void *stream);

/* ---- helpers --------------------------------------------------------------- */

/* Reads (synchronously, after all prior work on the device) the status word
 * kernels left in `workspace`: LMOE_OK, LMOE_ERR_DEVICE_CHECK or
 * LMOE_ERR_TIMEOUT into *device_status; returns LMOE_ERR_CUDA if the read
 * itself fails. */
lmoe_status lmoe_last_device_status(const void *workspace, int32_t *device_status);

/* Clears the status word (enqueued on `stream`). */
lmoe_status lmoe_clear_device_status(void *workspace, void *stream);

/* Number of CUDA kernels one lmoe_forward call with these dims launches
 * (0 for invalid dims or T == 0). */
int32_t lmoe_forward_kernel_count(const lmoe_dims *dims);

/* Profiling hook: when set, lmoe_forward records the n = LMOE_NUM_STAGE_EVENTS
 * CUDA events (cudaEvent_t handles, created by the caller) on its stream at
 * the stage boundaries: [0] start, [1] after routing, [2] after permute,
 * [3] after the MXFP8 activation scatter, [4] after the gate/up GEMM,
 * [5] after the down GEMM, [6] after combine.  Where the two expert GEMMs run
 * as one kernel (token tiles of up to 32 rows), [4] and [5] both follow that
 * kernel.  n = 0 clears the hook.  The setting is process-wide and not
 * thread-safe; it only adds event records. */
#define LMOE_NUM_STAGE_EVENTS 7
lmoe_status lmoe_set_stage_events(void *const *events, int32_t n);

/* ---- diagnostics (used by the parity tests; not needed to run the layer) ---- */

/* Where lmoe_forward keeps the expert GEMMs' MXFP8 operands inside its
 * workspace, as byte offsets from the workspace start, for these dims:
 *   xq  [rows][d]  e4m3 codes of x, one row per routed pair at its position
 *       in expert-sorted (permuted) order, code_row[p]; expert e's pairs
 *       form token tiles of tile_tokens rows from its first pair on,
 *   xs  scale atoms of x, one 512-byte atom per token tile and 128 columns:
 *       a pair's atom row R = dst_row[p] (its tile n = R / tile_tokens, row
 *       rr = R % tile_tokens in the tile, i = rr % 32, j = rr / 32), block b
 *       at byte ((n*(d/128) + b/4)*512 + 16*i + 4*j + b%4),
 *   hq  [rows][I]  e4m3 codes of the gated product h of each pair (row
 *       code_row[p]),
 *   hs  scale atoms of h (the same layout with roundup(I,128)/128 atoms per
 *       tile),
 *   dst_row   int32 [T*k]: the atom row of pair p = t*k + j,
 *   code_row  int32 [T*k]: the code row of pair p (the permute's inverse map);
 *   ksplit    int32 [128][4] or -1: at 16-token tiles, when the batch can
 *       have at most half as many gate/up work items as the GPU has SMs
 *       (items <= (T*k + m*15)/16 token tiles x roundup(I,128)/128 weight
 *       tiles, m = min(T*k, E); at most 128 items; d >= 256), each item runs
 *       as two K halves on two SMs and the later half forms h from the sum
 *       of both; entry [i][q] counts the halves of item i (items in
 *       token-tile order, weight tile fastest) that its epilogue warp q
 *       (rows 32q .. 32q+31 of the item's 128) stored: 2 for a split item
 *       whose warp holds rows of I, 0 otherwise (-1: no such layout);
 * rows = code rows reserved (T*k plus one tile), tile_tokens = tokens per
 * expert-GEMM tile, slot_rows = atom rows a tile occupies (tile_tokens).
 * Valid after an lmoe_forward call with the same dims has completed; rows no
 * pair maps to hold no defined data. */
typedef struct {
    int64_t xq, xs, hq, hs, dst_row;
    int64_t rows;
    int32_t tile_tokens, slot_rows;
    int32_t path; /* 0: as above; 1: small-batch path (lmoe_set_small_batch_pairs): xq/xs hold one row per
                     token t, hq/hs one row per pair p = t*k + j, dst_row = code_row = -1, rows = T*k; with
                     LMOE_ACT_MXFP4 a code row holds packed e2m1 codes (d/2 or I/2 bytes, element 2i in
                     the low nibble of byte i) */
    int64_t code_row;
    int64_t ksplit;
} lmoe_ffn_views;
lmoe_status lmoe_forward_workspace_views(const lmoe_dims *dims, lmoe_ffn_views *views);

/* When h_f32 is set (device buffer of `bytes` bytes, 16-byte aligned), every
 * later lmoe_forward / lmoe_expert_ffn call also writes the fp32 value of
 * each h its gate/up GEMM rounds to MXFP8 at h_f32[R][i] (R the pair's
 * code row as in lmoe_ffn_views, I floats per row), so a test can check
 * the rounding bit for bit.  Calls return LMOE_ERR_INVALID_ARG while the
 * buffer is smaller than rows * I * 4 bytes.  NULL clears the hook.  The
 * setting is process-wide and not thread-safe. */
lmoe_status lmoe_set_h_capture(float *h_f32, size_t bytes);

/* Failure-path test of the expert GEMMs' bounded waits.  Every wait on an
 * mbarrier in the expert GEMMs gives up after a limit of SM clocks (about
 * 2 s by default), records LMOE_ERR_TIMEOUT in the status word, and the
 * kernel winds down (an MMA issuer first waits, again bounded, for its MMAs
 * in flight) and returns; so does the wait of a down item, in the kernel
 * that runs both GEMMs, for its token tile's h.  With stall_first_fill set, the first pipeline
 * stage of every CTA of the following lmoe_forward / lmoe_expert_ffn calls
 * is never filled, so those waits run out after wait_limit_cycles; the host
 * then reads LMOE_ERR_TIMEOUT with lmoe_last_device_status.  (0, 0) restores
 * the normal behaviour; wait_limit_cycles alone (stall 0) only changes the
 * limit.  After LMOE_ERR_TIMEOUT the outputs of that call are undefined and
 * copies it had started may still land in its workspace; the caller should
 * synchronise and treat the call as failed.  Process-wide, not thread-safe. */
lmoe_status lmoe_set_wait_test(int32_t stall_first_fill, int64_t wait_limit_cycles);

const char *lmoe_status_string(lmoe_status s);

/* Library build tag (arch and version), e.g. "lmoe 0.1 sm_103a". */
const char *lmoe_version(void);

#ifdef __cplusplus
}
#endif
#endif /* LMOE_H */
