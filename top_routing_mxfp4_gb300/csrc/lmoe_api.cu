// C ABI of the lmoe library: argument checks, workspace carving, launches.
// Every entry point validates before it enqueues anything, so an argument
// error leaves all outputs untouched.
#include <stdio.h>

#include "lmoe_internal.cuh"

using namespace lmoe;

namespace {

constexpr int32_t kStatusBytes = 256;

cudaEvent_t g_stage_events[LMOE_NUM_STAGE_EVENTS] = {};
bool g_stage_events_on = false;
// diagnostics hook (lmoe_set_h_capture): fp32 h of the gate/up epilogue
float *g_hcap = nullptr;
size_t g_hcap_bytes = 0;
// failure-path test hook (lmoe_set_wait_test)
int32_t g_stall = 0;
int64_t g_wait_limit = 0;
// batches of at most this many pairs (T * k) take the small-batch path
int32_t g_small_pairs = LMOE_SMALL_BATCH_PAIRS_DEFAULT;

// Batches of at most 64 tokens on the tensor-core path: the routing kernel
// also does the permute (PermByMask: token masks per expert, the status
// region's third int32 its CTA counter), so no permute kernel runs.
bool permute_in_route(int T, int d, int E, int k, const FfnLayout &FL)
{
    return route_can_permute(T, d, E, k) && ffn_fused(FL) && FL.SLOT == FL.NT;
}

bool small_path(const lmoe_dims *d)
{
    return d->T > 0 && small_path_fits(d->T, d->d, d->E, d->k, d->I, g_small_pairs);
}

cudaError_t mark(int i, cudaStream_t st)
{
    return g_stage_events_on ? cudaEventRecord(g_stage_events[i], st) : cudaSuccess;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool dims_ok(const lmoe_dims *d)
{
    if (!d) return false;
    if (d->T < 0 || d->d <= 0 || d->E <= 0 || d->k <= 0 || d->I <= 0) return false;
    if (d->d % 128 != 0 || d->I % 32 != 0) return false;
    if (d->k > 32 || d->k > d->E || d->E > 2048) return false;
    if (int64_t(d->T) * d->k > INT32_MAX / 2) return false;
    return true;
}

lmoe_status act_ok(const lmoe_dims *d) { return d->act == LMOE_ACT_MXFP8 ? LMOE_OK : LMOE_ERR_UNSUPPORTED; }

lmoe_status cuda_status(cudaError_t e)
{
    if (e == cudaSuccess) return LMOE_OK;
    fprintf(stderr, "lmoe: CUDA error %s\n", cudaGetErrorString(e));
    return LMOE_ERR_CUDA;
}

bool weights_ok(const lmoe_expert_weights *W)
{
    if (!W || W->layout != LMOE_LAYOUT_TC) return false;
    const uint8_t *codes[3] = {W->gate_q, W->up_q, W->down_q};
    const uint8_t *scales[3] = {W->gate_s, W->up_s, W->down_s};
    for (int i = 0; i < 3; ++i)
        if (!codes[i] || !scales[i] || !aligned(codes[i], 32) || !aligned(scales[i], 16)) return false;
    return true;
}

// Workspace layout of lmoe_forward (each region 256-byte aligned):
//   status | token masks | logits | idx | w | counts | offsets | perm | inv | permute scratch
//   | ffn scratch (MXFP8 activations and h in permuted order, their scale atoms per token tile, schedule)
//   | yp (per-pair outputs [T*k][d]) or, with the fused combine, yacc ([T][d] fp32 sums)
// The small-batch path (lmoe_set_small_batch_pairs) uses
//   status (+ the routing kernel's counter) | logits | idx | w | small-path scratch.
struct FwdLayout {
    size_t status, tmask, logits, idx, w, counts, offsets, perm, inv, rscratch, pscratch, fscratch, yp, total;
    bool small;
    size_t sscratch;
};

FwdLayout fwd_layout(const lmoe_dims *d)
{
    const int64_t T = d->T, P = T * d->k, E = d->E;
    FwdLayout L{};
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += size_t(round_up(int64_t(bytes), 256));
        return o;
    };
    L.status = take(kStatusBytes);
    L.tmask = take(size_t(E * 8));  // small batches: the routing kernel's token masks (see permute_in_route)
    L.logits = take(size_t(T * E * 4));
    L.idx = take(size_t(P * 4));
    L.w = take(size_t(P * 4));
    L.small = small_path(d);
    if (L.small) {
        L.sscratch = take(small_layout(d->T, d->d, d->E, d->k, d->I).total);
        L.total = off;
        return L;
    }
    L.counts = take(size_t(E * 4));
    L.offsets = take(size_t((E + 1) * 4));
    L.perm = take(size_t(P * 4));
    L.inv = take(size_t(P * 4));
    L.rscratch = take(router_scratch_bytes(int(T), d->d, int(E)));
    L.pscratch = take(permute_scratch_bytes(P, int(E)));
    L.fscratch = take(ffn_layout(P, d->d, int(E), d->I).total);
    L.yp = take(size_t((ffn_layout(P, d->d, int(E), d->I).fused ? T : P) * d->d * 4));
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

const char *lmoe_version(void) { return "lmoe 0.1 sm_103a"; }

const char *lmoe_status_string(lmoe_status s)
{
    switch (s) {
    case LMOE_OK: return "ok";
    case LMOE_ERR_INVALID_ARG: return "invalid argument";
    case LMOE_ERR_UNSUPPORTED: return "unsupported";
    case LMOE_ERR_WORKSPACE: return "workspace missing or too small";
    case LMOE_ERR_CUDA: return "CUDA error";
    case LMOE_ERR_DEVICE_CHECK: return "device-side input check failed";
    case LMOE_ERR_TIMEOUT: return "device-side bounded wait timed out";
    }
    return "unknown status";
}

size_t lmoe_mxfp4_bytes(int64_t nmat, int32_t rows, int32_t K, int32_t layout, size_t *scale_bytes)
{
    if (nmat < 0 || rows <= 0 || K <= 0 || K % 32 != 0) return 0;
    if (layout == LMOE_LAYOUT_CANONICAL) {
        if (scale_bytes) *scale_bytes = size_t(nmat) * rows * (K / 32);
        return size_t(nmat) * rows * (K / 2);
    }
    if (layout == LMOE_LAYOUT_TC) {
        const int64_t Kp = round_up(K, 128);
        if (scale_bytes) *scale_bytes = size_t(nmat) * ceil_div(rows, 128) * (Kp / 128) * 512;
        return size_t(nmat) * rows * (Kp / 2);
    }
    return 0;
}

lmoe_status lmoe_quant_mxfp4(const float *w, int64_t nmat, int32_t rows, int32_t K, uint8_t *q, uint8_t *s,
                             int32_t layout, void *stream)
{
    if (nmat < 0 || rows <= 0 || K <= 0 || K % 32 != 0) return LMOE_ERR_INVALID_ARG;
    if (layout != LMOE_LAYOUT_CANONICAL && layout != LMOE_LAYOUT_TC) return LMOE_ERR_INVALID_ARG;
    if (nmat == 0) return LMOE_OK;
    if (!w || !q || !s || !aligned(w, 16) || !aligned(q, 32) || !aligned(s, 16)) return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_quant_mxfp4(w, nmat, rows, K, q, s, layout, cudaStream_t(stream)));
}

lmoe_status lmoe_repack_mxfp4(const uint8_t *q, const uint8_t *s, int64_t nmat, int32_t rows, int32_t K, uint8_t *q_tc,
                              uint8_t *s_tc, void *stream)
{
    if (nmat < 0 || rows <= 0 || K <= 0 || K % 32 != 0) return LMOE_ERR_INVALID_ARG;
    if (nmat == 0) return LMOE_OK;
    if (!q || !s || !q_tc || !s_tc || !aligned(q, 16) || !aligned(q_tc, 32) || !aligned(s_tc, 16))
        return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_repack_mxfp4(q, s, nmat, rows, K, q_tc, s_tc, cudaStream_t(stream)));
}

lmoe_status lmoe_mxfp4_scale_histogram(const uint8_t *s, int64_t nmat, int32_t rows, int32_t K, int32_t layout,
                                       uint32_t *hist, void *stream)
{
    if (nmat < 0 || nmat > INT32_MAX || rows <= 0 || K <= 0 || K % 32 != 0) return LMOE_ERR_INVALID_ARG;
    if (layout != LMOE_LAYOUT_CANONICAL && layout != LMOE_LAYOUT_TC) return LMOE_ERR_INVALID_ARG;
    if (nmat == 0) return LMOE_OK;
    if (!s || !hist || !aligned(hist, 4)) return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_scale_histogram(s, nmat, rows, K, layout, hist, cudaStream_t(stream)));
}

lmoe_status lmoe_quant_mxfp8(const uint16_t *x_bf16, int64_t rows, int32_t K, uint8_t *q, uint8_t *s, void *stream)
{
    if (rows < 0 || K <= 0 || K % 32 != 0) return LMOE_ERR_INVALID_ARG;
    if (rows == 0) return LMOE_OK;
    if (!x_bf16 || !q || !s || !aligned(x_bf16, 16) || !aligned(q, 16)) return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_quant_mxfp8(x_bf16, rows, K, q, s, cudaStream_t(stream)));
}

size_t lmoe_route_workspace_size(const lmoe_dims *dims)
{
    if (!dims_ok(dims)) return 0;
    return kStatusBytes + router_scratch_bytes(dims->T, dims->d, dims->E);
}

size_t lmoe_router_prepared_bytes(int32_t E, int32_t d)
{
    if (E <= 0 || d <= 0 || d % 64 != 0) return 0;
    return size_t(3) * size_t(E) * size_t(d) * 2;
}

lmoe_status lmoe_prepare_router(const float *Wr, int32_t E, int32_t d, uint16_t *Wr3, void *stream)
{
    if (E <= 0 || d <= 0 || d % 64 != 0 || !Wr || !Wr3 || !aligned(Wr, 16) || !aligned(Wr3, 16))
        return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_split_router(Wr, E, d, Wr3, cudaStream_t(stream)));
}

lmoe_status lmoe_route(const uint16_t *x_bf16, const uint16_t *Wr3, const float *bias, const lmoe_dims *dims,
                       float *logits, int32_t *topk_idx, float *topk_w, void *workspace, size_t ws_bytes,
                       void *stream)
{
    if (!dims_ok(dims)) return LMOE_ERR_INVALID_ARG;
    if (dims->T == 0) return LMOE_OK;
    if (!x_bf16 || !Wr3 || !logits || !topk_idx || !topk_w || !aligned(x_bf16, 16) || !aligned(Wr3, 16))
        return LMOE_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < lmoe_route_workspace_size(dims) || !aligned(workspace, 256)) return LMOE_ERR_WORKSPACE;
    cudaStream_t st = cudaStream_t(stream);
    char *ws = static_cast<char *>(workspace);
    int32_t *status = reinterpret_cast<int32_t *>(ws);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (e == cudaSuccess)
        e = launch_route(x_bf16, Wr3, bias, dims->T, dims->d, dims->E, dims->k, logits, topk_idx, topk_w,
                         ws + kStatusBytes, status, st);
    return cuda_status(e);
}

lmoe_status lmoe_topk_from_logits(const float *logits, const lmoe_dims *dims, int32_t *topk_idx, float *topk_w,
                                  void *stream)
{
    if (!dims_ok(dims)) return LMOE_ERR_INVALID_ARG;
    if (dims->T == 0) return LMOE_OK;
    if (!logits || !topk_idx || !topk_w) return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_topk_softmax(logits, dims->T, dims->E, dims->k, topk_idx, topk_w, cudaStream_t(stream)));
}

size_t lmoe_permute_workspace_size(const lmoe_dims *dims)
{
    if (!dims_ok(dims)) return 0;
    return kStatusBytes + permute_scratch_bytes(int64_t(dims->T) * dims->k, dims->E);
}

lmoe_status lmoe_permute(const int32_t *topk_idx, const lmoe_dims *dims, int32_t *counts, int32_t *offsets,
                         int32_t *perm, int32_t *inv, void *workspace, size_t ws_bytes, void *stream)
{
    if (!dims_ok(dims)) return LMOE_ERR_INVALID_ARG;
    if (!counts || !offsets || (dims->T > 0 && (!topk_idx || !perm || !inv))) return LMOE_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < lmoe_permute_workspace_size(dims) || !aligned(workspace, 256))
        return LMOE_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    cudaError_t e0 = cudaMemsetAsync(ws, 0, sizeof(int32_t), cudaStream_t(stream));
    if (e0 != cudaSuccess) return cuda_status(e0);
    return cuda_status(launch_permute(topk_idx, int64_t(dims->T) * dims->k, dims->E, counts, offsets, perm, inv,
                                      ws + kStatusBytes, reinterpret_cast<int32_t *>(ws), cudaStream_t(stream)));
}

size_t lmoe_expert_ffn_workspace_size(const lmoe_dims *dims)
{
    if (!dims_ok(dims)) return 0;
    const int64_t P = int64_t(dims->T) * dims->k;
    return kStatusBytes + ffn_layout(P, dims->d, dims->E, dims->I).total;
}

lmoe_status lmoe_expert_ffn(const uint8_t *xq, const uint8_t *xs, const lmoe_expert_weights *W,
                            const int32_t *offsets, const int32_t *perm, const float *topk_w, const lmoe_dims *dims,
                            float *yp, void *workspace, size_t ws_bytes, void *stream)
{
    if (!dims_ok(dims)) return LMOE_ERR_INVALID_ARG;
    lmoe_status a = act_ok(dims);
    if (a != LMOE_OK) return a;
    if (dims->T == 0) return LMOE_OK;
    if (!xq || !xs || !offsets || !perm || !topk_w || !yp || !aligned(xq, 16) || !aligned(xs, 16) ||
        !aligned(yp, 16))
        return LMOE_ERR_INVALID_ARG;
    if (!weights_ok(W)) return LMOE_ERR_INVALID_ARG;
    if (!workspace || ws_bytes < lmoe_expert_ffn_workspace_size(dims) || !aligned(workspace, 256))
        return LMOE_ERR_WORKSPACE;
    const int64_t P = int64_t(dims->T) * dims->k;
    char *ws = static_cast<char *>(workspace);
    char *fs = ws + kStatusBytes;
    const FfnLayout L = ffn_layout(P, dims->d, dims->E, dims->I);
    if (g_hcap && g_hcap_bytes < size_t(L.rows) * dims->I * sizeof(float)) return LMOE_ERR_INVALID_ARG;
    cudaStream_t st = cudaStream_t(stream);
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = launch_ffn_schedule(offsets, dims->E, dims->d, dims->I, L, fs, st);
    if (e == cudaSuccess) e = launch_gather_pad(xq, xs, dims->T, dims->d, dims->k, dims->E, offsets, perm, topk_w, L, fs,
                                                   st);
    if (e != cudaSuccess) return cuda_status(e);
    FfnArgs f{W, offsets, perm, topk_w, int(P), dims->d, dims->E, dims->k, dims->I, yp, nullptr, reinterpret_cast<int32_t *>(ws)};
    f.hcap = g_hcap;
    f.wait_limit = g_wait_limit;
    f.stall_first_fill = g_stall;
    return cuda_status(launch_expert_gemms(f, L, fs, st));
}

lmoe_status lmoe_combine(const float *yp, const int32_t *inv, const lmoe_dims *dims, uint16_t *y_bf16, void *stream)
{
    if (!dims_ok(dims)) return LMOE_ERR_INVALID_ARG;
    if (dims->T == 0) return LMOE_OK;
    if (!yp || !inv || !y_bf16 || !aligned(yp, 16) || !aligned(y_bf16, 16)) return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(yp, inv, dims->T, dims->d, dims->k, y_bf16, cudaStream_t(stream), false));
}

size_t lmoe_workspace_size(const lmoe_dims *dims)
{
    if (!dims_ok(dims)) return 0;
    return fwd_layout(dims).total;
}

lmoe_status lmoe_forward(const uint16_t *x_bf16, const uint16_t *Wr3, const float *bias, const lmoe_expert_weights *W,
                         const lmoe_dims *dims, uint16_t *y_bf16, int32_t *topk_idx, float *topk_w, float *logits,
                         void *workspace, size_t ws_bytes, void *stream)
{
    if (!dims_ok(dims)) return LMOE_ERR_INVALID_ARG;
    // MXFP4 activations exist on the small-batch path only
    lmoe_status a = (dims->act == LMOE_ACT_MXFP4 && small_path(dims)) ? LMOE_OK : act_ok(dims);
    if (a != LMOE_OK) return a;
    if (dims->T == 0) return LMOE_OK;
    if (!x_bf16 || !Wr3 || !y_bf16 || !aligned(x_bf16, 16) || !aligned(Wr3, 16) || !aligned(y_bf16, 16))
        return LMOE_ERR_INVALID_ARG;
    if (!weights_ok(W)) return LMOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(dims);
    if (!workspace || ws_bytes < L.total || !aligned(workspace, 256)) return LMOE_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    cudaStream_t st = cudaStream_t(stream);
    const int T = dims->T, E = dims->E, k = dims->k, d = dims->d;
    const int64_t P = int64_t(T) * k;
    float *lg = logits ? logits : reinterpret_cast<float *>(ws + L.logits);
    int32_t *idx = topk_idx ? topk_idx : reinterpret_cast<int32_t *>(ws + L.idx);
    float *w = topk_w ? topk_w : reinterpret_cast<float *>(ws + L.w);
    int32_t *counts = reinterpret_cast<int32_t *>(ws + L.counts);
    int32_t *offsets = reinterpret_cast<int32_t *>(ws + L.offsets);
    int32_t *perm = reinterpret_cast<int32_t *>(ws + L.perm);
    int32_t *inv = reinterpret_cast<int32_t *>(ws + L.inv);
    int32_t *status = reinterpret_cast<int32_t *>(ws + L.status);
    if (L.small) {
        // three kernels; the status word and the routing kernel's counter
        // (the next int32) start at zero
        if (g_hcap && g_hcap_bytes < size_t(P) * dims->I * sizeof(float)) return LMOE_ERR_INVALID_ARG;
        cudaError_t e = mark(0, st);
        if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, 2 * sizeof(int32_t), st);
        if (e == cudaSuccess)
            e = launch_small_forward(x_bf16, Wr3, bias, W, T, d, E, k, dims->I, dims->act, lg, idx, w, y_bf16,
                                     small_layout(T, d, E, k, dims->I), ws + L.sscratch, status, status + 1, g_hcap, st,
                                     g_stage_events_on ? g_stage_events : nullptr);
        if (e == cudaSuccess) e = mark(5, st);
        if (e == cudaSuccess) e = mark(6, st);
        return cuda_status(e);
    }
    char *fs = ws + L.fscratch;
    const FfnLayout FL = ffn_layout(P, d, E, dims->I);
    if (g_hcap && g_hcap_bytes < size_t(FL.rows) * dims->I * sizeof(float)) return LMOE_ERR_INVALID_ARG;
    float *yp = reinterpret_cast<float *>(ws + L.yp);
    // Large batches fuse the combine into the down GEMM: its epilogue adds
    // each pair's weighted output into the token's fp32 row (zeroed here),
    // which one pass then rounds to bf16.
    float *yacc = FL.fused ? yp : nullptr;

    const bool pr = permute_in_route(T, d, E, k, FL);
    PermByMask pm;
    if (pr) {
        pm.mask = reinterpret_cast<unsigned long long *>(ws + L.tmask);
        pm.counter = status + 2;
        pm.counts = counts;
        pm.offsets = offsets;
        pm.perm = perm;
        pm.inv = inv;
        pm.sc = ffn_sched(FL, d, dims->I, fs);
    }
    cudaError_t e = mark(0, st);
    // the status word (and, with the permute in the routing kernel, its counter and the token masks) start at zero
    if (e == cudaSuccess) e = cudaMemsetAsync(status, 0, pr ? L.tmask - L.status + size_t(E) * 8 : sizeof(int32_t), st);
    if (e == cudaSuccess) e = launch_route(x_bf16, Wr3, bias, T, d, E, k, lg, idx, w, ws + L.rscratch, status, st, pm);
    if (e == cudaSuccess) e = mark(1, st);
    if (e == cudaSuccess && !pr)
        e = launch_permute(idx, P, E, counts, offsets, perm, inv, ws + L.pscratch, status, st,
                           ffn_sched(FL, d, dims->I, fs));
    if (e == cudaSuccess) e = mark(2, st);
    if (e == cudaSuccess) e = launch_quant_scatter_pad(x_bf16, T, d, k, E, dims->I, inv, w, FL, fs, st);
    if (e == cudaSuccess) e = mark(3, st);
    if (e == cudaSuccess) {
        FfnArgs f{W, offsets, perm, w, int(P), d, E, k, dims->I, yp, yacc, status};
        f.hcap = g_hcap;
        f.wait_limit = g_wait_limit;
        f.stall_first_fill = g_stall;
        e = launch_expert_gemms(f, FL, fs, st, g_stage_events_on ? g_stage_events[4] : nullptr);
    }
    if (e == cudaSuccess) e = mark(5, st);
    if (e == cudaSuccess)
        e = yacc ? launch_acc_to_bf16(yacc, int64_t(T) * d, y_bf16, st) : launch_combine(yp, inv, T, d, k, y_bf16, st, true);
    if (e == cudaSuccess) e = mark(6, st);
    return cuda_status(e);
}

lmoe_status lmoe_linear_bf16(const uint16_t *x, const uint16_t *W, int64_t rows, int32_t K, int32_t N, uint16_t *out,
                             void *stream)
{
    if (rows < 0 || rows > INT32_MAX || K <= 0 || K % 64 != 0 || N <= 0 || N % 16 != 0) return LMOE_ERR_INVALID_ARG;
    if (rows == 0) return LMOE_OK;
    if (!x || !W || !out || !aligned(x, 16) || !aligned(W, 16) || !aligned(out, 16)) return LMOE_ERR_INVALID_ARG;
    return cuda_status(launch_linear_bf16(x, W, int(rows), K, N, out, nullptr, nullptr, cudaStream_t(stream)));
}

size_t lmoe_block_workspace_size(const lmoe_dims *dims, int32_t hidden)
{
    if (!dims_ok(dims) || hidden <= 0 || hidden % 64 != 0) return 0;
    const size_t lat = size_t(round_up(int64_t(dims->T) * dims->d * 2, 256));
    return 2 * lat + lmoe_workspace_size(dims);
}

lmoe_status lmoe_forward_block(const uint16_t *x_h, const uint16_t *W_in, const uint16_t *Wr3, const float *bias,
                               const lmoe_expert_weights *W, const uint16_t *W_out, const lmoe_dims *dims,
                               int32_t hidden, uint16_t *out, uint16_t *lat, uint16_t *y, int32_t *topk_idx,
                               float *topk_w, float *logits, void *workspace, size_t ws_bytes, void *stream)
{
    if (!dims_ok(dims) || hidden <= 0 || hidden % 64 != 0) return LMOE_ERR_INVALID_ARG;
    lmoe_status a = act_ok(dims);
    if (a != LMOE_OK) return a;
    if (dims->T == 0) return LMOE_OK;
    if (!x_h || !W_in || !W_out || !out || !aligned(x_h, 16) || !aligned(W_in, 16) || !aligned(W_out, 16) ||
        !aligned(out, 16) || (lat && !aligned(lat, 16)) || (y && !aligned(y, 16)))
        return LMOE_ERR_INVALID_ARG;
    if (!Wr3 || !aligned(Wr3, 16) || !weights_ok(W)) return LMOE_ERR_INVALID_ARG;
    const size_t need = lmoe_block_workspace_size(dims, hidden);
    if (!workspace || ws_bytes < need || !aligned(workspace, 256)) return LMOE_ERR_WORKSPACE;
    char *ws = static_cast<char *>(workspace);
    const size_t latb = size_t(round_up(int64_t(dims->T) * dims->d * 2, 256));
    uint16_t *lat_buf = lat ? lat : reinterpret_cast<uint16_t *>(ws);
    uint16_t *y_buf = y ? y : reinterpret_cast<uint16_t *>(ws + latb);
    void *fws = ws + 2 * latb;
    cudaStream_t st = cudaStream_t(stream);
    cudaError_t e = launch_linear_bf16(x_h, W_in, dims->T, hidden, dims->d, lat_buf, nullptr, nullptr, st);
    if (e != cudaSuccess) return cuda_status(e);
    lmoe_status s = lmoe_forward(lat_buf, Wr3, bias, W, dims, y_buf, topk_idx, topk_w, logits, fws,
                                 ws_bytes - 2 * latb, stream);
    if (s != LMOE_OK) return s;
    return cuda_status(launch_linear_bf16(y_buf, W_out, dims->T, dims->d, hidden, out, nullptr, nullptr, st));
}

int32_t lmoe_forward_kernel_count(const lmoe_dims *dims)
{
    if (!dims_ok(dims) || dims->T == 0) return 0;
    const int64_t P = int64_t(dims->T) * dims->k;
    if (small_path(dims)) return 3;  // route, gate/up, down
    // router (split, GEMM, (reduction), top-k), permute (with the GEMM schedule), scatter, the two
    // expert GEMMs (one fused kernel for small token tiles), combine
    const FfnLayout FL = ffn_layout(P, dims->d, dims->E, dims->I);
    const int gemms = ffn_fused(FL) ? 1 : 2;
    const int perms = permute_in_route(dims->T, dims->d, dims->E, dims->k, FL) ? 0 : permute_kernel_count(P);
    return router_kernel_count(dims->T, dims->d, dims->E) + perms + 1 + gemms + 1;
}

lmoe_status lmoe_set_stage_events(void *const *events, int32_t n)
{
    if (n == 0) {
        g_stage_events_on = false;
        return LMOE_OK;
    }
    if (n != LMOE_NUM_STAGE_EVENTS || !events) return LMOE_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i)
        if (!events[i]) return LMOE_ERR_INVALID_ARG;
    for (int i = 0; i < n; ++i) g_stage_events[i] = cudaEvent_t(events[i]);
    g_stage_events_on = true;
    return LMOE_OK;
}

lmoe_status lmoe_forward_workspace_views(const lmoe_dims *dims, lmoe_ffn_views *views)
{
    if (!dims_ok(dims) || !views) return LMOE_ERR_INVALID_ARG;
    const FwdLayout L = fwd_layout(dims);
    if (L.small) {
        const SmallLayout S = small_layout(dims->T, dims->d, dims->E, dims->k, dims->I);
        views->xq = int64_t(L.sscratch + S.xq);
        views->xs = int64_t(L.sscratch + S.xs);
        views->hq = int64_t(L.sscratch + S.hq);
        views->hs = int64_t(L.sscratch + S.hs);
        views->dst_row = -1;
        views->code_row = -1;
        views->ksplit = -1;
        views->rows = int64_t(dims->T) * dims->k;
        views->tile_tokens = 0;
        views->slot_rows = 0;
        views->path = 1;
        return LMOE_OK;
    }
    const FfnLayout F = ffn_layout(int64_t(dims->T) * dims->k, dims->d, dims->E, dims->I);
    views->path = 0;
    views->xq = int64_t(L.fscratch + F.xq);
    views->xs = int64_t(L.fscratch + F.xs);
    views->hq = int64_t(L.fscratch + F.hq);
    views->hs = int64_t(L.fscratch + F.hs);
    views->dst_row = int64_t(L.fscratch + F.dst_row);
    views->code_row = int64_t(L.inv);
    views->ksplit = F.NT == 16 ? int64_t(L.fscratch + F.kcnt) : -1;
    views->rows = F.rows;
    views->tile_tokens = F.NT;
    views->slot_rows = F.SLOT;
    return LMOE_OK;
}

lmoe_status lmoe_set_wait_test(int32_t stall_first_fill, int64_t wait_limit_cycles)
{
    if (wait_limit_cycles < 0 || (stall_first_fill && wait_limit_cycles == 0)) return LMOE_ERR_INVALID_ARG;
    g_stall = stall_first_fill ? 1 : 0;
    g_wait_limit = wait_limit_cycles;
    return LMOE_OK;
}

lmoe_status lmoe_set_small_batch_pairs(int32_t max_pairs)
{
    if (max_pairs < 0) return LMOE_ERR_INVALID_ARG;
    g_small_pairs = max_pairs;
    return LMOE_OK;
}

int32_t lmoe_small_batch_pairs(void) { return g_small_pairs; }

lmoe_status lmoe_set_h_capture(float *h_f32, size_t bytes)
{
    if (h_f32 && (bytes == 0 || !aligned(h_f32, 16))) return LMOE_ERR_INVALID_ARG;
    g_hcap = h_f32;
    g_hcap_bytes = h_f32 ? bytes : 0;
    return LMOE_OK;
}

lmoe_status lmoe_last_device_status(const void *workspace, int32_t *device_status)
{
    if (!workspace || !device_status) return LMOE_ERR_INVALID_ARG;
    int32_t v = 0;
    cudaError_t e = cudaDeviceSynchronize();
    if (e == cudaSuccess) e = cudaMemcpy(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_status(e);
    *device_status = v;
    return LMOE_OK;
}

lmoe_status lmoe_clear_device_status(void *workspace, void *stream)
{
    if (!workspace) return LMOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(workspace, 0, sizeof(int32_t), cudaStream_t(stream)));
}

}  // extern "C"
