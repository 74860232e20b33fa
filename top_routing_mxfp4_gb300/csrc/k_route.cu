// Router selection ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "MoE 稀疏激活": score all 896 experts, keep the best 16): per token the top-k
// experts by logit and the softmax over their logits.  The logits GEMM itself
// runs on the tensor cores (k_gemm_bf16.cu).
#include <float.h>
#include <math.h>

#include "lmoe_internal.cuh"
#include "tc_ptx.cuh"
#include "schedule.cuh"
#include "topk_select.cuh"

namespace lmoe {
namespace {

// One warp per token, logits in global memory.
template <int NV>
__global__ void __launch_bounds__(256) k_topk_softmax(const float *__restrict__ logits, int T, int E, int k,
                                                      int32_t *__restrict__ idx, float *__restrict__ w)
{
    __shared__ float2 cand[8][64];  // per warp: the selection's candidates
    pdl_enter();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    select_topk<NV>(logits + int64_t(t) * E, E, k, idx + int64_t(t) * k, w + int64_t(t) * k, cand[threadIdx.x >> 5]);
}

// Large batches: a persistent grid, 8 warps a CTA, each warp one token of a
// group of 8 consecutive tokens.  The group's logit rows (contiguous, E % 4
// == 0) arrive by one bulk asynchronous copy into one of two shared-memory
// buffers while the warps select the previous group's tokens from the other,
// so the selection never waits on a global load.
constexpr int TOPK_GROUP = 8;
template <int NV>
__global__ void __launch_bounds__(256) k_topk_softmax_staged(const float *__restrict__ logits, int T, int E, int k,
                                                             int32_t *__restrict__ idx, float *__restrict__ w,
                                                             int32_t *status)
{
    extern __shared__ __align__(128) float rows_s[];  // [2][TOPK_GROUP][E]
    __shared__ float2 cand[TOPK_GROUP][64];            // per warp: the selection's candidates
    __shared__ __align__(8) uint64_t bar[2];
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        tc::mbar_init_fence();
    }
    __syncthreads();
    pdl_enter();
    const int ngroups = (T + TOPK_GROUP - 1) / TOPK_GROUP;
    auto issue = [&](int gidx, int buf) {  // thread 0: the group's rows into buffer buf
        const int t0 = gidx * TOPK_GROUP, nt = min(TOPK_GROUP, T - t0);
        const uint32_t bytes = uint32_t(nt) * uint32_t(E) * 4;
        tc::fence_async_shared();
        tc::mbar_arrive_expect_tx(&bar[buf], bytes);
        tc::bulk_load(rows_s + size_t(buf) * TOPK_GROUP * E, logits + int64_t(t0) * E, bytes, &bar[buf]);
    };
    int gidx = blockIdx.x, it = 0;
    if (threadIdx.x == 0 && gidx < ngroups) issue(gidx, 0);
    for (; gidx < ngroups; gidx += gridDim.x, ++it) {
        const int buf = it & 1;
        const int gn = gidx + int(gridDim.x);
        if (threadIdx.x == 0 && gn < ngroups) issue(gn, buf ^ 1);  // the other buffer is free (barrier below)
        if (!tc::mbar_wait(&bar[buf], uint32_t((it >> 1) & 1))) {
            if (threadIdx.x == 0) set_status(status, LMOE_ERR_TIMEOUT);
            break;
        }
        const int t = gidx * TOPK_GROUP + warp;
        if (t < T)
            select_topk<NV>(rows_s + (size_t(buf) * TOPK_GROUP + warp) * E, E, k, idx + int64_t(t) * k,
                            w + int64_t(t) * k, cand[warp]);
        __syncthreads();  // every warp is done with buffer buf before it is refilled
    }
    // a copy issued for a group this CTA did not reach (after a timeout) lands before the CTA ends
    if (threadIdx.x == 0 && gidx < ngroups && gidx + int(gridDim.x) < ngroups)
        tc::mbar_wait(&bar[(it & 1) ^ 1], uint32_t(((it + 1) >> 1) & 1));
}

// Split-K partial logits summed in slice order (then + bias), written to
// `logits` and kept in shared memory, then the top-k: one CTA per token (one
// thread per expert), one launch instead of a reduction pass and a selection
// pass.  When every expert has its own thread and k is at most the number of
// warps, the block narrows the choice first, as select_topk does within a
// warp: the k-th largest of the warps' maxima is a lower bound of the k-th
// largest logit (k warps hold a value at least that large), so the k best are
// among the values not below it; each thread holding such a value appends it
// to a shared candidate list (in any order: the selection orders by value,
// then expert id), and with at most 64 candidates warp 0 runs the rounds over
// two values per lane.  Otherwise warp 0 runs the rounds over all values.
// Either way the selection is the same.
// The permute of a small batch from the token masks (PermByMask), by the
// last CTA of k_reduce_topk: NTHREADS threads, E <= 1024, T <= 64.  The
// pairs' expert ids are requested first; counts and token tiles per expert
// go through one scan as (count | tiles << 16) (both totals stay below 2^16:
// at most 64 * 32 pairs and as many tiles).
template <int NTHREADS>
__device__ void permute_from_masks(const PermByMask &pm, int T, int E, int k, const int32_t *idx)
{
    constexpr int PPT = (64 * 32 + NTHREADS - 1) / NTHREADS;  // pairs per thread: T * k <= 64 * 32
    __shared__ unsigned long long msk[1024];
    __shared__ int32_t pk[1024], scan[1025], tile0[1025], wt[32];
    const int P = T * k;
    int ep[PPT];
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
        const int p = threadIdx.x + i * NTHREADS;
        ep[i] = p < P ? __ldcg(idx + p) : 0;
    }
    for (int e = threadIdx.x; e < E; e += NTHREADS) {
        const unsigned long long m = __ldcg(pm.mask + e);
        const int32_t c = __popcll(m);
        msk[e] = m;
        pk[e] = c | (((c + pm.sc.NT - 1) / pm.sc.NT) << 16);
        pm.counts[e] = c;
    }
    __syncthreads();
    block_scan<NTHREADS>(pk, E, scan, wt);
    for (int e = threadIdx.x; e <= E; e += NTHREADS) {
        const int32_t off = scan[e] & 0xFFFF, tp = scan[e] >> 16;
        scan[e] = off;
        tile0[e] = tp;
        pm.offsets[e] = off;
        pm.sc.pad_off[e] = tp * pm.sc.SLOT;
        pm.sc.tiles_gu[e] = tp * pm.sc.MT_gu;
        pm.sc.tiles_dn[e] = tp * pm.sc.MT_dn;
    }
    __syncthreads();
    fill_tile_info(tile0, E, pm.sc, NTHREADS);
    // pair p = t*k + j of expert e: position offsets[e] + (tokens below t
    // that chose e), its atom row in the expert's token tiles
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
        const int p = threadIdx.x + i * NTHREADS;
        if (p >= P) break;
        const int t = p / k, e = ep[i];
        const int32_t pos = scan[e] + __popcll(msk[e] & ((1ull << t) - 1ull));
        pm.inv[p] = pos;
        pm.perm[pos] = p;
        pm.sc.dst_row[p] = padded_row(pos, scan[e], tile0[e] * pm.sc.SLOT, pm.sc.NT, pm.sc.SLOT);
    }
}

template <int NV, int NTHREADS>
__global__ void __launch_bounds__(NTHREADS) k_reduce_topk(const float *__restrict__ part, int KS, int T, int E,
                                                     const float *__restrict__ bias, float *__restrict__ logits, int k,
                                                     int32_t *__restrict__ idx, float *__restrict__ w, PermByMask pm)
{
    pdl_enter();
    extern __shared__ float row[];  // [E]
    __shared__ uint32_t wmax[32];   // per warp: the order key of its largest value
    __shared__ float2 cand[64];     // candidates: (value, expert id)
    __shared__ int ncand;
    __shared__ uint32_t s_bound;
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t TM = int64_t(T) * E, base = int64_t(t) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float acc = 0.f;
#pragma unroll 8
        for (int s = 0; s < KS; ++s) acc += __ldcg(part + int64_t(s) * TM + base + e);
        const float v = bias ? acc + __ldg(bias + e) : acc;
        row[e] = v;
        logits[base + e] = v;
    }
    const int nw = (E + 31) / 32;
    bool selected = false;  // by the block's candidate narrowing
    if (E <= int(blockDim.x) && k <= nw) {
        // thread e holds expert e (absent experts: key 0, below every value's key)
        const int e = threadIdx.x;
        const float v = e < E ? row[e] : -INFINITY;
        const uint32_t key = e < E ? order_key(v) : 0u;
        uint32_t m;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(m) : "r"(key));
        if (lane == 0) wmax[warp] = m;
        if (threadIdx.x == 0) ncand = 0;
        __syncthreads();
        if (warp == 0) {
            // the k-th largest warp maximum (ranks by key desc, warp asc: distinct)
            const uint32_t mk = lane < nw ? wmax[lane] : 0u;
            int rank = 0;
#pragma unroll
            for (int o = 0; o < 32; ++o) {
                const uint32_t ok = __shfl_sync(0xFFFFFFFFu, mk, o);
                rank += (ok > mk || (ok == mk && o < lane)) ? 1 : 0;
            }
            const unsigned who = __ballot_sync(0xFFFFFFFFu, lane < nw && rank == k - 1);
            if (lane == 0) s_bound = wmax[__ffs(int(who)) - 1];  // exactly one warp has rank k - 1
        }
        __syncthreads();
        if (e < E && key >= s_bound) {
            const int pos = atomicAdd(&ncand, 1);
            if (pos < 64) cand[pos] = make_float2(v, __int_as_float(e));
        }
        __syncthreads();
        const int nc = ncand;
        if (nc <= 64) {
            if (warp == 0) {
                const float2 c0 = lane < nc ? cand[lane] : make_float2(-INFINITY, __int_as_float(0x7FFFFFFF));
                const float2 c1 = lane + 32 < nc ? cand[lane + 32] : make_float2(-INFINITY, __int_as_float(0x7FFFFFFF));
                RoundOut out;
                topk_rounds_two(c0.x, __float_as_int(c0.y), c1.x, __float_as_int(c1.y), k, out);
                softmax_store(out, k, idx + int64_t(t) * k, w + int64_t(t) * k);
            }
            selected = true;
        }
    } else {
        __syncthreads();
    }
    if (!selected && threadIdx.x < 32) select_topk<NV, false>(row, E, k, idx + int64_t(t) * k, w + int64_t(t) * k, nullptr);
    if (!pm.mask) return;
    // this token's bit in its experts' masks; the last CTA to count itself in
    // does the permute
    if (threadIdx.x < 32) {
        __syncwarp();
        if (threadIdx.x < k) atomicOr(pm.mask + idx[int64_t(t) * k + threadIdx.x], 1ull << t);
    }
    __shared__ int s_last;
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(pm.counter, 1) == int(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    permute_from_masks<NTHREADS>(pm, T, E, k, idx);
}

}  // namespace

cudaError_t launch_reduce_topk(const float *part, int KS, int T, int E, const float *bias, float *logits, int k,
                               int32_t *idx, float *w, cudaStream_t st, const PermByMask &pm)
{
    if (T == 0) return cudaSuccess;
    const size_t smem = size_t(E) * sizeof(float);  // E <= 2048: within the default 48 KB
    // one thread per expert (KS loads each) up to 896 experts; beyond, 256
    // threads, so that the selecting warp may keep its 64 values per lane in
    // registers (a 1024-thread block allows 64 registers a thread)
    const dim3 block(unsigned(E <= 896 ? (pm.mask ? 1024 : round_up(E, 32)) : 256));
    if (pm.mask && (E > 896 || T > 64)) return cudaErrorInvalidValue;  // the block's permute: 1024 threads, 64 tokens
    if (E <= 256)
        return launch_pdl(k_reduce_topk<8, 1024>, dim3(T), block, smem, st, part, KS, T, E, bias, logits, k, idx, w, pm);
    if (E <= 896)
        return launch_pdl(k_reduce_topk<28, 1024>, dim3(T), block, smem, st, part, KS, T, E, bias, logits, k, idx, w, pm);
    return launch_pdl(k_reduce_topk<64, 256>, dim3(T), block, smem, st, part, KS, T, E, bias, logits, k, idx, w, pm);
}

cudaError_t launch_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx, float *w, cudaStream_t st,
                                int32_t *status)
{
    if (T == 0) return cudaSuccess;
    if (status && E % 4 == 0 && E <= 896 && T >= 1024) {
        // large batches: staged rows, a persistent grid of two CTAs per SM
        // (what the selection's registers allow)
        const size_t smem = size_t(2) * TOPK_GROUP * E * 4;
        const int ngroups = int(ceil_div(T, TOPK_GROUP));
        const int grid = ngroups < 2 * 152 ? ngroups : 2 * 152;
        cudaError_t e = E <= 256 ? cudaFuncSetAttribute(k_topk_softmax_staged<8>,
                                                         cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem))
                                 : cudaFuncSetAttribute(k_topk_softmax_staged<28>,
                                                        cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        e = E <= 256 ? launch_pdl(k_topk_softmax_staged<8>, dim3(grid), dim3(256), smem, st, logits, T, E, k, idx, w,
                                  status)
                     : launch_pdl(k_topk_softmax_staged<28>, dim3(grid), dim3(256), smem, st, logits, T, E, k, idx, w,
                                  status);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    const int grid = int(ceil_div(T, 8));
    if (E <= 256) { const cudaError_t le_ = launch_pdl(k_topk_softmax<8>, dim3(grid), dim3(256), 0, st, logits, T, E, k, idx, w); if (le_ != cudaSuccess) return le_; }
    else if (E <= 896) { const cudaError_t le_ = launch_pdl(k_topk_softmax<28>, dim3(grid), dim3(256), 0, st, logits, T, E, k, idx, w); if (le_ != cudaSuccess) return le_; }
    else { const cudaError_t le_ = launch_pdl(k_topk_softmax<64>, dim3(grid), dim3(256), 0, st, logits, T, E, k, idx, w); if (le_ != cudaSuccess) return le_; }
    return cudaGetLastError();
}

}  // namespace lmoe
