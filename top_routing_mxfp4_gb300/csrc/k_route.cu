// Router selection ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "MoE 稀疏激活": score all 896 experts, keep the best 16): per token the top-k
// experts by logit and the softmax over their logits.  The logits GEMM itself
// runs on the tensor cores (k_gemm_bf16.cu).
#include <float.h>
#include <math.h>

#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

// Best (value, slot) of a lane's NV values by a pairwise tournament: depth
// log2(NV) instead of an NV-long dependent chain.  Equal values keep the
// smaller slot, i.e. the smaller expert id (id = lane + 32 * slot).
template <int NV>
__device__ __forceinline__ void lane_best(const float *v, float &bv, int &bs)
{
    float tv[NV];
    int ts[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        tv[i] = v[i];
        ts[i] = i;
    }
#pragma unroll
    for (int width = 1; width < NV; width *= 2) {
#pragma unroll
        for (int i = 0; i + width < NV; i += 2 * width) {
            // tv[i] holds the best of [i, i+width), tv[i+width] of [i+width, i+2*width)
            const bool take = tv[i + width] > tv[i];  // ties keep the left (smaller slot)
            tv[i] = take ? tv[i + width] : tv[i];
            ts[i] = take ? ts[i + width] : ts[i];
        }
    }
    bv = tv[0];
    bs = ts[0];
}

// Order-preserving 32-bit key of a float: larger value, larger key; -0 and +0
// share one key (they compare equal).
__device__ __forceinline__ uint32_t order_key(float v)
{
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u) b = 0;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One warp per token.  Lane l holds experts l, l+32, ... (NV values); a taken
// or absent expert holds -inf.  Each round: every lane's best (value, slot),
// then the warp's largest value (redux max over the keys) and, among the lanes
// holding it, the smallest expert id (redux min) -- the (value desc, id asc)
// order.
// The selection of one token by one warp from its logits row `row` (any
// memory space): slots j = 0..k-1 of idx / w.
template <int NV>
__device__ __forceinline__ void select_topk(const float *row, int E, int k, int32_t *idx_t, float *w_t)
{
    const int lane = threadIdx.x & 31;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? row[e] : -INFINITY;
    }
    float sel_v = 0.f, top_v = 0.f;
    int sel_id = 0;
    for (int j = 0; j < k; ++j) {
        float bv;
        int bs;
        lane_best<NV>(v, bv, bs);
        const uint32_t key = order_key(bv);
        uint32_t kmax, bi;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(kmax) : "r"(key));
        const uint32_t cand = (key == kmax && bv != -INFINITY) ? uint32_t(lane + 32 * bs) : 0xFFFFFFFFu;
        asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(bi) : "r"(cand));
        const float wv = key_value(kmax);
        // the owner marks the winner taken
        if (int(bi & 31) == lane) {
            const int slot = int(bi >> 5);
#pragma unroll
            for (int i = 0; i < NV; ++i) v[i] = (i == slot) ? -INFINITY : v[i];
        }
        if (j == 0) top_v = wv;
        if (lane == j) { sel_v = wv; sel_id = int(bi); }
    }
    const float ex = lane < k ? expf(sel_v - top_v) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < k) {
        idx_t[lane] = sel_id;
        w_t[lane] = ex / sum;
    }
}

// One warp per token, logits in global memory.
template <int NV>
__global__ void __launch_bounds__(256) k_topk_softmax(const float *__restrict__ logits, int T, int E, int k,
                                                      int32_t *__restrict__ idx, float *__restrict__ w)
{
    pdl_enter();
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    select_topk<NV>(logits + int64_t(t) * E, E, k, idx + int64_t(t) * k, w + int64_t(t) * k);
}

// Split-K partial logits summed in slice order (then + bias), written to
// `logits` and kept in shared memory, where warp 0 selects the top-k: one CTA
// per token (one thread per expert), one launch instead of a reduction pass
// and a selection pass.
template <int NV, int NTHREADS>
__global__ void __launch_bounds__(NTHREADS) k_reduce_topk(const float *__restrict__ part, int KS, int T, int E,
                                                     const float *__restrict__ bias, float *__restrict__ logits, int k,
                                                     int32_t *__restrict__ idx, float *__restrict__ w)
{
    pdl_enter();
    extern __shared__ float row[];  // [E]
    const int t = blockIdx.x;
    const int64_t TM = int64_t(T) * E, base = int64_t(t) * E;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        float acc = 0.f;
#pragma unroll 8
        for (int s = 0; s < KS; ++s) acc += __ldcg(part + int64_t(s) * TM + base + e);
        const float v = bias ? acc + __ldg(bias + e) : acc;
        row[e] = v;
        logits[base + e] = v;
    }
    __syncthreads();
    if (threadIdx.x < 32) select_topk<NV>(row, E, k, idx + int64_t(t) * k, w + int64_t(t) * k);
}

}  // namespace

cudaError_t launch_reduce_topk(const float *part, int KS, int T, int E, const float *bias, float *logits, int k,
                               int32_t *idx, float *w, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    const size_t smem = size_t(E) * sizeof(float);  // E <= 2048: within the default 48 KB
    // one thread per expert (KS loads each) up to 896 experts; beyond, 256
    // threads, so that the selecting warp may keep its 64 values per lane in
    // registers (a 1024-thread block allows 64 registers a thread)
    const dim3 block(unsigned(E <= 896 ? round_up(E, 32) : 256));
    if (E <= 256)
        return launch_pdl(k_reduce_topk<8, 1024>, dim3(T), block, smem, st, part, KS, T, E, bias, logits, k, idx, w);
    if (E <= 896)
        return launch_pdl(k_reduce_topk<28, 1024>, dim3(T), block, smem, st, part, KS, T, E, bias, logits, k, idx, w);
    return launch_pdl(k_reduce_topk<64, 256>, dim3(T), block, smem, st, part, KS, T, E, bias, logits, k, idx, w);
}

cudaError_t launch_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx, float *w, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    const int grid = int(ceil_div(T, 8));
    if (E <= 256) { const cudaError_t le_ = launch_pdl(k_topk_softmax<8>, dim3(grid), dim3(256), 0, st, logits, T, E, k, idx, w); if (le_ != cudaSuccess) return le_; }
    else if (E <= 896) { const cudaError_t le_ = launch_pdl(k_topk_softmax<28>, dim3(grid), dim3(256), 0, st, logits, T, E, k, idx, w); if (le_ != cudaSuccess) return le_; }
    else { const cudaError_t le_ = launch_pdl(k_topk_softmax<64>, dim3(grid), dim3(256), 0, st, logits, T, E, k, idx, w); if (le_ != cudaSuccess) return le_; }
    return cudaGetLastError();
}

}  // namespace lmoe
