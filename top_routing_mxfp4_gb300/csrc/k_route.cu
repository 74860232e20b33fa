// Router selection ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "MoE 稀疏激活": score all 896 experts, keep the best 16): per token the top-k
// experts by logit and the softmax over their logits.  The logits GEMM itself
// runs on the tensor cores (k_gemm_bf16.cu).
#include <float.h>

#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

// (value, id) ordering of the selection: larger value first, then smaller id.
__device__ __forceinline__ bool better(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}

// One warp per token.  Lane l holds experts l, l+32, ... (NV values).
template <int NV>
__global__ void __launch_bounds__(256) k_topk_softmax(const float *__restrict__ logits, int T, int E, int k,
                                                      int32_t *__restrict__ idx, float *__restrict__ w)
{
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + int64_t(t) * E;
    float v[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        v[i] = e < E ? row[e] : -FLT_MAX;
    }
    uint64_t taken = 0;
    float sel_v = 0.f, top_v = 0.f;
    int sel_id = 0;
    for (int j = 0; j < k; ++j) {
        float bv = -FLT_MAX;
        int bi = INT32_MAX, bslot = -1;
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            if (e < E && !((taken >> i) & 1) && better(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
                bslot = i;
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
            const int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
            if (better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        // the owner marks the winner taken
        if (bslot >= 0 && lane + 32 * bslot == bi) taken |= (1ull << bslot);
        if (j == 0) top_v = bv;
        if (lane == j) { sel_v = bv; sel_id = bi; }
    }
    const float ex = lane < k ? expf(sel_v - top_v) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < k) {
        idx[int64_t(t) * k + lane] = sel_id;
        w[int64_t(t) * k + lane] = ex / sum;
    }
}

}  // namespace

cudaError_t launch_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx, float *w, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    const int grid = int(ceil_div(T, 8));
    if (E <= 256) k_topk_softmax<8><<<grid, 256, 0, st>>>(logits, T, E, k, idx, w);
    else if (E <= 896) k_topk_softmax<28><<<grid, 256, 0, st>>>(logits, T, E, k, idx, w);
    else k_topk_softmax<64><<<grid, 256, 0, st>>>(logits, T, E, k, idx, w);
    return cudaGetLastError();
}

}  // namespace lmoe
