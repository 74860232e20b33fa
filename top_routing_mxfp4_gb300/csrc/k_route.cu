// Router selection ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "MoE 稀疏激活": score all 896 experts, keep the best 16): per token the top-k
// experts by logit and the softmax over their logits.  The logits GEMM itself
// runs on the tensor cores (k_gemm_bf16.cu).
#include <float.h>
#include <math.h>

#include "lmoe_internal.cuh"
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
    if (threadIdx.x < 32) select_topk<NV, false>(row, E, k, idx + int64_t(t) * k, w + int64_t(t) * k, nullptr);
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
