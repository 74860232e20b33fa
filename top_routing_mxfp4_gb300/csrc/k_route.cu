// Router: logits = x W_r^T (+ bias), then per token the top-k experts and the
// softmax over their logits ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析",
// section "MoE 稀疏激活": score all 896 experts, keep the best 16).
#include <float.h>

#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

// fp32 tiled GEMM, 32 tokens x 32 experts per CTA, K in chunks of 32.
// Thread (tx, ty): expert column tx, tokens ty*4 .. ty*4+3.
constexpr int RB = 32;

__global__ void __launch_bounds__(256) k_router_logits(const uint16_t *__restrict__ x, const float *__restrict__ Wr,
                                                       const float *__restrict__ bias, int T, int d, int E,
                                                       float *__restrict__ logits)
{
    __shared__ float xs[RB][RB + 1];
    __shared__ float ws[RB][RB + 1];
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    const int e0 = blockIdx.x * RB, t0 = blockIdx.y * RB;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
    for (int c0 = 0; c0 < d; c0 += RB) {
        // 256 threads load 32x32 of x and 32x32 of Wr (4 each)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int r = ty * 4 + i;
            const int t = t0 + r, e = e0 + r;
            xs[r][tx] = t < T ? bf16_bits_to_f32(x[int64_t(t) * d + c0 + tx]) : 0.f;
            ws[r][tx] = e < E ? Wr[int64_t(e) * d + c0 + tx] : 0.f;
        }
        __syncthreads();
#pragma unroll 8
        for (int c = 0; c < RB; ++c) {
            const float wv = ws[tx][c];
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[i] = fmaf(xs[ty * 4 + i][c], wv, acc[i]);
        }
        __syncthreads();
    }
    const int e = e0 + tx;
    if (e < E) {
        const float b = bias ? bias[e] : 0.f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int t = t0 + ty * 4 + i;
            if (t < T) logits[int64_t(t) * E + e] = bias ? acc[i] + b : acc[i];
        }
    }
}

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

cudaError_t launch_router_logits(const uint16_t *x, const float *Wr, const float *bias, int T, int d, int E,
                                 float *logits, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    dim3 grid(unsigned(ceil_div(E, RB)), unsigned(ceil_div(T, RB)));
    k_router_logits<<<grid, 256, 0, st>>>(x, Wr, bias, T, d, E, logits);
    return cudaGetLastError();
}

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
