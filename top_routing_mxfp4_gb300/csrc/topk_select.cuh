// Top-k selection of one token's logits by one warp (larger logit first,
// equal logits by smaller expert id, -0 equal to +0) and the softmax over the
// selected logits ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "MoE 稀疏激活": keep the 16 best of the 896 experts).  Shared by the
// router's selection kernels and the small-batch routing kernel.
#pragma once

#include <math.h>

#include "lmoe_internal.cuh"

namespace lmoe {

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

}  // namespace lmoe
