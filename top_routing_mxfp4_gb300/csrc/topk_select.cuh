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

// Rounds of selection.  Each round: every lane's best (value desc, expert id
// asc), then the warp's largest value (redux max over the keys) and, among
// the lanes holding it, the smallest expert id (redux min); the owner marks
// the winner taken (-inf, as absent values are).  Lane j ends with the j-th
// selection.  `RoundsAll`: lane l holds experts l, l+32, ... (NV values);
// `RoundsTwo`: two values per lane with explicit expert ids.
struct RoundOut {
    float sel_v = 0.f, top_v = 0.f;
    int sel_id = 0;
};
__device__ __forceinline__ void round_finish(int j, uint32_t kmax, uint32_t bi, RoundOut &o)
{
    const float wv = key_value(kmax);
    if (j == 0) o.top_v = wv;
    if ((threadIdx.x & 31) == j) {
        o.sel_v = wv;
        o.sel_id = int(bi);
    }
}
template <int NV>
__device__ __forceinline__ void topk_rounds_all(float *v, int k, RoundOut &o)
{
    const int lane = threadIdx.x & 31;
    for (int j = 0; j < k; ++j) {
        float bv;
        int bs;
        lane_best<NV>(v, bv, bs);
        const uint32_t key = order_key(bv);
        uint32_t kmax, bi;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(kmax) : "r"(key));
        const uint32_t cand = (key == kmax && bv != -INFINITY) ? uint32_t(lane + 32 * bs) : 0xFFFFFFFFu;
        asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(bi) : "r"(cand));
        if (int(bi & 31) == lane) {
            const int slot = int(bi >> 5);
#pragma unroll
            for (int i = 0; i < NV; ++i) v[i] = (i == slot) ? -INFINITY : v[i];
        }
        round_finish(j, kmax, bi, o);
    }
}
__device__ __forceinline__ void topk_rounds_two(float v0, int id0, float v1, int id1, int k, RoundOut &o)
{
    for (int j = 0; j < k; ++j) {
        const bool second = v1 > v0 || (v1 == v0 && id1 < id0);
        const float bv = second ? v1 : v0;
        const int bid = second ? id1 : id0;
        const uint32_t key = order_key(bv);
        uint32_t kmax, bi;
        asm volatile("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(kmax) : "r"(key));
        const uint32_t cand = (key == kmax && bv != -INFINITY) ? uint32_t(bid) : 0xFFFFFFFFu;
        asm volatile("redux.sync.min.u32 %0, %1, 0xffffffff;" : "=r"(bi) : "r"(cand));
        v0 = uint32_t(id0) == bi ? -INFINITY : v0;
        v1 = uint32_t(id1) == bi ? -INFINITY : v1;
        round_finish(j, kmax, bi, o);
    }
}

// The selection of one token by one warp from its logits row `row` (any
// memory space): slots j = 0..k-1 of idx / w, larger logit first, equal
// logits by smaller expert id.  Lane l holds experts l, l+32, ... (NV
// values).  The k-th largest of the 32 lane maxima is a lower bound of the
// k-th largest logit (k lanes hold a value at least that large), so the k
// best are among the values not below it; when there are at most 64 such
// candidates (the usual case) they are compacted into `cand` (64 entries of
// warp-private shared memory) and the rounds run over two values per lane
// instead of NV, a short dependent chain.  Otherwise, for rows wider than
// 1024 experts, and where the caller asks (CANDIDATES = false: the
// candidate pass needs more registers than a 1024-thread block allows), the
// rounds run over all values.  Every way gives the same selection.
// Softmax over the k selected logits (lane j holds the j-th), stored in slot order.
__device__ __forceinline__ void softmax_store(const RoundOut &out, int k, int32_t *idx_t, float *w_t)
{
    const int lane = threadIdx.x & 31;
    const float ex = lane < k ? expf(out.sel_v - out.top_v) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xFFFFFFFFu, sum, o);
    if (lane < k) {
        idx_t[lane] = out.sel_id;
        w_t[lane] = ex / sum;
    }
}

// (The candidate path of select_topk, below.)
template <int NV>
__device__ __forceinline__ void select_topk_candidates(const float *row, int E, int k, int32_t *idx_t, float *w_t,
                                                       float2 *cand)
{
    const int lane = threadIdx.x & 31;
    int total;
    {
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? row[e] : -INFINITY;
        }
        float bv;
        int bs;
        lane_best<NV>(v, bv, bs);
        // rank of this lane's maximum among the 32 (value desc, lane asc)
        const uint32_t bk = order_key(bv);
        int rank = 0;
#pragma unroll
        for (int o = 0; o < 32; ++o) {
            const uint32_t ok = __shfl_sync(0xFFFFFFFFu, bk, o);
            rank += (ok > bk || (ok == bk && o < lane)) ? 1 : 0;
        }
        const unsigned who = __ballot_sync(0xFFFFFFFFu, rank == k - 1);
        const uint32_t tkey = __shfl_sync(0xFFFFFFFFu, bk, __ffs(int(who)) - 1);
        int cnt = 0;
#pragma unroll
        for (int i = 0; i < NV; ++i) cnt += order_key(v[i]) >= tkey ? 1 : 0;
        int pre = cnt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(0xFFFFFFFFu, pre, o);
            if (lane >= o) pre += n;
        }
        total = __shfl_sync(0xFFFFFFFFu, pre, 31);
        if (total <= 64) {
            int pos = pre - cnt;
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                if (order_key(v[i]) >= tkey) {
                    cand[pos] = make_float2(v[i], __int_as_float(lane + 32 * i));
                    ++pos;
                }
            }
        }
    }
    RoundOut out;
    if (total <= 64) {
        __syncwarp();
        const float2 c0 = lane < total ? cand[lane] : make_float2(-INFINITY, __int_as_float(0x7FFFFFFF));
        const float2 c1 = lane + 32 < total ? cand[lane + 32] : make_float2(-INFINITY, __int_as_float(0x7FFFFFFF));
        __syncwarp();
        topk_rounds_two(c0.x, __float_as_int(c0.y), c1.x, __float_as_int(c1.y), k, out);
    } else {
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? row[e] : -INFINITY;
        }
        topk_rounds_all<NV>(v, k, out);
    }
    softmax_store(out, k, idx_t, w_t);
}

// select_topk: see above.
template <int NV, bool CANDIDATES = true>
__device__ __forceinline__ void select_topk(const float *row, int E, int k, int32_t *idx_t, float *w_t, float2 *cand)
{
    const int lane = threadIdx.x & 31;
    if constexpr (NV > 32 || !CANDIDATES) {
        // wide rows (E > 1024), or a caller short of registers: the rounds
        // over all values
        float v[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int e = lane + 32 * i;
            v[i] = e < E ? row[e] : -INFINITY;
        }
        RoundOut out;
        topk_rounds_all<NV>(v, k, out);
        softmax_store(out, k, idx_t, w_t);
    } else {
        select_topk_candidates<NV>(row, E, k, idx_t, w_t, cand);
    }
}

}  // namespace lmoe
