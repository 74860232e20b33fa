// Block-level pieces of the dispatch schedule shared by the permute kernels
// and the small-batch routing kernel (k_route.cu): an exclusive scan over
// experts and the FFN schedule (token tiles, slot rows, work-item starts, the
// expert of each token tile) from per-expert pair counts.
#pragma once
#include "lmoe_internal.cuh"

namespace lmoe {

constexpr int SCHED_MAXE = 2048;  // experts a block scan covers at most

// Exclusive scan of v[0..n) (n <= 2048) into out[0..n], out[n] = total, by a
// block of nthreads (256 or 1024) threads; each thread owns MAXE/nthreads
// consecutive entries.  Ends with __syncthreads().
template <int NTHREADS>
__device__ void block_scan(const int32_t *v, int n, int32_t *out, int32_t *warp_tot)
{
    constexpr int PER = SCHED_MAXE / NTHREADS;
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    int32_t x[PER], tsum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = threadIdx.x * PER + j;
        x[j] = e < n ? v[e] : 0;
        tsum += x[j];
    }
    int32_t incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int32_t base = 0;
    for (int w = 0; w < wid; ++w) base += warp_tot[w];
    int32_t run = base + incl - tsum;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = threadIdx.x * PER + j;
        if (e < n) out[e] = run;
        run += x[j];
    }
    if (threadIdx.x == NTHREADS - 1) out[n] = run;
    __syncthreads();
}

// The FFN schedule from per-expert counts (shared memory, E entries):
// token tiles per expert, exclusive scan, slot rows, work-item starts and the
// expert of each token tile.
template <int NTHREADS>
__device__ void ffn_schedule_from_counts(const int32_t *cnt_s, int E, const FfnSched &sc, int32_t *tmp_s,
                                         int32_t *scan_s, int32_t *warp_tot)
{
    for (int e = threadIdx.x; e < E; e += NTHREADS) tmp_s[e] = (cnt_s[e] + sc.NT - 1) / sc.NT;
    __syncthreads();
    block_scan<NTHREADS>(tmp_s, E, scan_s, warp_tot);
    for (int e = threadIdx.x; e <= E; e += NTHREADS) {
        sc.pad_off[e] = scan_s[e] * sc.SLOT;
        sc.tiles_gu[e] = scan_s[e] * sc.MT_gu;
        sc.tiles_dn[e] = scan_s[e] * sc.MT_dn;
    }
    fill_tile_info(scan_s, E, sc, NTHREADS);
}

__device__ __forceinline__ int32_t padded_row(int32_t pos, int32_t off_e, int32_t pad_e, int NT, int SLOT)
{
    const int32_t r = pos - off_e;
    return pad_e + (r / NT) * SLOT + r % NT;
}

}  // namespace lmoe
