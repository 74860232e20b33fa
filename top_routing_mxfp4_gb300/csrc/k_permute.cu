// Dispatch metadata ("Kimi K3 Day-0 适配剖析" section 四: index computation and
// bucketing of token->expert pairs): a stable counting sort of the pair ids
// p = t*k + j by expert, in three passes with no atomics deciding any order.
//
//   1. k_perm_hist    per chunk of CHUNK pairs: histogram over experts
//                     (shared-memory atomics only count, so order-free).
//   2. k_perm_scan    per expert: exclusive scan over chunks (each chunk's
//                     start within the expert), counts; then an exclusive scan
//                     over experts -> offsets.
//   3. k_perm_scatter per chunk, 8 warps on 8 consecutive sub-chunks: per-warp
//                     histograms -> each warp's start per expert; each warp then
//                     walks its pairs in order, ranking equal experts within a
//                     32-pair step with __match_any_sync.
#include "lmoe_internal.cuh"
#include "schedule.cuh"

namespace lmoe {
namespace {

constexpr int CHUNK = PERMUTE_CHUNK;
constexpr int WARPS = 8;
constexpr int SUB = CHUNK / WARPS;  // 512 pairs per warp
constexpr int MAXE = SCHED_MAXE;

__global__ void __launch_bounds__(256) k_perm_hist(const int32_t *__restrict__ idx, int64_t P, int E,
                                                   int32_t *__restrict__ blockhist, int32_t *status)
{
    pdl_enter();
    __shared__ int32_t h[MAXE];
    for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
    __syncthreads();
    const int64_t p0 = int64_t(blockIdx.x) * CHUNK;
    const int64_t p1 = min(P, p0 + CHUNK);
    for (int64_t p = p0 + threadIdx.x; p < p1; p += blockDim.x) {
        const int e = __ldg(idx + p);
        if (e < 0 || e >= E) set_status(status, LMOE_ERR_DEVICE_CHECK);
        else atomicAdd(&h[e], 1);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) blockhist[int64_t(blockIdx.x) * E + e] = h[e];
}

// Single CTA of 1024 threads.
__global__ void __launch_bounds__(1024) k_perm_scan(int32_t *__restrict__ blockhist, int nblk, int E,
                                                    int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                                    FfnSched sc)
{
    pdl_enter();
    __shared__ int32_t cnt[MAXE];
    __shared__ int32_t warp_tot[32];
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        // 16 chunks' counts loaded before any is overwritten, so the loads
        // overlap instead of one round trip per chunk
        int32_t run = 0;
        for (int b0 = 0; b0 < nblk; b0 += 16) {
            int32_t c[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) c[j] = b0 + j < nblk ? blockhist[int64_t(b0 + j) * E + e] : 0;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (b0 + j < nblk) blockhist[int64_t(b0 + j) * E + e] = run;
                run += c[j];
            }
        }
        cnt[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    // exclusive scan of cnt[0..E) -- each thread owns two consecutive entries
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int i0 = 2 * threadIdx.x;
    const int32_t a = i0 < E ? cnt[i0] : 0, b = i0 + 1 < E ? cnt[i0 + 1] : 0;
    int32_t s = a + b, incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int32_t wt = warp_tot[lane], wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t n = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += n;
        }
        warp_tot[lane] = wi - wt;  // exclusive prefix of warp totals
    }
    __syncthreads();
    const int32_t excl = warp_tot[wid] + incl - s;
    if (i0 < E) offsets[i0] = excl;
    if (i0 + 1 < E) offsets[i0 + 1] = excl + a;
    if (i0 + 1 == E || i0 + 2 == E) offsets[E] = excl + a + (i0 + 1 < E ? b : 0);
    if (sc.pad_off) {
        __syncthreads();
        __shared__ int32_t tmp[MAXE], scn[MAXE + 1];
        ffn_schedule_from_counts<1024>(cnt, E, sc, tmp, scn, warp_tot);
    }
}

__global__ void __launch_bounds__(256) k_perm_scatter(const int32_t *__restrict__ idx, int64_t P, int E,
                                                      const int32_t *__restrict__ blockstart,
                                                      int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                                                      const int32_t *__restrict__ offsets, FfnSched sc)
{
    pdl_enter();
    extern __shared__ int32_t wh[];  // [WARPS][E] per-warp counts, then cursors
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < WARPS * E; i += blockDim.x) wh[i] = 0;
    __syncthreads();
    const int64_t c0 = int64_t(blockIdx.x) * CHUNK;
    const int64_t s0 = c0 + int64_t(wid) * SUB;
    const int64_t s1 = min(P, s0 + SUB);
    int32_t my[SUB / 32];
#pragma unroll
    for (int i = 0; i < SUB / 32; ++i) {
        const int64_t p = s0 + 32 * i + lane;
        my[i] = p < s1 ? __ldg(idx + p) : -1;
        if (my[i] >= E) my[i] = -1;  // recorded by k_perm_hist
        if (my[i] >= 0) atomicAdd(&wh[wid * E + my[i]], 1);
    }
    __syncthreads();
    // per expert: exclusive scan over the warps, plus the chunk's start
    // (the expert's offset + the chunk's start within the expert)
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = blockstart[int64_t(blockIdx.x) * E + e] + __ldg(offsets + e);
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const int32_t c = wh[w * E + e];
            wh[w * E + e] = run;
            run += c;
        }
    }
    __syncthreads();
    int32_t *cur = wh + wid * E;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < SUB / 32; ++i) {
        const int e = my[i];
        const int64_t p = s0 + 32 * i + lane;
        const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        int32_t pos = -1;
        if (e >= 0) pos = cur[e] + __popc(m & lt);
        __syncwarp();
        if (e >= 0 && (m & lt) == 0) cur[e] += __popc(m);
        __syncwarp();
        if (p < s1) {
            inv[p] = pos;
            if (pos >= 0) perm[pos] = int32_t(p);
            if (sc.dst_row && pos >= 0)
                sc.dst_row[p] = padded_row(pos, __ldg(offsets + e), __ldg(sc.pad_off + e), sc.NT, sc.SLOT);
        }
    }
}

// All of the above in one CTA when the pairs fit one chunk (P <= CHUNK):
// per-warp histograms -> counts and per-warp starts -> exclusive scan over
// experts -> ordered scatter.  Used for decode-sized batches, where three
// launches would cost more than the work.  The P pairs are split over the 8
// warps in consecutive runs of `sub` (a multiple of 32), so every warp
// works; all expert ids are loaded before the shared-memory atomics.
__global__ void __launch_bounds__(256) k_perm_single(const int32_t *__restrict__ idx, int P, int E,
                                                     int32_t *__restrict__ counts, int32_t *__restrict__ offsets,
                                                     int32_t *__restrict__ perm, int32_t *__restrict__ inv,
                                                     int32_t *status, FfnSched sc)
{
    pdl_enter();
    extern __shared__ int4 wh_raw[];
    int32_t *wh = reinterpret_cast<int32_t *>(wh_raw);  // [WARPS][E]
    __shared__ int32_t warp_tot[WARPS];
    int32_t *off_s = wh + WARPS * E;                    // [E]
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    for (int i = threadIdx.x; i < (WARPS * E) / 4; i += blockDim.x) wh_raw[i] = make_int4(0, 0, 0, 0);
    const int sub = (P + WARPS * 32 - 1) / (WARPS * 32) * 32;  // pairs per warp, <= SUB
    const int steps = sub / 32;
    const int s0 = wid * sub, s1 = min(P, s0 + sub);
    int32_t my[SUB / 32];
#pragma unroll
    for (int i = 0; i < SUB / 32; ++i) {
        const int p = s0 + 32 * i + lane;
        my[i] = (i < steps && p < s1) ? __ldg(idx + p) : -1;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < SUB / 32; ++i) {
        int e = my[i];
        if (e >= E) {
            set_status(status, LMOE_ERR_DEVICE_CHECK);
            e = -1;
        } else if (e < 0 && i < steps && s0 + 32 * i + lane < s1) {
            set_status(status, LMOE_ERR_DEVICE_CHECK);
        }
        my[i] = e;
        if (e >= 0) atomicAdd(&wh[wid * E + e], 1);
    }
    __syncthreads();
    // per expert: total count and each warp's start inside the expert
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < WARPS; ++w) {
            const int32_t c = wh[w * E + e];
            wh[w * E + e] = run;
            run += c;
        }
        off_s[e] = run;
        counts[e] = run;
    }
    __syncthreads();
    // exclusive scan of the counts: thread i owns experts [i*PER, (i+1)*PER)
    constexpr int PER = MAXE / 256;
    int32_t v[PER], tsum = 0;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = threadIdx.x * PER + j;
        v[j] = e < E ? off_s[e] : 0;
        tsum += v[j];
    }
    int32_t incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t n = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int32_t base = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) base += (w < wid) ? warp_tot[w] : 0;
    int32_t run = base + incl - tsum;
#pragma unroll
    for (int j = 0; j < PER; ++j) {
        const int e = threadIdx.x * PER + j;
        if (e < E) {
            off_s[e] = run;
            offsets[e] = run;
        }
        run += v[j];
    }
    if (threadIdx.x == 255) offsets[E] = run;
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int32_t o = off_s[e];
#pragma unroll
        for (int w = 0; w < WARPS; ++w) wh[w * E + e] += o;
    }
    __syncthreads();
    int32_t *pad_s = nullptr;
    if (sc.pad_off) {
        // counts are offsets[e+1] - offsets[e]; reuse the shared tail for the schedule
        __shared__ int32_t tmp[MAXE], scn[MAXE + 1], wt2[WARPS];
        for (int e = threadIdx.x; e < E; e += blockDim.x) tmp[e] = counts[e];
        __syncthreads();
        ffn_schedule_from_counts<256>(tmp, E, sc, tmp, scn, wt2);
        pad_s = scn;  // slot index of each expert (times SLOT = pad_off)
    }
    int32_t *cur = wh + wid * E;
    const unsigned lt = (1u << lane) - 1u;
#pragma unroll
    for (int i = 0; i < SUB / 32; ++i) {
        if (i >= steps) break;
        const int e = my[i];
        const int p = s0 + 32 * i + lane;
        const unsigned m = __match_any_sync(0xFFFFFFFFu, e);
        int32_t pos = -1;
        if (e >= 0) pos = cur[e] + __popc(m & lt);
        __syncwarp();
        if (e >= 0 && (m & lt) == 0) cur[e] += __popc(m);
        __syncwarp();
        if (p < s1) {
            inv[p] = pos;
            if (pos >= 0) perm[pos] = p;
            if (pad_s && pos >= 0) sc.dst_row[p] = padded_row(pos, off_s[e], pad_s[e] * sc.SLOT, sc.NT, sc.SLOT);
        }
    }
}

}  // namespace

int permute_kernel_count(int64_t P)
{
    const int64_t nblk = ceil_div(P, CHUNK);
    return nblk == 1 ? 1 : (nblk == 0 ? 1 : 3);
}

size_t permute_scratch_bytes(int64_t P, int E)
{
    const int64_t nblk = ceil_div(P, CHUNK);
    return size_t(round_up(nblk * E * 4, 256));
}

cudaError_t launch_permute(const int32_t *idx, int64_t P, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                           int32_t *inv, void *scratch, int32_t *status, cudaStream_t st, const FfnSched &sched)
{
    const int nblk = int(ceil_div(P, CHUNK));
    int32_t *blockhist = static_cast<int32_t *>(scratch);
    if (nblk == 1) {
        // dynamic part; the kernel also has ~16 KB of static shared memory, so
        // the limit is raised explicitly
        const size_t smem = size_t(WARPS + 1) * E * sizeof(int32_t) + 16;
        cudaError_t e = cudaFuncSetAttribute(k_perm_single, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        {
            const cudaError_t le_ = launch_pdl(k_perm_single, dim3(1), dim3(256), smem, st, idx, int(P), E, counts, offsets, perm, inv, status, sched);
            if (le_ != cudaSuccess) return le_;
        }
        return cudaGetLastError();
    }
    if (nblk > 0) {
        {
            const cudaError_t le_ = launch_pdl(k_perm_hist, dim3(nblk), dim3(256), 0, st, idx, P, E, blockhist, status);
            if (le_ != cudaSuccess) return le_;
        }
    }
    {
        const cudaError_t le_ = launch_pdl(k_perm_scan, dim3(1), dim3(1024), 0, st, blockhist, nblk, E, counts, offsets, sched);
        if (le_ != cudaSuccess) return le_;
    }
    if (nblk > 0) {
        const size_t smem = size_t(WARPS) * E * sizeof(int32_t);
        if (smem > 48 * 1024) {  // above the default dynamic shared-memory limit (E > 1536)
            cudaError_t e = cudaFuncSetAttribute(k_perm_scatter, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
            if (e != cudaSuccess) return e;
        }
        {
            const cudaError_t le_ = launch_pdl(k_perm_scatter, dim3(nblk), dim3(256), smem, st, idx, P, E, blockhist, perm, inv, offsets, sched);
            if (le_ != cudaSuccess) return le_;
        }
    }
    return cudaGetLastError();
}

}  // namespace lmoe
