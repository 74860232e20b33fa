// The layer for small batches (batch-1 to 8-token decode steps): three
// weight-streaming kernels on the CUDA cores instead of the tensor-core
// path's seven launches.  At these sizes every touched expert serves one or
// two tokens, so the work is a set of matrix-vector products whose cost is
// reading the touched experts' MXFP4 weights once ("从Kimi K3到MiniMax-H3",
// section 二, second layer: batch-1 decode speed after kernel work; section
// 二, first layer: 4-bit weights cut the bytes a decode step streams).
//
//   k_small_route   router logits x W_r^T (the three prepared bf16 planes,
//                   fp32 sums), every CTA also rounding a share of x to MXFP8;
//                   the last CTA to finish selects each token's top-k, the
//                   softmax weights, and sorts the pairs by expert
//                   ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
//                   "MoE 稀疏激活"; "Kimi K3 Day-0 适配剖析" section 四, dispatch).
//   k_small_gateup  per (touched expert, 32 rows of I): g and u for the
//                   expert's tokens, h = silu(g) u, h rounded to MXFP8 along I.
//   k_small_down    per block of output rows, for every token: the sum over
//                   its k pairs of w * (W_down h^), rounded to bf16 (the
//                   combine, "Kimi K3 Day-0 适配剖析" section 四).  Before
//                   waiting for h it prefetches its weight rows of every routed
//                   expert into L2 (the routing is known by then).
//
// Arithmetic: each e2m1 x e4m3 product is exact in fp32 (an fp16 x fp16
// product); 16-element partial sums are accumulated in fp32, multiplied by
// the two E8M0 block scales (powers of two) and added in fp32.  The MXFP8
// rounding of x and h uses the same rules and instructions as the tensor-core
// path.  Every reduction runs in a fixed order, so results are deterministic.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lmoe_internal.cuh"
#include "tc_ptx.cuh"
#include "topk_select.cuh"

namespace lmoe {
namespace {

// ---- shared helpers -------------------------------------------------------------------

// Scale byte offset of (row R, block b) in 512-byte atoms of 128 rows x 4
// blocks, KC atoms per 128 rows: row 32*j + i of an atom, block b at byte
// 16*i + 4*j + b % 4.
__device__ __forceinline__ int64_t atom_offset(int64_t R, int b, int KC)
{
    return ((R >> 7) * KC + (b >> 2)) * 512 + (R & 31) * 16 + ((R & 127) >> 5) * 4 + (b & 3);
}

// Two e4m3 codes (low byte first) -> f16x2 (exact: e4m3 values are fp16 values).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes)
{
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(uint16_t(two_codes & 0xFFFF)));
    return h2;
}

// 16 e2m1 codes (8 bytes, element 2i in the low nibble of byte i) -> 8 f16x2
// words (exact: e2m1 values are fp16 values).
__device__ __forceinline__ void e2m1x16_to_f16x2(uint2 codes, uint32_t *out)
{
    asm("{\n\t.reg .b8 c0, c1, c2, c3, c4, c5, c6, c7;\n\t"
        "mov.b32 {c0, c1, c2, c3}, %8;\n\tmov.b32 {c4, c5, c6, c7}, %9;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, c0;\n\tcvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c2;\n\tcvt.rn.f16x2.e2m1x2 %3, c3;\n\t"
        "cvt.rn.f16x2.e2m1x2 %4, c4;\n\tcvt.rn.f16x2.e2m1x2 %5, c5;\n\t"
        "cvt.rn.f16x2.e2m1x2 %6, c6;\n\tcvt.rn.f16x2.e2m1x2 %7, c7;\n\t}"
        : "=r"(out[0]), "=r"(out[1]), "=r"(out[2]), "=r"(out[3]), "=r"(out[4]), "=r"(out[5]), "=r"(out[6]),
          "=r"(out[7])
        : "r"(codes.x), "r"(codes.y));
}

// Two fp32 values (already divided by the block scale) -> two e2m1 codes in
// the low byte (lo in the low nibble): round to nearest even, saturate at 6.
__device__ __forceinline__ uint32_t e2m1x2(float hi, float lo)
{
    uint32_t out;
    asm("{\n\t.reg .b8 b;\n\tcvt.rn.satfinite.e2m1x2.f32 b, %1, %2;\n\tcvt.u32.u8 %0, b;\n\t}"
        : "=r"(out)
        : "f"(hi), "f"(lo));
    return out;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

// ---- kernel 1: router, MXFP8 of x, top-k, pair lists ------------------------------------

constexpr int R_WARPS = 8;       // warps per routing CTA; a warp takes one half of one expert's row
constexpr int MAX_CH = 8;        // 16-byte chunks per lane of a half row (d <= 4096)

struct SmallPlan {
    int32_t *counter;      // CTAs of the routing kernel done (zero before the call; the last CTA resets it)
    int32_t *status;       // the workspace's status word
    int32_t *n_touched;    // experts with at least one pair
    int32_t *seg_expert;   // [P] touched experts, ascending
    int32_t *seg_start;    // [P + 1] first sorted position of each touched expert
    int32_t *seg_pair;     // [P] pairs sorted by (expert, pair id)
    uint8_t *xq;           // [T][d] e4m3 codes of x
    uint8_t *xs;           // scale atoms of x (rows = tokens)
    uint8_t *hq;           // [P][I] e4m3 codes of h (rows = pairs)
    uint8_t *hs;           // scale atoms of h (rows = pairs)
    float *hcap;           // diagnostics: fp32 h [P][I] before rounding, or null
};

// Router: CTA b takes experts 4b .. 4b+3, warp w the half (w & 1) of expert
// 4b + w/2's row.  Lane l loads the 16-byte chunks l, l + 32, ... of its half
// row from each of the three bf16 planes (all loads issued first), rebuilds
// the fp32 weight exactly as hi + mid + lo, and accumulates w * x for every
// token (x in shared memory as bf16).  The two halves meet in shared memory
// and the CTA writes its experts' logits.  The last CTA to finish loads all
// logits with every thread, then one warp per token selects the top k.
template <int TMAX, bool FP4>
__global__ void __launch_bounds__(32 * R_WARPS, 2) k_small_route(const uint16_t *__restrict__ x,
                                                              const uint16_t *__restrict__ Wr3,
                                                              const float *__restrict__ bias, int T, int d, int E,
                                                              int k, float *__restrict__ logits,
                                                              int32_t *__restrict__ idx, float *__restrict__ wts,
                                                              SmallPlan sp)
{
    extern __shared__ __align__(16) uint8_t r_smem[];
    uint16_t *x_s = reinterpret_cast<uint16_t *>(r_smem);  // [T][d] bf16
    __shared__ float hsum[R_WARPS][TMAX];
    __shared__ int s_last;
    __shared__ float2 s_cand[TMAX][64];  // per selecting warp: the selection's candidates
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_enter();
    const int nch = d / 16;  // 16-byte chunks of a half row
    const int task = blockIdx.x * R_WARPS + warp;  // < 2E except in the last CTA
    const int e = task >> 1, h = task & 1;
    // this warp's weights are requested before anything else
    uint4 pl[3][MAX_CH];
#pragma unroll
    for (int p = 0; p < 3; ++p) {
        const uint4 *row = reinterpret_cast<const uint4 *>(Wr3 + (int64_t(p) * E + e) * d + h * (d / 2));
#pragma unroll
        for (int i = 0; i < MAX_CH; ++i) {
            const int c = lane + 32 * i;
            pl[p][i] = (task < 2 * E && c < nch) ? __ldg(row + c) : make_uint4(0, 0, 0, 0);
        }
    }
    // x into shared memory
    for (int i = threadIdx.x; i < T * d / 8; i += blockDim.x)
        reinterpret_cast<uint4 *>(x_s)[i] = __ldg(reinterpret_cast<const uint4 *>(x) + i);
    __syncthreads();
    float acc[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) acc[t] = 0.f;
#pragma unroll
    for (int i = 0; i < MAX_CH; ++i) {
        const int c = lane + 32 * i;
        if (c < nch) {
            float wv[8];
            const uint32_t hw[4] = {pl[0][i].x, pl[0][i].y, pl[0][i].z, pl[0][i].w};
            const uint32_t mw[4] = {pl[1][i].x, pl[1][i].y, pl[1][i].z, pl[1][i].w};
            const uint32_t lw[4] = {pl[2][i].x, pl[2][i].y, pl[2][i].z, pl[2][i].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                wv[2 * q] = (__uint_as_float(hw[q] << 16) + __uint_as_float(mw[q] << 16)) + __uint_as_float(lw[q] << 16);
                wv[2 * q + 1] = (__uint_as_float(hw[q] & 0xFFFF0000u) + __uint_as_float(mw[q] & 0xFFFF0000u)) +
                                __uint_as_float(lw[q] & 0xFFFF0000u);
            }
#pragma unroll
            for (int t = 0; t < TMAX; ++t) {
                if (t < T) {
                    const uint4 xv = *reinterpret_cast<const uint4 *>(x_s + int64_t(t) * d + h * (d / 2) + c * 8);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        acc[t] = fmaf(wv[2 * q], __uint_as_float(xw[q] << 16), acc[t]);
                        acc[t] = fmaf(wv[2 * q + 1], __uint_as_float(xw[q] & 0xFFFF0000u), acc[t]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < TMAX; ++t) {
        if (t < T) {
            const float v = warp_sum(acc[t]);
            if (lane == 0) hsum[warp][t] = v;
        }
    }
    // MXFP8 of x: blocks (t, b) spread one per thread over the CTAs
    const int nb = d / 32, KC = d / 128;
    for (int g = blockIdx.x + gridDim.x * threadIdx.x; g < T * nb; g += gridDim.x * blockDim.x) {
        const int t = g / nb, b = g - t * nb;
        const uint4 *src = reinterpret_cast<const uint4 *>(x_s + int64_t(t) * d + b * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 r = src[i];
            const uint32_t rw[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                v[8 * i + 2 * q] = __uint_as_float(rw[q] << 16);
                v[8 * i + 2 * q + 1] = __uint_as_float(rw[q] & 0xFFFF0000u);
            }
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
        const uint32_t sb = mx_scale_byte(__uint_as_float(amax), FP4 ? 2 : 8);
        const float inv = mx_inv_scale(sb);
        if constexpr (FP4) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] *= inv;
            *reinterpret_cast<uint4 *>(sp.xq + int64_t(t) * (d / 2) + b * 16) =
                make_uint4(e2m1x8(v), e2m1x8(v + 8), e2m1x8(v + 16), e2m1x8(v + 24));
        } else {
            uint32_t c[8];
#pragma unroll
            for (int i = 0; i < 8; ++i)
                c[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
            uint4 *dst = reinterpret_cast<uint4 *>(sp.xq + int64_t(t) * d + b * 32);
            dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
            dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
        }
        sp.xs[atom_offset(t, b, KC)] = uint8_t(sb);
    }
    __syncthreads();
    // this CTA's logits: the two halves of each of its experts
    for (int i = threadIdx.x; i < (R_WARPS / 2) * T; i += blockDim.x) {
        const int el = i / T, t = i - el * T;
        const int ee = blockIdx.x * (R_WARPS / 2) + el;
        if (ee < E) {
            const float v = hsum[2 * el][t] + hsum[2 * el + 1][t];
            logits[int64_t(t) * E + ee] = bias ? v + __ldg(bias + ee) : v;
        }
    }
    // the last CTA to finish selects and sorts
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s_last = atomicAdd(sp.counter, 1) == int(gridDim.x) - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    float *lg_s = reinterpret_cast<float *>(r_smem);  // [T][E]
    for (int i = threadIdx.x; i < T * E; i += blockDim.x) lg_s[i] = __ldcg(logits + i);
    __syncthreads();
    if (warp < T) {
        const int t = warp;
        float2 *cand = s_cand[t];
        if (E <= 256) select_topk<8>(lg_s + t * E, E, k, idx + int64_t(t) * k, wts + int64_t(t) * k, cand);
        else if (E <= 896) select_topk<28>(lg_s + t * E, E, k, idx + int64_t(t) * k, wts + int64_t(t) * k, cand);
        else select_topk<64>(lg_s + t * E, E, k, idx + int64_t(t) * k, wts + int64_t(t) * k, cand);
    }
    __syncthreads();
    // pairs sorted by (expert, pair id): position = number of pairs before it
    const int P = T * k;
    int32_t *s_e = reinterpret_cast<int32_t *>(lg_s + T * E);  // [256] expert of each sorted position
    int32_t *s_p = s_e + 256;                                  // [256] pair at each sorted position
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        const int ep = idx[p];
        int pos = 0;
        for (int q = 0; q < P; ++q) {
            const int eq = idx[q];
            pos += (eq < ep || (eq == ep && q < p)) ? 1 : 0;
        }
        s_e[pos] = ep;
        s_p[pos] = p;
    }
    __syncthreads();
    for (int q = threadIdx.x; q < P; q += blockDim.x) {
        sp.seg_pair[q] = s_p[q];
        if (q == 0 || s_e[q] != s_e[q - 1]) {
            int u = 0;  // heads before q
            for (int r = 1; r <= q; ++r) u += (s_e[r] != s_e[r - 1]) ? 1 : 0;
            sp.seg_expert[u] = s_e[q];
            sp.seg_start[u] = q;
        }
    }
    if (threadIdx.x == 0) {
        int n = P > 0 ? 1 : 0;
        for (int r = 1; r < P; ++r) n += (s_e[r] != s_e[r - 1]) ? 1 : 0;
        *sp.n_touched = n;
        sp.seg_start[n] = P;
        *sp.counter = 0;  // ready for the next call on this workspace
    }
}

// ---- kernel 2: gate/up, SwiGLU, MXFP8 of h --------------------------------------------------

constexpr int G_WARPS = 16;   // 4 row tiles of 16 (32 gate + 32 up rows) x 4 quarters of K per unit
constexpr int G_PAIRS = SMALL_MAX_TOKENS;  // pairs of one expert a unit serves at most (one per token)

// Four e2m1 code pairs (a 32-bit word, element 2i in the low nibble of byte
// i) -> four f16x2 words (exact: e2m1 values are fp16 values), element 2i in
// the low half of word i.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t codes, uint32_t &w0, uint32_t &w1, uint32_t &w2, uint32_t &w3)
{
    asm("{\n\t.reg .b8 c0, c1, c2, c3;\n\t"
        "mov.b32 {c0, c1, c2, c3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, c0;\n\tcvt.rn.f16x2.e2m1x2 %1, c1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, c2;\n\tcvt.rn.f16x2.e2m1x2 %3, c3;\n\t}"
        : "=r"(w0), "=r"(w1), "=r"(w2), "=r"(w3)
        : "r"(codes));
}

// D += A B for one 16 x 16 (row-major fp16) by 16 x 8 (column-major fp16)
// block, fp32 accumulation: the warp-level tensor-core instruction, used
// here for its cheap exact fp16 products at one to eight tokens.
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
                 "{%0, %1, %2, %3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Shared-memory layout of one gate/up unit (byte offsets; row strides padded
// so that the warps' loads hit distinct banks).
struct GateupSmem {
    int wrow, xrow;                      // weight row stride (bytes), x row stride (halves)
    size_t w, sf, sx, xh, part, total;
    __host__ __device__ GateupSmem(int d, int npair)
    {
        wrow = d / 2 + 16;
        xrow = d + 32;
        w = 0;                                         // [64][wrow] e2m1 codes
        sf = w + size_t(64) * wrow;                    // [d/32][64] weight block scales (fp32)
        sx = sf + size_t(d / 32) * 64 * 4;             // [d/32][G_PAIRS] x block scales (fp32)
        xh = sx + size_t(d / 32) * G_PAIRS * 4;        // [npair][xrow] x^ as fp16
        part = xh + size_t(npair) * xrow * 2;          // [2][4][64][G_PAIRS] K-quarter partial sums (x^ rows: tokens)
        total = part + size_t(2) * 4 * 64 * G_PAIRS * 4;  // two units' sums
    }
};

// Unit = (touched expert u, block rb of 32 rows of I): its 32 gate and 32 up
// weight rows, in four quarters of K.  Warp group q (warps 4q .. 4q+3) owns
// quarter q throughout: it copies that quarter of the unit's 64 rows into
// shared memory (one bulk asynchronous copy per row, rows padded), turns the
// quarter's block scales and x^ of the expert's pairs (at most one per token,
// so at most G_PAIRS) into fp32 scales and fp16 code values (both exact),
// waits for its copies, and forms the quarter's block products: warp 4q + m
// takes the 16-row tile m; per 32-element scale block, two m16n8k16
// tensor-core products (e2m1 codes widened to fp16, x^ in fp16, exact
// products) give the block's sums for the unit's pairs (the MMA's N
// columns), which are scaled by the two E8M0 block scales and added in fp32.
// K is consumed in a permuted order inside each block, the same for both
// operands: lane (g, t) takes elements 8t .. 8t+7 of the block (one 32-bit
// word of codes per row), the first four in the first product and the last
// four in the second.  As soon as a group is done with its quarter it issues
// the copies of the next unit's quarter, so the next unit's weights stream
// in while this unit is finished.  The four quarters' sums meet in shared
// memory (added in quarter order) and warp j forms h of pair slot j:
// silu(g) * u, its MXFP8 block over the 32 rows, stored as the pair's row.
template <bool FP4>
__global__ void __launch_bounds__(32 * G_WARPS) k_small_gateup(const uint8_t *__restrict__ gate_q,
                                                               const uint8_t *__restrict__ gate_s,
                                                               const uint8_t *__restrict__ up_q,
                                                               const uint8_t *__restrict__ up_s, int T, int d, int I,
                                                               int k, int npair_max, SmallPlan sp)
{
    extern __shared__ __align__(128) uint8_t g_smem[];
    const GateupSmem L(d, npair_max);
    uint8_t *wq = g_smem + L.w;
    float *sf = reinterpret_cast<float *>(g_smem + L.sf);
    float *sx = reinterpret_cast<float *>(g_smem + L.sx);
    uint16_t *xh = reinterpret_cast<uint16_t *>(g_smem + L.xh);
    float *part = reinterpret_cast<float *>(g_smem + L.part);
    __shared__ __align__(8) uint64_t bar[4];
    const int KCd = d / 128, RTI = (I + 127) / 128, KCi = (I + 127) / 128;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q = warp >> 2, mt = warp & 3, gt = threadIdx.x & 127;  // quarter, row tile, thread in group
    if (threadIdx.x < 4) tc::mbar_init(&bar[threadIdx.x], 1);
    if (threadIdx.x == 0) tc::mbar_init_fence();
    __syncthreads();
    // this quarter's 128-element chunks of K: [kc0, kc1) (a quarter may be
    // empty when d < 512), 64 code bytes per row each
    const int kc0 = q * KCd / 4, kc1 = (q + 1) * KCd / 4, nkq = kc1 - kc0;
    const uint32_t qbytes = uint32_t(nkq) * 64, qoff = uint32_t(kc0) * 64;
    const int nrb = I / 32;
    pdl_enter();
    // First round of loads: n_touched, this CTA's first unit (expert, pair
    // range; blockIdx.x < P * I / 32 keeps the reads in bounds) and quarter q
    // of x^ of every token with its block scales (the same for every unit).
    const int nt = __ldcg(sp.n_touched);
    int e_n = __ldcg(sp.seg_expert + blockIdx.x / nrb);
    int q0_n = __ldcg(sp.seg_start + blockIdx.x / nrb), q1_n = __ldcg(sp.seg_start + blockIdx.x / nrb + 1);
    const int cq = 8 * nkq;  // 16-element chunks of the quarter
    {
        uint4 xv[4];
        uint32_t xb[4];
#pragma unroll
        for (int m = 0; m < 4; ++m) {  // T * cq <= 512 (T <= 8, d <= 4096)
            const int i = gt + 128 * m;
            xv[m] = make_uint4(0, 0, 0, 0);
            xb[m] = 0;
            if (i < T * cq) {
                const int t = i / cq, c = 8 * kc0 + (i - t * cq);
                if constexpr (FP4) {
                    const uint2 v = __ldcg(reinterpret_cast<const uint2 *>(sp.xq + int64_t(t) * (d / 2)) + c);
                    xv[m] = make_uint4(v.x, v.y, 0, 0);
                } else {
                    xv[m] = __ldcg(reinterpret_cast<const uint4 *>(sp.xq + int64_t(t) * d) + c);
                }
                if ((c & 1) == 0) xb[m] = __ldcg(sp.xs + atom_offset(t, c >> 1, KCd));
            }
        }
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i = gt + 128 * m;
            if (i < T * cq) {
                const int t = i / cq, c = 8 * kc0 + (i - t * cq);
                uint32_t h[8];
                if constexpr (FP4) {
                    e2m1x16_to_f16x2(make_uint2(xv[m].x, xv[m].y), h);
                } else {
                    const uint32_t vw[4] = {xv[m].x, xv[m].y, xv[m].z, xv[m].w};
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        h[2 * v] = e4m3x2_to_f16x2(vw[v]);
                        h[2 * v + 1] = e4m3x2_to_f16x2(vw[v] >> 16);
                    }
                }
                uint4 *dst = reinterpret_cast<uint4 *>(xh + t * L.xrow + 16 * c);
                dst[0] = make_uint4(h[0], h[1], h[2], h[3]);
                dst[1] = make_uint4(h[4], h[5], h[6], h[7]);
                if ((c & 1) == 0) sx[(c >> 1) * G_PAIRS + t] = e8m0_to_f32(xb[m]);
            }
        }
    }
    const int nunits = nt * nrb;
    // this group's copies of quarter q of `unit`'s 64 rows (expert e)
    auto issue = [&](int unit, int e) {
        if (warp != 4 * q) return;
        const int rb = unit % nrb;
        if (lane == 0) {
            tc::fence_async_shared();
            tc::mbar_arrive_expect_tx(&bar[q], 64 * qbytes);
        }
        __syncwarp();
        if (qbytes == 0) return;
        const int64_t r0 = int64_t(e) * I + rb * 32 + lane;
        tc::bulk_load(wq + lane * L.wrow + qoff, gate_q + r0 * (d / 2) + qoff, qbytes, &bar[q]);
        tc::bulk_load(wq + (32 + lane) * L.wrow + qoff, up_q + r0 * (d / 2) + qoff, qbytes, &bar[q]);
    };
    // a unit's quarter-q block-scale words (<= 512 per quarter: 4 a thread) and
    // the pair ids of its pair slots (loads only: used one unit later)
    auto fetch = [&](int unit, int e, int q0, int q1, uint32_t (&wd)[4], int (&pid)[G_PAIRS]) {
        const int rb = unit % nrb;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i = gt + 128 * m;
            wd[m] = 0;
            if (i < 64 * nkq) {
                const int r = i / nkq, kc = kc0 + (i - r * nkq);
                const int row = rb * 32 + (r & 31);
                const uint8_t *ms = r < 32 ? gate_s : up_s;
                wd[m] = __ldg(reinterpret_cast<const uint32_t *>(
                    ms + ((int64_t(e) * RTI + (row >> 7)) * KCd + kc) * 512 + (row & 31) * 16 + ((row & 127) >> 5) * 4));
            }
        }
        const int np = min(q1 - q0, npair_max);
#pragma unroll
        for (int j = 0; j < G_PAIRS; ++j) pid[j] = j < np ? __ldcg(sp.seg_pair + q0 + j) : -1;
    };
    // the tokens of the pair slots, 4 bits each (0xF: no pair)
    auto slot_tokens = [&](const int (&pid)[G_PAIRS]) {
        uint32_t sl = 0xFFFFFFFFu;
#pragma unroll
        for (int j = 0; j < G_PAIRS; ++j)
            if (pid[j] >= 0) sl = (sl & ~(0xFu << (4 * j))) | (uint32_t(pid[j] / k) << (4 * j));
        return sl;
    };
    auto group_sync = [&]() { asm volatile("bar.sync %0, 128;" ::"r"(1 + q) : "memory"); };
    uint32_t wd[4] = {0, 0, 0, 0};
    int pid[G_PAIRS];
#pragma unroll
    for (int j = 0; j < G_PAIRS; ++j) pid[j] = -1;
    int e = e_n, q0 = q0_n, q1 = q1_n;
    if (int(blockIdx.x) < nunits) {
        issue(blockIdx.x, e);
        fetch(blockIdx.x, e, q0, q1, wd, pid);
    }
    uint32_t parity = 0;
    int it = 0;
    for (int unit = blockIdx.x; unit < nunits; unit += gridDim.x, ++it) {
        const int rb = unit % nrb;
        const int np = min(q1 - q0, npair_max);
        const uint32_t slots = slot_tokens(pid);
        // the next unit's descriptor (used after this unit's products)
        const int unit_n = unit + int(gridDim.x);
        if (unit_n < nunits) {
            e_n = __ldcg(sp.seg_expert + unit_n / nrb);
            q0_n = __ldcg(sp.seg_start + unit_n / nrb);
            q1_n = __ldcg(sp.seg_start + unit_n / nrb + 1);
        }
        // quarter q's weight block scales as fp32
#pragma unroll
        for (int m = 0; m < 4; ++m) {
            const int i = gt + 128 * m;
            if (i < 64 * nkq) {
                const int r = i / nkq, kc = kc0 + (i - r * nkq);
#pragma unroll
                for (int j = 0; j < 4; ++j) sf[(4 * kc + j) * 64 + r] = e8m0_to_f32((wd[m] >> (8 * j)) & 0xFF);
            }
        }
        group_sync();  // the quarter's scales are in place (and, the first time, x^)
        // a wait that runs out records the timeout; every thread then leaves
        // at the CTA barrier below (the products of this unit are discarded)
        const bool landed = tc::mbar_wait(&bar[q], parity);
        if (!landed && gt == 0) set_status(sp.status, LMOE_ERR_TIMEOUT);
        // block products on the tensor cores: lane (g, t4) reads pair slot g's
        // token (the B column) and accumulates pair slots 2 t4, 2 t4 + 1 (C)
        const int g = lane >> 2, t4 = lane & 3;
        const uint8_t *rowg = wq + (16 * mt + g) * L.wrow + 4 * t4;
        const uint8_t *rowg8 = rowg + 8 * L.wrow;
        const int tb = int((slots >> (4 * g)) & 0xF);          // token of B column g (15: none)
        const int tc0 = int((slots >> (8 * t4)) & 0xF);        // token of C column 2 t4
        const int tc1 = int((slots >> (8 * t4 + 4)) & 0xF);    // token of C column 2 t4 + 1
        const bool col_ok = g < np;
        const uint16_t *xcol = xh + (col_ok ? tb : 0) * L.xrow + 8 * t4;
        const float *sx0 = sx + (2 * t4 < np ? tc0 : 0), *sx1 = sx + (2 * t4 + 1 < np ? tc1 : 0);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        const int b0 = 4 * kc0, b1 = 4 * kc1;
#pragma unroll 4
        for (int b = b0; b < b1; ++b) {
            const uint32_t wg = *reinterpret_cast<const uint32_t *>(rowg + 16 * b);
            const uint32_t wg8 = *reinterpret_cast<const uint32_t *>(rowg8 + 16 * b);
            uint4 xv = make_uint4(0, 0, 0, 0);
            if (col_ok) xv = *reinterpret_cast<const uint4 *>(xcol + 32 * b);
            uint32_t ag0, ag1, ag2, ag3, ah0, ah1, ah2, ah3;
            e2m1x8_to_f16x2(wg, ag0, ag1, ag2, ag3);
            e2m1x8_to_f16x2(wg8, ah0, ah1, ah2, ah3);
            // the block's two halves as independent products, then added
            float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
            mma_16816(c0, ag0, ah0, ag1, ah1, xv.x, xv.y);
            mma_16816(c1, ag2, ah2, ag3, ah3, xv.z, xv.w);
            const float s0 = sf[b * 64 + 16 * mt + g], s8 = sf[b * 64 + 16 * mt + g + 8];
            const float x0 = sx0[b * G_PAIRS], x1 = sx1[b * G_PAIRS];
            acc[0] = fmaf((c0[0] + c1[0]) * s0, x0, acc[0]);
            acc[1] = fmaf((c0[1] + c1[1]) * s0, x1, acc[1]);
            acc[2] = fmaf((c0[2] + c1[2]) * s8, x0, acc[2]);
            acc[3] = fmaf((c0[3] + c1[3]) * s8, x1, acc[3]);
        }
        float *pw = part + (((it & 1) * 4 + q) * 64 + 16 * mt + g) * G_PAIRS + 2 * t4;
        pw[0] = acc[0];
        pw[1] = acc[1];
        pw[8 * G_PAIRS] = acc[2];
        pw[8 * G_PAIRS + 1] = acc[3];
        parity ^= 1;
        // the next unit's scale words and pair tokens (its descriptor has arrived)
        uint32_t wd_n[4] = {0, 0, 0, 0};
        int pid_n[G_PAIRS];
#pragma unroll
        for (int j = 0; j < G_PAIRS; ++j) pid_n[j] = -1;
        const bool next = landed && unit_n < nunits;
        if (next) fetch(unit_n, e_n, q0_n, q1_n, wd_n, pid_n);
        group_sync();  // the group is done with its quarter of the weights and scales
        if (next) issue(unit_n, e_n);
        if (__syncthreads_or(!landed)) {  // every quarter's sums are in place, or some wait ran out
            // copies already issued for the next unit land before the CTA ends (bounded)
            if (next) tc::mbar_wait(&bar[q], parity);
            return;
        }
        if (warp < np) {
            const int j = warp;
            int p = 0;
#pragma unroll
            for (int jj = 0; jj < G_PAIRS; ++jj) p = jj == j ? pid[jj] : p;
            const float *pu = part + (it & 1) * 4 * 64 * G_PAIRS;
            float gv = 0.f, uv = 0.f;
#pragma unroll
            for (int qq = 0; qq < 4; ++qq) {
                gv += pu[(qq * 64 + lane) * G_PAIRS + j];
                uv += pu[(qq * 64 + 32 + lane) * G_PAIRS + j];
            }
            const float h = __fdividef(gv, 1.f + __expf(-gv)) * uv;
            if (sp.hcap) sp.hcap[int64_t(p) * I + rb * 32 + lane] = h;
            uint32_t amax;
            asm("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(amax) : "r"(__float_as_uint(h) & 0x7FFFFFFFu));
            const uint32_t sb = mx_scale_byte(__uint_as_float(amax), FP4 ? 2 : 8);
            if constexpr (FP4) {
                // e2m1 code of this lane's h; lanes 2i and 2i+1 share byte i (element 2i in the low nibble)
                const uint32_t code = e2m1x2(0.f, h * mx_inv_scale(sb)) & 0xF;
                const uint32_t hi = __shfl_down_sync(0xFFFFFFFFu, code, 1);
                if ((lane & 1) == 0) sp.hq[int64_t(p) * (I / 2) + rb * 16 + lane / 2] = uint8_t(code | (hi << 4));
            } else {
                sp.hq[int64_t(p) * I + rb * 32 + lane] = uint8_t(e4m3x2(h * mx_inv_scale(sb), 0.f) & 0xFF);
            }
            if (lane == 0) sp.hs[atom_offset(p, rb, KCi)] = uint8_t(sb);
        }
        e = e_n;
        q0 = q0_n;
        q1 = q1_n;
#pragma unroll
        for (int m = 0; m < 4; ++m) wd[m] = wd_n[m];
#pragma unroll
        for (int j = 0; j < G_PAIRS; ++j) pid[j] = pid_n[j];
    }
}

// a += the 16 products of e2m1 codes (8 bytes, element 2i in the low nibble
// of byte i) with fp16 values (8 f16x2 words, element 2i in the low half):
// each code is widened to fp16 and multiplied in fp16, which is exact (at
// most 6 significant bits, within the fp16 range), then the products are
// added in fp32, even and odd elements into separate sums.
__device__ __forceinline__ void dot16(uint2 codes, const uint32_t *xv, float &a0, float &a1)
{
    uint32_t w[8];
    e2m1x16_to_f16x2(codes, w);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const __half2 prod = __hmul2(*reinterpret_cast<const __half2 *>(&w[i]), *reinterpret_cast<const __half2 *>(&xv[i]));
        const float2 f = __half22float2(prod);
        a0 += f.x;
        a1 += f.y;
    }
}

// ---- kernel 3: down, gate weights, combine ----------------------------------------------------

constexpr int D_WARPS = 12;
constexpr int D_RPW = 3;   // at most 3 output rows per warp (rows per CTA <= 36)
constexpr int D_PB = 4;    // pairs whose dot products are formed together

// CTA = block of `rpc` consecutive output rows (warp w takes rows w, w + 12,
// ...).  The rows of W_down[e] for those outputs are contiguous, so each
// routed pair's weights arrive by one bulk copy into shared memory; pairs go
// in groups of `gp` through two buffers.  The routing is complete when this
// kernel starts (the kernel before it waited for it), so the first two
// groups' copies are issued before waiting for h.  h^ of every pair is kept
// in shared memory as fp16 code values (exact) with its block scales.  Lane
// l covers the 16-element chunks l, l + 32, ... of a weight row; for each row
// and token it accumulates sum_j w_j * (its part of W_down[e_j][row] .
// h^_(t,j)) over the token's pairs in slot order (the dot products of D_PB
// pairs are formed together), then one warp reduction gives y[t][row].
template <bool FP4>
__global__ void __launch_bounds__(32 * D_WARPS) k_small_down(const uint8_t *__restrict__ down_q,
                                                             const uint8_t *__restrict__ down_s,
                                                             const int32_t *__restrict__ idx,
                                                             const float *__restrict__ wts, int T, int d, int I,
                                                             int k, int rpc, int gp, uint16_t *__restrict__ y,
                                                             SmallPlan sp)
{
    extern __shared__ __align__(128) uint8_t d_smem[];
    const int P = T * k;
    const int Ip = (I + 127) / 128 * 128, KCi = Ip / 128, RTd = d / 128;
    const uint32_t row_bytes = uint32_t(Ip / 2);
    const int c0 = blockIdx.x * rpc, c1 = min(d, c0 + rpc), nr = c1 - c0;
    const size_t wbuf_bytes = size_t(gp) * rpc * row_bytes;
    uint8_t *wbuf = d_smem;                                                         // [2][gp][rpc][Ip/2]
    uint32_t *swb = reinterpret_cast<uint32_t *>(d_smem + 2 * wbuf_bytes);           // [2][gp][rpc][KCi]
    uint32_t *hh = swb + 2 * gp * rpc * KCi;                                         // [P][I/2] f16x2
    float *hsf = reinterpret_cast<float *>(hh + size_t(P) * (I / 2));                // [P][I/32] scales
    int32_t *e_s = reinterpret_cast<int32_t *>(hsf + size_t(P) * (I / 32));          // [P]
    float *w_s = reinterpret_cast<float *>(e_s + P);                                 // [P]
    __shared__ __align__(8) uint64_t bar[2];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ngroups = (P + gp - 1) / gp;
    if (threadIdx.x == 0) {
        tc::mbar_init(&bar[0], 1);
        tc::mbar_init(&bar[1], 1);
        tc::mbar_init_fence();
    }
    // the routing: complete (the kernel before this one waited for it)
    for (int p = threadIdx.x; p < P; p += blockDim.x) {
        e_s[p] = __ldcg(idx + p);
        w_s[p] = __ldcg(wts + p);
    }
    __syncthreads();
    auto issue = [&](int g) {  // group g's weights into buffer g % 2
        const int pa = g * gp, np = min(gp, P - pa);
        uint8_t *wb = wbuf + (g & 1) * wbuf_bytes;
        uint32_t *sb = swb + (g & 1) * gp * rpc * KCi;
        if (threadIdx.x == 0) {
            tc::fence_async_shared();
            tc::mbar_arrive_expect_tx(&bar[g & 1], uint32_t(np) * nr * row_bytes);
            for (int i = 0; i < np; ++i)
                tc::bulk_load(wb + size_t(i) * rpc * row_bytes, down_q + (int64_t(e_s[pa + i]) * d + c0) * row_bytes,
                              uint32_t(nr) * row_bytes, &bar[g & 1]);
        }
        for (int i = threadIdx.x; i < np * nr * KCi; i += blockDim.x) {
            const int pi = i / (nr * KCi), rem = i - pi * (nr * KCi), r = rem / KCi, kc = rem - r * KCi;
            const int c = c0 + r;
            sb[(pi * rpc + r) * KCi + kc] = __ldg(reinterpret_cast<const uint32_t *>(
                down_s + ((int64_t(e_s[pa + pi]) * RTd + (c >> 7)) * KCi + kc) * 512 + (c & 31) * 16 +
                ((c & 127) >> 5) * 4));
        }
    };
    issue(0);
    if (ngroups > 1) issue(1);
    pdl_enter();
    // h^ of every pair, as fp16 code values, and its block scales
    for (int i = threadIdx.x; i < P * I / 16; i += blockDim.x) {
        uint4 *dst = reinterpret_cast<uint4 *>(hh + size_t(i) * 8);
        if constexpr (FP4) {
            uint32_t f[8];
            e2m1x16_to_f16x2(__ldcg(reinterpret_cast<const uint2 *>(sp.hq) + i), f);
            dst[0] = make_uint4(f[0], f[1], f[2], f[3]);
            dst[1] = make_uint4(f[4], f[5], f[6], f[7]);
        } else {
            const uint4 v = __ldcg(reinterpret_cast<const uint4 *>(sp.hq) + i);
            dst[0] = make_uint4(e4m3x2_to_f16x2(v.x), e4m3x2_to_f16x2(v.x >> 16), e4m3x2_to_f16x2(v.y),
                                e4m3x2_to_f16x2(v.y >> 16));
            dst[1] = make_uint4(e4m3x2_to_f16x2(v.z), e4m3x2_to_f16x2(v.z >> 16), e4m3x2_to_f16x2(v.w),
                                e4m3x2_to_f16x2(v.w >> 16));
        }
    }
    for (int i = threadIdx.x; i < P * (I / 32); i += blockDim.x) {
        const int p = i / (I / 32), b = i - p * (I / 32);
        hsf[i] = e8m0_to_f32(__ldcg(sp.hs + atom_offset(p, b, KCi)));
    }
    __syncthreads();
    const int nchunk = I / 16;
    float acc[D_RPW];
#pragma unroll
    for (int i = 0; i < D_RPW; ++i) acc[i] = 0.f;
    int cur_t = 0;
    auto flush = [&]() {
#pragma unroll
        for (int i = 0; i < D_RPW; ++i) {
            const int r = warp + D_WARPS * i;
            const float v = warp_sum(acc[i]);  // every lane takes part
            if (lane == 0 && r < nr) y[int64_t(cur_t) * d + c0 + r] = __bfloat16_as_ushort(__float2bfloat16_rn(v));
            acc[i] = 0.f;
        }
    };
    for (int g = 0; g < ngroups; ++g) {
        if (!tc::mbar_wait(&bar[g & 1], uint32_t((g >> 1) & 1))) {
            set_status(sp.status, LMOE_ERR_TIMEOUT);
            return;
        }
        const int pa = g * gp, np = min(gp, P - pa);
        const uint8_t *wb = wbuf + (g & 1) * wbuf_bytes;
        const uint32_t *sb = swb + (g & 1) * gp * rpc * KCi;
        for (int pb = 0; pb < np; pb += D_PB) {
            float dots[D_PB][D_RPW];
#pragma unroll
            for (int u = 0; u < D_PB; ++u) {
                const int pi = pb + u, p = pa + pi;
#pragma unroll
                for (int i = 0; i < D_RPW; ++i) {
                    const int r = warp + D_WARPS * i;
                    float dj = 0.f;
                    if (pi < np && r < nr) {
                        for (int ch = lane; ch < nchunk; ch += 32) {
                            const uint2 cw =
                                *reinterpret_cast<const uint2 *>(wb + (size_t(pi) * rpc + r) * row_bytes + ch * 8);
                            const int b = ch >> 1;
                            const float s_w = e8m0_to_f32((sb[(pi * rpc + r) * KCi + (b >> 2)] >> (8 * (b & 3))) & 0xFF);
                            const uint4 ha = *reinterpret_cast<const uint4 *>(hh + size_t(p) * (I / 2) + ch * 8);
                            const uint4 hb = *reinterpret_cast<const uint4 *>(hh + size_t(p) * (I / 2) + ch * 8 + 4);
                            const uint32_t hv[8] = {ha.x, ha.y, ha.z, ha.w, hb.x, hb.y, hb.z, hb.w};
                            float a0 = 0.f, a1 = 0.f;
                            dot16(cw, hv, a0, a1);
                            dj = fmaf((a0 + a1) * s_w, hsf[p * (I / 32) + b], dj);
                        }
                    }
                    dots[u][i] = dj;
                }
            }
#pragma unroll
            for (int u = 0; u < D_PB; ++u) {
                const int pi = pb + u, p = pa + pi;
                if (pi < np) {
                    const int t = p / k;
                    if (t != cur_t) {
                        flush();
                        cur_t = t;
                    }
                    const float wp = w_s[p];
#pragma unroll
                    for (int i = 0; i < D_RPW; ++i) acc[i] = fmaf(wp, dots[u][i], acc[i]);
                }
            }
        }
        __syncthreads();  // buffer g % 2 is free
        if (g + 2 < ngroups) issue(g + 2);
    }
    flush();
}

}  // namespace

// ---- host side --------------------------------------------------------------------------------

SmallLayout small_layout(int T, int d, int E, int k, int I)
{
    SmallLayout L{};
    const int64_t P = int64_t(T) * k;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += size_t(round_up(int64_t(bytes), 256));
        return o;
    };
    const int Ip = int(round_up(I, 128));
    L.n_touched = take(16);
    L.seg_expert = take(size_t(P) * 4);
    L.seg_start = take(size_t(P + 1) * 4);
    L.seg_pair = take(size_t(P) * 4);
    L.xq = take(size_t(T) * d);
    L.xs = take(size_t(ceil_div(T, 128)) * (d / 128) * 512);
    L.hq = take(size_t(P) * I);
    L.hs = take(size_t(ceil_div(P, 128)) * (Ip / 128) * 512);
    L.total = off;
    return L;
}

namespace {

constexpr size_t kSmemLimit = 220 * 1024;

size_t route_smem(int T, int d, int E)
{
    const size_t sel = size_t(T) * E * 4 + 2 * 256 * 4;  // the last CTA: all logits, then the pair sort
    const size_t xs = size_t(T) * d * 2;
    return xs > sel ? xs : sel;
}
size_t gateup_smem(int T, int d) { return GateupSmem(d, T < G_PAIRS ? T : G_PAIRS).total; }
int down_rows_per_cta(int d) { return int(round_up(ceil_div(d, 152), 8)); }
size_t down_fixed_smem(int P, int I) { return size_t(P) * I * 2 + size_t(P) * (I / 32) * 4 + size_t(P) * 8; }
size_t down_pair_bytes(int d, int I)
{
    const int Ip = int(round_up(I, 128));
    const int rpc = down_rows_per_cta(d);
    return size_t(rpc) * (Ip / 2) + size_t(rpc) * (Ip / 128) * 4;
}
// pairs per weight buffer (two buffers)
int down_group(int P, int d, int I)
{
    const size_t fixed = down_fixed_smem(P, I);
    if (fixed >= kSmemLimit) return 0;
    const int g = int((kSmemLimit - fixed) / 2 / down_pair_bytes(d, I));
    return g < P ? g : P;
}
size_t down_smem(int P, int d, int I, int gp) { return down_fixed_smem(P, I) + 2 * size_t(gp) * down_pair_bytes(d, I); }

template <typename K>
cudaError_t smem_attr(K kernel, size_t bytes)
{
    return cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(bytes));
}

}  // namespace

bool small_path_fits(int T, int d, int E, int k, int I, int max_pairs)
{
    const int64_t P = int64_t(T) * k;
    if (T < 1 || P > max_pairs || P > SMALL_MAX_PAIRS || T > SMALL_MAX_TOKENS) return false;
    if (E > 2048 || d % 128 != 0 || d > 32 * 16 * MAX_CH || I % 32 != 0 || I > 1024) return false;
    if (down_rows_per_cta(d) > D_WARPS * D_RPW) return false;
    return route_smem(T, d, E) <= kSmemLimit && gateup_smem(T, d) <= kSmemLimit && down_group(int(P), d, I) >= 1;
}

namespace {

template <bool FP4>
cudaError_t launch_small_t(const uint16_t *x, const uint16_t *Wr3, const float *bias, const lmoe_expert_weights *W,
                           int T, int d, int E, int k, int I, float *logits, int32_t *idx, float *w, uint16_t *y,
                           const SmallPlan &sp, cudaStream_t st, const cudaEvent_t *stage_events)
{
    const int P = T * k;
    cudaError_t e = cudaSuccess;
    const size_t rs = route_smem(T, d, E);
    const int rgrid = int(ceil_div(2 * E, R_WARPS));
    if (T <= 1) {
        if ((e = smem_attr(k_small_route<1, FP4>, rs)) != cudaSuccess) return e;
        e = launch_pdl(k_small_route<1, FP4>, dim3(rgrid), dim3(32 * R_WARPS), rs, st, x, Wr3, bias, T, d, E, k,
                       logits, idx, w, sp);
    } else if (T <= 2) {
        if ((e = smem_attr(k_small_route<2, FP4>, rs)) != cudaSuccess) return e;
        e = launch_pdl(k_small_route<2, FP4>, dim3(rgrid), dim3(32 * R_WARPS), rs, st, x, Wr3, bias, T, d, E, k,
                       logits, idx, w, sp);
    } else if (T <= 4) {
        if ((e = smem_attr(k_small_route<4, FP4>, rs)) != cudaSuccess) return e;
        e = launch_pdl(k_small_route<4, FP4>, dim3(rgrid), dim3(32 * R_WARPS), rs, st, x, Wr3, bias, T, d, E, k,
                       logits, idx, w, sp);
    } else {
        if ((e = smem_attr(k_small_route<SMALL_MAX_TOKENS, FP4>, rs)) != cudaSuccess) return e;
        e = launch_pdl(k_small_route<SMALL_MAX_TOKENS, FP4>, dim3(rgrid), dim3(32 * R_WARPS), rs, st, x, Wr3, bias,
                       T, d, E, k, logits, idx, w, sp);
    }
    if (e != cudaSuccess) return e;
    // stage events 1..3 (routing, permute, activation rounding) all follow the routing kernel
    for (int i = 1; stage_events && i <= 3; ++i)
        if ((e = cudaEventRecord(stage_events[i], st)) != cudaSuccess) return e;
    const int npair_max = T < G_PAIRS ? T : G_PAIRS;
    const size_t gs = gateup_smem(T, d);
    if ((e = smem_attr(k_small_gateup<FP4>, gs)) != cudaSuccess) return e;
    const int max_units = P * (I / 32);
    const int ggrid = max_units < 152 ? max_units : 152;
    e = launch_pdl(k_small_gateup<FP4>, dim3(ggrid), dim3(32 * G_WARPS), gs, st, W->gate_q, W->gate_s, W->up_q,
                   W->up_s, T, d, I, k, npair_max, sp);
    if (e != cudaSuccess) return e;
    if (stage_events && (e = cudaEventRecord(stage_events[4], st)) != cudaSuccess) return e;
    const int gp = down_group(P, d, I);
    const size_t ds = down_smem(P, d, I, gp);
    if ((e = smem_attr(k_small_down<FP4>, ds)) != cudaSuccess) return e;
    const int rpc = down_rows_per_cta(d);
    const int dgrid = int(ceil_div(d, rpc));
    e = launch_pdl(k_small_down<FP4>, dim3(dgrid), dim3(32 * D_WARPS), ds, st, W->down_q, W->down_s, idx, w, T, d, I,
                   k, rpc, gp, y, sp);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_small_forward(const uint16_t *x, const uint16_t *Wr3, const float *bias, const lmoe_expert_weights *W,
                                 int T, int d, int E, int k, int I, int act, float *logits, int32_t *idx, float *w,
                                 uint16_t *y, const SmallLayout &L, char *scratch, int32_t *status, int32_t *counter,
                                 float *hcap, cudaStream_t st, const cudaEvent_t *stage_events)
{
    SmallPlan sp;
    sp.counter = counter;
    sp.status = status;
    sp.n_touched = reinterpret_cast<int32_t *>(scratch + L.n_touched);
    sp.seg_expert = reinterpret_cast<int32_t *>(scratch + L.seg_expert);
    sp.seg_start = reinterpret_cast<int32_t *>(scratch + L.seg_start);
    sp.seg_pair = reinterpret_cast<int32_t *>(scratch + L.seg_pair);
    sp.xq = reinterpret_cast<uint8_t *>(scratch + L.xq);
    sp.xs = reinterpret_cast<uint8_t *>(scratch + L.xs);
    sp.hq = reinterpret_cast<uint8_t *>(scratch + L.hq);
    sp.hs = reinterpret_cast<uint8_t *>(scratch + L.hs);
    sp.hcap = hcap;
    return act == LMOE_ACT_MXFP4
               ? launch_small_t<true>(x, Wr3, bias, W, T, d, E, k, I, logits, idx, w, y, sp, st, stage_events)
               : launch_small_t<false>(x, Wr3, bias, W, T, d, E, k, I, logits, idx, w, y, sp, st, stage_events);
}

}  // namespace lmoe
