// Expert FFN on the 5th-generation tensor cores: two grouped GEMMs over the
// experts, MXFP4 weights x MXFP8 activations with hardware block scaling
// (tcgen05.mma kind::mxf8f6f4, E8M0 scales), fp32 accumulation in TMEM.
//   [MX]  "SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section "MXFP4 原生支持":
//         one scale per 32-element block, dequantisation fused into the GEMM.
//   [L1]  "从Kimi K3到MiniMax-H3", section 二 first layer: 4-bit weights with
//         higher-precision activations and accumulation; section 一: gated
//         expert FFN in the latent space (SiLU gating assumed, K3's SiTU is
//         not defined on the pages).
//
// Orientation ("swap AB"): the weight rows are the M = 128 operand (A, e2m1,
// K-major) and the expert's tokens are the N operand (B, e4m3, K-major), so N
// follows the token count of the expert (16..NT in steps of 16) and small
// batches waste no tensor work on padding rows.
//
//   gate/up GEMM, item (expert e, 128 rows of I, token tile):
//     G = Wg[e] x^T, U = Wu[e] x^T (two TMEM accumulators), epilogue
//     h = silu(G) * U, MXFP8-quantised along I (a warp's 32 lanes are one
//     32-row block of I) -> hq / hs in the tiled token layout;
//   down GEMM, item (expert e, 128 or 256 rows of d, token tile):
//     Y = Wd[e] h^T, epilogue yp[q][row] = topk_w[perm[q]] * Y (fp32), or,
//     with the combine fused (large token tiles), yacc[perm[q] / k][row] +=
//     topk_w[perm[q]] * Y by fp32 vector atomics in L2 (the k terms of a
//     token are then summed in fp32 in an unspecified order).
//
// Token layout: the codes of the activations (x^ for gate/up, h^ for down)
// are one row per routed pair in permuted order: expert e's pairs occupy rows
// offsets[e] .. offsets[e+1]-1, and its token tile n is the NT rows from
// offsets[e] + n*NT (a partial last tile reads the next expert's rows, or the
// NT rows reserved past the end, as padding whose product columns are
// dropped).  Each tile's scale factors are a 512-byte atom per 128 columns
// (the tile's rows 0..NT-1 of a 128-row atom), which one bulk copy moves and
// one tcgen05.cp puts in TMEM; tiles are numbered per expert from
// pad_off[e] / NT, and a pair's "atom row" (tile * NT + row in tile) is its
// dst_row.
//
// Persistent, warp-specialised CTA (256 or 384 threads, one per SM):
//   warp 0     TMA producer 0 (first A tile via the packed-FP4 tensor map that
//              expands 16 x 4-bit into 16-byte smem units, its scale atom, the
//              B tile)
//   warp 1     TMEM allocator + MMA issuer 0 (gate / first weight tile of down)
//   warps 2..  epilogue, 4 or 8 warps: TMEM lane quarter = warp % 4; with 8,
//              two warps per quarter take alternate column chunks
//   next warp  MMA issuer 1 (up / second weight tile of down)
//   last warp  TMA producer 1 (second A tile, its scale atom, B scale atoms)
// Every mbarrier wait is bounded; a wait that runs out records
// LMOE_ERR_TIMEOUT in the status word and the CTA winds down.
#include <cuda.h>

#include "lmoe_internal.cuh"
#include "tc_ptx.cuh"

#ifdef LMOE_TRACE
// Diagnostic build only: CTA 0 of each expert GEMM records (tag, item, k chunk,
// SM clock) at its pipeline events into shared memory (one region per role,
// plain stores), copied to global memory when the CTA ends;
// lmoe_debug_trace() returns them.
constexpr int TRACE_PER_ROLE = 500;
__device__ uint32_t g_lmoe_trace[2 * 65536];
__device__ uint32_t g_lmoe_trace_n;
#define LMOE_TRACE_DECL uint32_t tr_n_ = 0;
#define LMOE_TRACE_EV(role, tag, item, kc)                                                                   \
    do {                                                                                                    \
        if (blockIdx.x == 0 && tr_n_ < TRACE_PER_ROLE) {                                                    \
            s_trace[2 * ((role) * TRACE_PER_ROLE + tr_n_)] =                                                \
                (uint32_t(tag) << 24) | ((uint32_t(item) & 0xFFFF) << 8) | (uint32_t(kc) & 0xFF);           \
            s_trace[2 * ((role) * TRACE_PER_ROLE + tr_n_) + 1] = uint32_t(clock64());                       \
            ++tr_n_;                                                                                        \
        }                                                                                                   \
    } while (0)
#define LMOE_TRACE_END(role)                                                                                \
    do {                                                                                                    \
        if (blockIdx.x == 0 && tr_n_) {                                                                     \
            const uint32_t base_ = atomicAdd(&g_lmoe_trace_n, tr_n_);                                       \
            for (uint32_t i_ = 0; i_ < tr_n_ && base_ + i_ < 65536; ++i_) {                                 \
                g_lmoe_trace[2 * (base_ + i_)] = s_trace[2 * ((role) * TRACE_PER_ROLE + i_)];               \
                g_lmoe_trace[2 * (base_ + i_) + 1] = s_trace[2 * ((role) * TRACE_PER_ROLE + i_) + 1];       \
            }                                                                                               \
        }                                                                                                   \
    } while (0)
__shared__ uint32_t s_trace[2 * 3 * TRACE_PER_ROLE];
// Every CTA's start and end (%globaltimer, ns) per GEMM mode (gate/up, down, fused): [mode][cta][2].
__device__ unsigned long long g_lmoe_cta_ns[3][1024][2];
__device__ __forceinline__ unsigned long long lmoe_globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}
#define LMOE_TRACE_CTA(mode, which) \
    do {                            \
        if (threadIdx.x == 0 && blockIdx.x < 1024) g_lmoe_cta_ns[mode][blockIdx.x][which] = lmoe_globaltimer(); \
    } while (0)
extern "C" int lmoe_debug_cta_times(unsigned long long *host)
{
    return cudaMemcpyFromSymbol(host, g_lmoe_cta_ns, sizeof(g_lmoe_cta_ns)) == cudaSuccess ? 0 : -1;
}
extern "C" int lmoe_debug_trace(uint32_t *host, int max_events)
{
    uint32_t n = 0;
    if (cudaMemcpyFromSymbol(&n, g_lmoe_trace_n, sizeof(n)) != cudaSuccess) return -1;
    if (n > 65536) n = 65536;
    if (int(n) > max_events) n = uint32_t(max_events);
    if (n && cudaMemcpyFromSymbol(host, g_lmoe_trace, size_t(n) * 8) != cudaSuccess) return -1;
    const uint32_t zero = 0;
    cudaMemcpyToSymbol(g_lmoe_trace_n, &zero, sizeof(zero));
    return int(n);
}
#else
#define LMOE_TRACE_DECL
#define LMOE_TRACE_EV(role, tag, item, kc) \
    do {                                   \
    } while (0)
#define LMOE_TRACE_END(role) \
    do {                     \
    } while (0)
#define LMOE_TRACE_CTA(mode, which) \
    do {                            \
    } while (0)
#endif

namespace lmoe {
namespace {

using namespace tc;

// Four consecutive fp32 adds to global memory as one vector reduction that
// returns nothing (the issuing thread never waits for it); 16-byte aligned;
// `policy` is the L2 cache policy of the line.
__device__ __forceinline__ void red_add_v4(float *dst, float4 v, uint64_t policy)
{
    asm volatile("red.global.add.L2::cache_hint.v4.f32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(dst), "f"(v.x), "f"(v.y),
                 "f"(v.z), "f"(v.w), "l"(policy)
                 : "memory");
}

// FUSED: one persistent kernel runs the gate/up items and then the down
// items; a down item's h loads wait until every gate/up item of its token
// tile has stored h (a per-tile counter), so CTAs done with gate/up start on
// down items instead of idling through the gate/up tail and a kernel boundary.
enum { GATEUP = 0, DOWN = 1, FUSED = 2 };

// fp32 accumulators of one split-K gate/up half: 4 epilogue warps x 2
// matrices x 16 token columns x 32 rows
constexpr size_t kKsplitHalfBytes = size_t(4) * 2 * 16 * 32 * 4;

struct GemmArgs {
    const uint8_t *sfa0, *sfa1;  // weight scale atoms [E][RTa][KC][512]
    const uint8_t *sfb;          // activation scale atoms [rows/128][KC][512]
    const int32_t *offsets;      // [E+1] segment starts in permuted order
    const int32_t *tiles;        // [E+1] first work item of each expert (tiles[E]: the item count)
    const int32_t *pad_off;      // [E+1] first token row of each expert (tiled layout)
    const int2 *items;           // work-item table in execution order (fill_item_entries)
    const float *w_sorted;  // gate weight of each permuted row q (topk_w[perm[q]])
    uint8_t *hq;    // gate/up out: [rows][Ih] e4m3
    uint8_t *hs;    // gate/up out: scale atoms [rows/128][KCh][512]
    float *hcap;    // gate/up, diagnostics only (normally null): every fp32 h before its MXFP8 rounding, [rows][Ih]
    float *yp;      // down out: [P][Mtot]
    float *yacc;    // down out when set (fused combine): [T][Mtot] fp32 sums, zeroed before the kernel (by the gate/up kernel)
    const int32_t *perm;  // [P] pair of each permuted row (token = perm / k)
    int k;
    int E, Mtot, MTA, KC, KCh, Ih;  // MTA: 128-row tiles of A
    int stages;  // shared-memory pipeline depth (<= Cfg::MAX_STAGES)
    int32_t *status;
    long long wait_limit;  // SM clocks a bounded wait may take before it gives up
    int stall_first_fill;  // failure-path test only: producer 0 withholds each CTA's first stage
    int32_t *tile_done;    // fused kernel: per token tile, epilogue warps done storing h (zeroed by the schedule)
    // fused kernel at 16-token tiles, gate/up items split in two K halves:
    // each half's fp32 accumulators (kKsplitHalfBytes per item and half) and
    // per item and epilogue warp the halves done (zeroed by the schedule); null: no split
    float *kpart;
    int32_t *kcnt;
    // gate/up kernel: a buffer its epilogue warps zero between items (the down
    // GEMM's fused-combine sums), n4 16-byte units; null: none
    float4 *zero;
    int64_t zero_n4;
};

template <int MODE, int NT>
struct Cfg {
    // Weight tiles per stage: gate and up rows of the same 128 features; for
    // down, two consecutive 128-row tiles sharing the stage's token tile (more
    // weight bytes per stage, half the h traffic) up to 96-token tiles, one
    // tile beyond (so the accumulators still fit twice in TMEM).
    static constexpr int MATS = (MODE == GATEUP || NT <= 96) ? 2 : 1;
    static constexpr int SLOT = NT;  // rows a token tile occupies (tiles are packed)
    static constexpr int NAT = (NT + 127) / 128;  // B scale atoms per stage
    static constexpr uint32_t A_TILE = 128 * 128;  // smem bytes of one expanded FP4 A tile
    static constexpr uint32_t B_TILE = NT * 128;
    static constexpr uint32_t SFA_OFF = MATS * A_TILE + B_TILE;
    static constexpr uint32_t SFB_OFF = SFA_OFF + MATS * 512;
    static constexpr uint32_t STAGE_BYTES = (SFB_OFF + NAT * 512 + 1023) / 1024 * 1024;
    // global bytes per stage: packed FP4 tiles count 64 bytes per 128-element row.
    // Two producer threads share a stage's copies (one thread issues an async
    // copy only every ~80 cycles): producer 0 the first weight tile, its scale
    // atom and the token tile; producer 1 the second weight tile, its scales
    // and the token scale atoms.
    static constexpr uint32_t TX_BYTES0 = 128 * 64 + 512 + B_TILE;
    static constexpr uint32_t TX_BYTES1 = (MATS - 1) * (128 * 64 + 512) + NAT * 512;
    // One MMA-issuing thread per weight tile, each with its own accumulator.
    // One thread issues a tcgen05 instruction only every few dozen cycles, so
    // two issuers keep small-N MMAs from pacing the pipeline.
    static constexpr int ACC_COLS_ITEM = MATS * NT;
    static constexpr int SF_COLS_ISSUER = 4 + 4 * NAT;  // this issuer's SFA and SFB copies
    static constexpr int SF_COLS = MATS * SF_COLS_ISSUER;
    // accumulator stages: double-buffered (the epilogue of one item overlaps
    // the next item's MMAs) whenever two items and 4 stages of scale factors
    // fit the 512 TMEM columns
    static constexpr int ACC_STAGES =
        (ACC_COLS_ITEM <= 64) ? 4 : (2 * ACC_COLS_ITEM + 4 * SF_COLS <= 512 ? 2 : 1);
    static constexpr int ACC_COLS = ACC_STAGES * ACC_COLS_ITEM;
    static constexpr int SF_BASE = (ACC_COLS + 31) / 32 * 32;
    static constexpr int MAX_STAGES = (512 - SF_BASE) / SF_COLS < 16 ? (512 - SF_BASE) / SF_COLS : 16;
    static_assert(MAX_STAGES >= 2, "TMEM columns");
    // Epilogue.  Large token tiles: 8 warps (two per TMEM lane quarter, on
    // alternate column chunks) that transpose each chunk through a per-warp
    // shared-memory tile (down: CW tokens x 32 fp32, 36-float row stride;
    // gate/up: 16 tokens x 32 e4m3 codes) so that every lane stores 16
    // contiguous bytes.  Small tiles (decode): 4 warps storing straight from
    // registers, leaving the shared memory to the pipeline stages.
    static constexpr bool STAGED = NT >= 64;
    static constexpr int EPI_WARPS = STAGED ? 8 : 4;
    static constexpr int NW = EPI_WARPS / 4;  // epilogue warps per lane quarter
    static constexpr int THREADS = 32 * (4 + EPI_WARPS);
    static constexpr int CW = NT < 32 ? NT : 32;  // accumulator columns per TMEM load (down)
    static constexpr int STG_STRIDE = 36;
    static constexpr uint32_t EPI_WARP_BYTES = !STAGED ? 0 : (MODE != GATEUP ? CW * STG_STRIDE * 4 : 16 * 32);
    static_assert(MODE != FUSED || MATS == 2, "the fused kernel needs the same stage layout for both GEMMs");
    // gate/up items in two K halves (small batches): one 16-column chunk per epilogue warp
    static constexpr bool KSPLIT = MODE == FUSED && NT == 16;
    static_assert(!KSPLIT || (NW == 1 && !STAGED), "split-K epilogue layout");
    static constexpr uint32_t EPI_BYTES = EPI_WARPS * EPI_WARP_BYTES;
};

struct Item {
    int e, n_tile, m_tile, n_valid;
};

// Work-item table entry -> (expert, token tile, weight tile, valid tokens).
// The table (written with the schedule) fixes the execution order: weight
// tile fastest within a token tile, so the weight-tile items of one token
// tile run together and share its activation rows in L2; for the down GEMM
// with large token tiles (the fused combine), the first half of the weight
// tiles of every token tile before the second half.  Each role loads its
// entries an item or two ahead (a table load is a global-memory round trip;
// a search of the per-expert prefix in shared memory took ~1,400 cycles).
__device__ __forceinline__ Item item_at(int2 v, const int32_t *s_off, int nt)
{
    Item r;
    r.e = v.x & 0xFFFF;
    r.m_tile = int(uint32_t(v.x) >> 16);
    r.n_tile = v.y;
    r.n_valid = min(nt, s_off[r.e + 1] - s_off[r.e] - r.n_tile * nt);
    return r;
}

template <int MODE, int NT, bool SPLIT = false>
__global__ void __launch_bounds__(Cfg<MODE, NT>::THREADS, 1)
    k_moe_gemm(const __grid_constant__ CUtensorMap tmA0, const __grid_constant__ CUtensorMap tmA1,
               const __grid_constant__ CUtensorMap tmB, const __grid_constant__ CUtensorMap tmD,
               const __grid_constant__ CUtensorMap tmH, const GemmArgs p, const GemmArgs q)
{
    // p: the kernel's GEMM (the gate/up GEMM in the fused kernel), q: the
    // fused kernel's down GEMM (tmD: its weights, tmH: h); unused otherwise
    using C = Cfg<MODE, NT>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int S = p.stages;
    uint8_t *stages = smem;
    uint8_t *epi_stage = stages + S * C::STAGE_BYTES;
    uint64_t *full = reinterpret_cast<uint64_t *>(epi_stage + C::EPI_BYTES);
    uint64_t *empty = full + S;
    uint64_t *acc_full = empty + S;
    uint64_t *acc_empty = acc_full + C::ACC_STAGES;
    uint64_t *drain = acc_empty + C::ACC_STAGES;  // per MMA issuer: its MMAs done (after a timeout)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 2);
    int32_t *s_pad = reinterpret_cast<int32_t *>(tmem_slot + 4);
    int32_t *s_off = s_pad + (p.E + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    LMOE_TRACE_CTA(MODE, 0);
    // the schedule is an output of an earlier kernel than the previous one
    // (complete before this grid starts); read through L2
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
        s_pad[i] = __ldcg(p.pad_off + i);
        s_off[i] = __ldcg(p.offsets + i);
    }
    const int G = int(gridDim.x);
    // Small batches, whose gate/up items fit in half the CTAs: each gate/up
    // item runs as two K halves on two CTAs (items [0, n_gu_tab) the first
    // halves, [n_gu_tab, 2 n_gu_tab) the second).  One SM streams an item's
    // weights only as fast as its ring's bytes in flight allow, so two SMs
    // per item halve that phase; each half stores its fp32 accumulators and
    // the later of the two forms h from their sum.
    const int n_gu_tab = MODE == FUSED ? __ldcg(p.tiles + p.E) : 0;
    constexpr bool KSPLIT = SPLIT && C::KSPLIT;  // a separate instance: the other batches' code is unchanged
    const int KS = (KSPLIT && p.kpart && p.kcnt && n_gu_tab > 0 && 2 * n_gu_tab <= G &&
                    n_gu_tab <= KSPLIT_MAX_ITEMS && p.KC >= 2)
                       ? 2
                       : 1;
    // fused: gate/up items [0, n_gu), then down items [n_gu, total)
    const int n_gu = KS * n_gu_tab;
    const int total = MODE == FUSED ? n_gu + __ldcg(q.tiles + q.E) : __ldcg(p.tiles + p.E);
    // this CTA's item-table entries at index i (clamped: entries past the end
    // are loaded but never used); the table may come from the previous kernel
    auto entry = [&](int i) {
        const int j = i < total ? i : total - 1;
        if (MODE == FUSED && j >= n_gu) return __ldcg(q.items + (j - n_gu));
        return __ldcg(p.items + (KS == 2 && j >= n_gu_tab ? j - n_gu_tab : j));
    };
    // the K chunks [k0, k1) item it accumulates (of KCf)
    auto krange = [&](int it, int KCf, int &k0, int &k1) {
        const bool second = KS == 2 && it < n_gu && it >= n_gu_tab;
        k0 = KS == 2 && it < n_gu ? (second ? KCf / 2 : 0) : 0;
        k1 = KS == 2 && it < n_gu && !second ? KCf / 2 : KCf;
    };
    auto mode_of = [&](int i) { return MODE == FUSED ? (i < n_gu ? int(GATEUP) : int(DOWN)) : int(MODE); };
    // This CTA's items in order: ordinal i -> item index.  One GEMM: every
    // G-th item.  Fused: the gate/up items every G-th, then the down items in
    // rounds over the CTAs (consecutive items, adjacent weight rows, run at
    // the same time on neighbouring CTAs), where the first X rounds leave out
    // the r CTAs that drew an extra gate/up item (r = n_gu mod G; X down
    // items take about the pipeline stages of one gate/up item), so that
    // those CTAs do not finish last.
    const int c = int(blockIdx.x);
    const int gu_c = MODE == FUSED ? (n_gu > c ? (n_gu - c + G - 1) / G : 0) : 0;
    const int n_dn = total - n_gu;
    const int r_gu = n_gu % G;
    const int X = (MODE == FUSED && r_gu > 0 && KS == 1) ? (p.KC + q.KC / 2) / q.KC : 0;
    int dn_c = 0;  // this CTA's down items
    if (MODE == FUSED) {
        if (c >= r_gu)
            for (int k = 0; k < X && k * (G - r_gu) + (c - r_gu) < n_dn; ++k) ++dn_c;
        const int base = X * (G - r_gu) + c;
        if (n_dn > base) dn_c += (n_dn - base + G - 1) / G;
    }
    // h of a token tile is complete once every epilogue warp of each of its
    // gate/up items has counted itself in
    [[maybe_unused]] const int h_ready = p.MTA * C::EPI_WARPS;
    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 2);  // one expect_tx arrival per producer
            mbar_init(&empty[s], C::MATS);  // one commit per MMA issuer
        }
        for (int a = 0; a < C::ACC_STAGES; ++a) {
            mbar_init(&acc_full[a], C::MATS);
            mbar_init(&acc_empty[a], 32 * C::EPI_WARPS);
        }
        mbar_init(&drain[0], 1);
        mbar_init(&drain[1], 1);
        mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA0);
        if (C::MATS == 2) prefetch_tensormap(&tmA1);
        prefetch_tensormap(&tmB);
        if (MODE == FUSED) {
            prefetch_tensormap(&tmD);
            prefetch_tensormap(&tmH);
        }
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    auto slot_row = [&](int e) { return s_pad[e]; };  // first token row of expert e
    const int n_mine = MODE == FUSED ? gu_c + dn_c : (total > c ? (total - c + G - 1) / G : 0);
    auto seq = [&](int i) {
        if (MODE != FUSED || i < gu_c) return c + i * G;
        const int j = i - gu_c;
        if (c >= r_gu && j < X) return n_gu + j * (G - r_gu) + (c - r_gu);
        return n_gu + X * (G - r_gu) + (j - (c >= r_gu ? X : 0)) * G + c;
    };
    // Everything above reads only inputs of earlier kernels; the previous
    // kernel's outputs are read after this wait.
    pdl_enter();
    int2 ent0 = make_int2(0, 0), ent1 = make_int2(0, 0);  // the first two entries
    if (n_mine > 0) {
        ent0 = entry(seq(0));
        ent1 = entry(seq(1));
    }

    if (warp == 0 || warp == 3 + C::EPI_WARPS) {
        // ---------------- TMA producers (warp 0 and the last warp) ----------------
        if (lane == 0) {
            const int pr = warp == 0 ? 0 : 1;
            LMOE_TRACE_DECL
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            int2 ent = ent0, ent_next = ent1;
            for (int i = 0; i < n_mine && ok; ++i) {
                const int it = seq(i);
                const Item w = item_at(ent, s_off, NT);
                ent = ent_next;
                ent_next = entry(seq(i + 2));
                const int mode = mode_of(it);
                const GemmArgs &a = (MODE == FUSED && mode == DOWN) ? q : p;
                const int R = slot_row(w.e) + w.n_tile * C::SLOT;  // the tile's atom row (scale factors)
                const int Rc = s_off[w.e] + w.n_tile * NT;         // its first code row (permuted order)
                // gate/up: tile m of both matrices; down: tiles 2m and 2m+1 (an odd
                // last tile loads tile 2m twice and the epilogue drops the copy)
                const int mt0 = mode == GATEUP ? w.m_tile : C::MATS * w.m_tile;
                const int mt1 = mode == GATEUP ? w.m_tile : (mt0 + 1 < a.MTA ? mt0 + 1 : mt0);
                const int arow = w.e * a.Mtot + (pr == 0 ? mt0 : mt1) * 128;
                const int64_t sfa_base = (int64_t(w.e) * a.MTA + (pr == 0 ? mt0 : mt1)) * a.KC;
                const CUtensorMap *tmA = (MODE == FUSED && mode == DOWN) ? &tmD : (pr == 0 ? &tmA0 : &tmA1);
                const CUtensorMap *tmBx = (MODE == FUSED && mode == DOWN) ? &tmH : &tmB;
                const uint8_t *sfa = pr == 0 ? a.sfa0 : a.sfa1;
                bool h_waited = !(MODE == FUSED && mode == DOWN);
                int k0, k1;
                krange(it, a.KC, k0, k1);
                for (int kc = k0; kc < k1; ++kc) {
                    if (!mbar_wait(&empty[stage], phase ^ 1, p.wait_limit)) {
                        set_status(p.status, LMOE_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    if (pr == 0) LMOE_TRACE_EV(0, 0x10 | MODE, it, kc);  // producer: stage free
                    uint8_t *sb = stages + stage * C::STAGE_BYTES;
                    if (pr == 0 && p.stall_first_fill && it == int(blockIdx.x) && kc == k0) {
                        // failure-path test: this stage never fills, so every wait on it runs out
                    } else if (pr == 0) {
                        mbar_arrive_expect_tx(&full[stage], C::TX_BYTES0);
                        tma_load_2d(sb, tmA, kc * 128, arow, &full[stage]);
                        bulk_load(sb + C::SFA_OFF, sfa + (sfa_base + kc) * 512, 512, &full[stage]);
                        if (!h_waited) {
                            // fused down item: the weights are on their way; h of
                            // this token tile must be complete before it is read
                            h_waited = wait_count(a.tile_done + R / NT, h_ready, p.wait_limit);
                            if (!h_waited) {
                                set_status(p.status, LMOE_ERR_TIMEOUT);
                                ok = false;
                                break;
                            }
                        }
                        tma_load_2d(sb + C::MATS * C::A_TILE, tmBx, kc * 128, Rc, &full[stage]);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], C::TX_BYTES1);
                        if (C::MATS == 2) {
                            tma_load_2d(sb + C::A_TILE, tmA, kc * 128, arow, &full[stage]);
                            bulk_load(sb + C::SFA_OFF + 512, sfa + (sfa_base + kc) * 512, 512, &full[stage]);
                        }
                        if (!h_waited) {
                            h_waited = wait_count(a.tile_done + R / NT, h_ready, p.wait_limit);
                            if (!h_waited) {
                                set_status(p.status, LMOE_ERR_TIMEOUT);
                                ok = false;
                                break;
                            }
                        }
#pragma unroll
                        for (int a2 = 0; a2 < C::NAT; ++a2)
                            bulk_load(sb + C::SFB_OFF + a2 * 512, a.sfb + (int64_t(R / NT + a2) * a.KC + kc) * 512, 512,
                                      &full[stage]);
                    }
                    if (pr == 0) LMOE_TRACE_EV(0, 0x70 | MODE, it, kc);  // producer: copies issued
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (pr == 0) LMOE_TRACE_END(0);
        }
    } else if (warp == 1 || warp == 2 + C::EPI_WARPS) {
        // ---------------- MMA issuers (warp 1: gate / first tile, last warp: up / second tile) ----------------
        if (lane == 0 && (warp == 1 || C::MATS == 2)) {
            LMOE_TRACE_DECL
            const int iss = warp == 1 ? 0 : 1;
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            int2 ent = ent0, ent_next = ent1;
            for (int i = 0; i < n_mine && ok; ++i) {
                const int it = seq(i);
                const Item w = item_at(ent, s_off, NT);
                ent = ent_next;
                ent_next = entry(seq(i + 2));
                int k0, k1;
                krange(it, (MODE == FUSED && mode_of(it) == DOWN) ? q.KC : p.KC, k0, k1);
                const uint32_t N = uint32_t((w.n_valid + 15) & ~15);
                if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1, p.wait_limit)) {
                    set_status(p.status, LMOE_ERR_TIMEOUT);
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (iss == 0) LMOE_TRACE_EV(1, 0x20 | MODE, it, 0);  // mma: accumulator free
                const uint32_t d = tmem + uint32_t(acc * C::ACC_COLS_ITEM + iss * NT);
                for (int kc = k0; kc < k1; ++kc) {
                    if (!mbar_wait(&full[stage], phase, p.wait_limit)) {
                        set_status(p.status, LMOE_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (iss == 0) LMOE_TRACE_EV(1, 0x30 | MODE, it, kc);  // mma: stage data landed
                    const uint8_t *sb = stages + stage * C::STAGE_BYTES;
                    const uint32_t sfa = tmem + uint32_t(C::SF_BASE + stage * C::SF_COLS + iss * C::SF_COLS_ISSUER);
                    const uint32_t sfb = sfa + 4;
                    tc_cp_sf(sfa, sdesc_sf(smem_u32(sb + C::SFA_OFF + iss * 512)));
#pragma unroll
                    for (int a = 0; a < C::NAT; ++a) tc_cp_sf(sfb + 4 * a, sdesc_sf(smem_u32(sb + C::SFB_OFF + a * 512)));
                    const uint64_t ad = sdesc_k128(smem_u32(sb + iss * C::A_TILE));
                    const uint64_t bd = sdesc_k128(smem_u32(sb + C::MATS * C::A_TILE));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_mxf8f6f4(d, ad + 2 * kk, bd + 2 * kk, idesc_mxf4_e4m3(N, uint32_t(kk)), sfa, sfb,
                                     (kc > k0 || kk > 0) ? 1u : 0u);
                    tc_commit(&empty[stage]);
                    if (iss == 0) LMOE_TRACE_EV(1, 0x80 | MODE, it, kc);  // mma: stage issued
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(&acc_full[acc]);
                if (++acc == C::ACC_STAGES) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (!ok) {
                // after a timeout: let this issuer's MMAs already in flight finish
                // (bounded) before the tensor memory is freed
                tc_commit(&drain[iss]);
                mbar_wait(&drain[iss], 0, p.wait_limit);
            }
            if (iss == 0) LMOE_TRACE_END(1);
        }
    } else {
        // ---------------- epilogue (warps 2 .. 1 + EPI_WARPS) ----------------
        const int lq = warp & 3;            // TMEM lane quarter of this warp
        const int half = (warp - 2) >> 2;   // which of the quarter's NW warps
        // the fused combine's per-token fp32 rows take every pair's reduction:
        // keep them in L2 in preference to the streamed weights
        [[maybe_unused]] const uint64_t keep_policy = l2_policy_evict_last();
        [[maybe_unused]] uint8_t *stg = epi_stage + (warp - 2) * C::EPI_WARP_BYTES;
        LMOE_TRACE_DECL
        int acc = 0;
        uint32_t acc_phase = 0;
        // The gate weights and tokens of an item are loaded two items ahead
        // (their latency under the output traffic is several microseconds),
        // into two register sets used alternately, so no register waits on an
        // outstanding load before its item comes up; the item's table entry
        // was loaded two items before that.
        constexpr int NV = (NT + 31) / 32;
        // the down GEMM's arguments (the fused kernel's second GEMM)
        const GemmArgs &dn = MODE == FUSED ? q : p;
        auto fetch = [&](int i, int2 ent, Item &nx, float (&wn)[NV], int (&tn)[NV]) {
            nx = item_at(ent, s_off, NT);
            if (mode_of(i) == DOWN) {
                // Unconditional loads at clamped rows (entries past the tile are
                // never used) of raw pair ids: a select or a division here would
                // wait for the load.
                const int qb = s_off[nx.e] + nx.n_tile * NT;
                const int qlast = s_off[p.E] - 1;
#pragma unroll
                for (int i = 0; i < NV; ++i) {
                    const int qq = min(qb + 32 * i + lane, qlast);
                    wn[i] = __ldg(dn.w_sorted + qq);
                    tn[i] = __ldg(dn.perm + qq);
                }
            }
        };
        auto process = [&](int it, const Item &w, const float (&wl)[NV], const int (&tl)[NV]) -> bool {
            const int mode = mode_of(it);
            [[maybe_unused]] const int qbase = s_off[w.e] + w.n_tile * NT;  // first permuted row of the tile (down)
            if (threadIdx.x == 64) LMOE_TRACE_EV(2, 0x40 | MODE, it, 0);  // epilogue: waiting
            if (!mbar_wait(&acc_full[acc], acc_phase, p.wait_limit)) {
                set_status(p.status, LMOE_ERR_TIMEOUT);
                return false;
            }
            tc_fence_after();
            if (threadIdx.x == 64) LMOE_TRACE_EV(2, 0x50 | MODE, it, 0);  // epilogue: accumulator ready
            const uint32_t tbase = tmem + (uint32_t(32 * lq) << 16) + uint32_t(acc * C::ACC_COLS_ITEM);
            // split-K half: which half, and the gate/up item it belongs to
            const int kh = (KS == 2 && mode == GATEUP && it >= n_gu_tab) ? 1 : 0;
            const int kj = it - kh * n_gu_tab;
            bool count_h = KS == 1 || kh == 1;  // this warp counts its part of h in (rows past I: the second half)
            if (mode == GATEUP && w.m_tile * 128 + 32 * lq < p.Mtot) {
                const int row0 = w.m_tile * 128 + 32 * lq;  // first row of I held by this warp
                const int blk = row0 / 32;                 // MX block of I held by this warp
                const int64_t Rbase = int64_t(slot_row(w.e)) + int64_t(w.n_tile) * C::SLOT;  // atom rows
                const int64_t Cbase = int64_t(s_off[w.e]) + int64_t(w.n_tile) * NT;           // code rows
                for (int c0 = 16 * half; c0 < w.n_valid; c0 += 16 * C::NW) {
                    uint32_t v0[16], v1[16];
                    tmem_ld16(tbase + c0, v0);
                    tmem_ld16(tbase + NT + c0, v1);
                    tmem_ld_wait();
                    if constexpr (KSPLIT) {
                        if (KS == 2) {
                            // store this half's sums, count in; the later half adds the other's
                            constexpr int HW = 2 * 16 * 32;  // floats per warp and half
                            float *mine = p.kpart + ((int64_t(kj) * 2 + kh) * 4 + lq) * HW;
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                mine[j * 32 + lane] = __uint_as_float(v0[j]);
                                mine[(16 + j) * 32 + lane] = __uint_as_float(v1[j]);
                            }
                            __threadfence();
                            __syncwarp();
                            int first = 0;
                            if (lane == 0) first = atomicAdd(p.kcnt + kj * 4 + lq, 1) == 0;
                            first = __shfl_sync(0xFFFFFFFFu, first, 0);
                            count_h = !first;
                            if (first) break;
                            __threadfence();
                            const float *other = p.kpart + ((int64_t(kj) * 2 + (1 - kh)) * 4 + lq) * HW;
                            float o0[16], o1[16];
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                o0[j] = __ldcg(other + j * 32 + lane);
                                o1[j] = __ldcg(other + (16 + j) * 32 + lane);
                            }
                            // first half + second half, the same sum whichever finishes last
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                const float a0 = __uint_as_float(v0[j]), a1 = __uint_as_float(v1[j]);
                                v0[j] = __float_as_uint(kh ? o0[j] + a0 : a0 + o0[j]);
                                v1[j] = __float_as_uint(kh ? o1[j] + a1 : a1 + o1[j]);
                            }
                        }
                    }
                    // 16 independent columns: SiLU-gated product, block amax over
                    // the warp's 32 rows of I, E8M0 scale, e4m3 code
                    uint32_t sbv[16], code[16];
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const float gv = __uint_as_float(v0[j]), uv = __uint_as_float(v1[j]);
                        const float h = __fdividef(gv, 1.f + __expf(-gv)) * uv;
                        if (p.hcap && c0 + j < w.n_valid) p.hcap[(Cbase + c0 + j) * p.Ih + row0 + lane] = h;
                        uint32_t amax;
                        asm("redux.sync.max.u32 %0, %1, 0xffffffff;" : "=r"(amax) : "r"(__float_as_uint(h) & 0x7FFFFFFFu));
                        sbv[j] = mx_scale_byte(__uint_as_float(amax), 8);
                        code[j] = e4m3x2(h * mx_inv_scale(sbv[j]), 0.f) & 0xFF;
                    }
                    if constexpr (C::STAGED) {
                        __syncwarp();  // the previous chunk's staged codes have been read
#pragma unroll
                        for (int j = 0; j < 16; ++j) stg[j * 32 + lane] = uint8_t(code[j]);
                        __syncwarp();
                        // lane l stores 16 codes of token column l/2 (rows 16*(l&1) ..)
                        const int c = lane >> 1;
                        if (c0 + c < w.n_valid)
                            *reinterpret_cast<uint4 *>(p.hq + (Cbase + c0 + c) * p.Ih + row0 + 16 * (lane & 1)) =
                                *reinterpret_cast<const uint4 *>(stg + 16 * lane);
                    } else {
                        uint8_t *hrow = p.hq + (Cbase + c0) * p.Ih + row0 + lane;
#pragma unroll
                        for (int j = 0; j < 16; ++j)
                            if (c0 + j < w.n_valid) hrow[int64_t(j) * p.Ih] = uint8_t(code[j]);
                    }
                    if (c0 + lane < w.n_valid && lane < 16) {  // lane j writes column j's scale byte
                        uint32_t sbl = 0;
#pragma unroll
                        for (int j = 0; j < 16; ++j) sbl = (lane == j) ? sbv[j] : sbl;
                        const int64_t R = Rbase + c0 + lane;
                        p.hs[tile_atom_off(R, blk, p.KCh, NT)] = uint8_t(sbl);
                    }
                }
            }
            if (MODE == FUSED && mode == GATEUP && count_h) {
                // this warp's part of h for the token tile is stored: count it
                // in (release), for the down items that read the tile's h
                __threadfence();
                asm volatile("fence.proxy.async.global;" ::: "memory");
                __syncwarp();
                if (lane == 0) atomicAdd(p.tile_done + (slot_row(w.e) / NT + w.n_tile), 1);
            }
            if (mode == DOWN) {
                // accumulator h holds output rows (MATS m + h) * 128 + 32q + lane;
                // work units (h, column chunk) alternate between the quarter's NW warps
                constexpr int CW = C::CW;
                [[maybe_unused]] float *sf = reinterpret_cast<float *>(stg);
                const int nch = (w.n_valid + CW - 1) / CW;
                for (int u = half; u < C::MATS * nch; u += C::NW) {
                    const int h = u / nch, c0 = (u - h * nch) * CW;
                    const int mt = C::MATS * w.m_tile + h;
                    if (mt >= dn.MTA) continue;  // odd last tile: second accumulator is a copy
                    uint32_t v[CW];
                    tmem_ld_cols<CW>(tbase + h * NT + c0, v);
                    tmem_ld_wait();
                    // gate weights of this chunk's columns: column c's weight is lane (c0 & 31) + c of wl[c0 / 32]
                    float wsel = wl[0];
                    int tsel = tl[0];
#pragma unroll
                    for (int i = 1; i < (NT + 31) / 32; ++i) {
                        wsel = (c0 / 32 == i) ? wl[i] : wsel;
                        tsel = (c0 / 32 == i) ? tl[i] : tsel;
                    }
                    tsel /= dn.k;  // pair -> token
                    if constexpr (C::STAGED) {
                        // transpose through shared memory: sf[c][row], row stride STG_STRIDE
                        __syncwarp();
#pragma unroll
                        for (int j = 0; j < CW; ++j) sf[j * C::STG_STRIDE + lane] = __uint_as_float(v[j]);
                        __syncwarp();
                        // lane l: token column c = 4 pp + l / 8, 4 rows starting at 4 (l % 8)
                        const int f4 = 4 * (lane & 7);
                        const int col = mt * 128 + 32 * lq + f4;
#pragma unroll
                        for (int pp = 0; pp < CW / 4; ++pp) {
                            const int c = 4 * pp + (lane >> 3);
                            const float wc = __shfl_sync(0xFFFFFFFFu, wsel, (c0 & 31) + c);
                            const int tc = __shfl_sync(0xFFFFFFFFu, tsel, (c0 & 31) + c);
                            if (c0 + c < w.n_valid) {
                                float4 a = *reinterpret_cast<const float4 *>(sf + c * C::STG_STRIDE + f4);
                                a.x *= wc;
                                a.y *= wc;
                                a.z *= wc;
                                a.w *= wc;
                                if (dn.yacc)
                                    red_add_v4(dn.yacc + int64_t(tc) * dn.Mtot + col, a, keep_policy);
                                else
                                    *reinterpret_cast<float4 *>(dn.yp + int64_t(qbase + c0 + c) * dn.Mtot + col) = a;
                            }
                        }
                    } else {
                        // lane = output row; each column's 32 rows are one 128-byte store
                        float *yrow = dn.yp + int64_t(qbase + c0) * dn.Mtot + mt * 128 + 32 * lq + lane;
#pragma unroll
                        for (int j = 0; j < CW; ++j) {
                            const float wc = __shfl_sync(0xFFFFFFFFu, wsel, (c0 & 31) + j);
                            if (c0 + j < w.n_valid) yrow[int64_t(j) * dn.Mtot] = wc * __uint_as_float(v[j]);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            if (threadIdx.x == 64) LMOE_TRACE_EV(2, 0x60 | MODE, it, 0);  // epilogue: done
            if (++acc == C::ACC_STAGES) {
                acc = 0;
                acc_phase ^= 1;
            }
            return true;
        };
        // the buffer to zero: this CTA's slice [z, z1), a few units per
        // epilogue thread after each item, the rest after the last one
        int64_t z = 0, z1 = 0;
        if (MODE == GATEUP && p.zero) {
            const int64_t per = (p.zero_n4 + G - 1) / G;
            z = min(p.zero_n4, int64_t(blockIdx.x) * per);
            z1 = min(p.zero_n4, z + per);
        }
        const int et = threadIdx.x - 64, ne = 32 * C::EPI_WARPS;  // epilogue thread index and count
        const int64_t zstep = n_mine > 0 ? ((z1 - z) / n_mine + ne - 1) / ne * ne : 0;
        auto zero_some = [&](int64_t count) {
            const int64_t end = min(z1, z + count);
            for (int64_t u = z + et; u < end; u += ne) p.zero[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            z = end;
        };
        Item nA{}, nB{};
        float wA[NV], wB[NV];
        int tA[NV], tB[NV];
        if (0 < n_mine) fetch(seq(0), ent0, nA, wA, tA);
        if (1 < n_mine) fetch(seq(1), ent1, nB, wB, tB);
        int2 eA = entry(seq(2)), eB = entry(seq(3));  // next entries of the two sets
        for (int i = 0; i < n_mine; i += 2) {
            if (!process(seq(i), nA, wA, tA)) break;
            if (i + 2 < n_mine) {
                fetch(seq(i + 2), eA, nA, wA, tA);
                eA = entry(seq(i + 4));
            }
            zero_some(zstep);
            if (i + 1 >= n_mine) break;
            if (!process(seq(i + 1), nB, wB, tB)) break;
            if (i + 3 < n_mine) {
                fetch(seq(i + 3), eB, nB, wB, tB);
                eB = entry(seq(i + 5));
            }
            zero_some(zstep);
        }
        zero_some(z1 - z);
        if (threadIdx.x == 64) LMOE_TRACE_END(2);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    LMOE_TRACE_CTA(MODE, 1);
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// ---- schedule: slot starts and work-item prefixes (one CTA) ---------------------------
// Exclusive scan of v over [0, n), n <= 2048, by a 1024-thread block.
__device__ void block_exclusive_scan(const int32_t *v, int n, int32_t *out, int32_t *total, int32_t *warp_tot)
{
    const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
    const int i0 = 2 * threadIdx.x;
    const int32_t a = i0 < n ? v[i0] : 0, b = i0 + 1 < n ? v[i0 + 1] : 0;
    const int32_t s = a + b;
    int32_t incl = s;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int32_t t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        const int32_t wt = warp_tot[lane];
        int32_t wi = wt;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t t = __shfl_up_sync(0xFFFFFFFFu, wi, o);
            if (lane >= o) wi += t;
        }
        warp_tot[lane] = wi - wt;
        if (lane == 31) *total = wi;
    }
    __syncthreads();
    const int32_t excl = warp_tot[wid] + incl - s;
    if (i0 < n) out[i0] = excl;
    if (i0 + 1 < n) out[i0 + 1] = excl + a;
    __syncthreads();
}

__global__ void __launch_bounds__(1024) k_ffn_schedule(const int32_t *__restrict__ offsets, int E, FfnSched sc)
{
    pdl_enter();
    __shared__ int32_t v[2048], o[2049], warp_tot[32], tot;
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        const int n = offsets[e + 1] - offsets[e];
        v[e] = (n + sc.NT - 1) / sc.NT;  // token tiles of expert e
    }
    __syncthreads();
    block_exclusive_scan(v, E, o, &tot, warp_tot);
    if (threadIdx.x == 0) o[E] = tot;
    __syncthreads();
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
        sc.pad_off[e] = o[e] * sc.SLOT;
        sc.tiles_gu[e] = o[e] * sc.MT_gu;
        sc.tiles_dn[e] = o[e] * sc.MT_dn;
    }
    fill_tile_info(o, E, sc, blockDim.x);
    __syncthreads();
    fill_item_entries(sc, tot * sc.MT_gu, tot * sc.MT_dn, threadIdx.x, blockDim.x);
}

// ---- activations into the tiled token layout ------------------------------------------
__device__ __forceinline__ int64_t pad_row(int r, int32_t pad, int NT, int SLOT)
{
    return int64_t(pad) + int64_t(r / NT) * SLOT + (r % NT);
}


// bf16 x[T][d] -> MXFP8 rows at every token row the token's pairs go to
// (dst_row, written by the permute).  Work unit (token t, destination group,
// block b): block b of token t quantised and stored to the group's up to
// SCATTER_KG destination rows; a token's groups are separate units, so more
// threads (and stores) are in flight per token.  b runs fastest, so a warp's
// stores to one destination row are contiguous.
constexpr int SCATTER_KG = 8;
__global__ void k_quant_scatter_pad(const uint16_t *__restrict__ x, int64_t nunits, int d, int k,
                                    const int32_t *__restrict__ dst_row, const int32_t *__restrict__ inv,
                                    const float *__restrict__ topk_w, uint8_t *__restrict__ xq,
                                    uint8_t *__restrict__ xs, float *__restrict__ w_sorted, FfnSched sc, int E)
{
    pdl_enter();
    // the expert GEMMs' work-item tables, from the permute's tile_info
    fill_item_entries(sc, sc.tiles_gu[E], sc.tiles_dn[E], blockIdx.x * int64_t(blockDim.x) + threadIdx.x,
                      int64_t(gridDim.x) * blockDim.x);
    const int nb = d / 32, KC = d / 128;
    const int ng = (k + SCATTER_KG - 1) / SCATTER_KG;
    // unit g = half h (16 elements) of block b: lanes 2i and 2i+1 share a
    // block (its amax by one shuffle), and a warp's store to a destination
    // row is 512 contiguous bytes, 16 per lane
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < 2 * nunits; g += int64_t(gridDim.x) * blockDim.x) {
        const int h = int(g & 1);
        const int64_t gb = g >> 1;
        const int64_t tg = gb / nb;  // t * ng + group
        const int b = int(gb - tg * nb);
        const int64_t t = tg / ng;
        const int j0 = int(tg - t * ng) * SCATTER_KG;
        const int nj = min(SCATTER_KG, k - j0);
        const int64_t p0 = t * k + j0;  // first pair of the group
        // destination rows first: their loads overlap the quantisation below
        // a pair the permute rejected (expert id out of range, inv < 0) has
        // no token row: nothing is stored for it
        int32_t rows[SCATTER_KG], qs[SCATTER_KG];
#pragma unroll
        for (int j = 0; j < SCATTER_KG; ++j) {
            qs[j] = j < nj ? __ldg(inv + p0 + j) : -1;
            rows[j] = qs[j] >= 0 ? __ldg(dst_row + p0 + j) : -1;
        }
        const uint4 *src = reinterpret_cast<const uint4 *>(x + t * d + b * 32 + h * 16);
        uint4 raw[2];
#pragma unroll
        for (int i = 0; i < 2; ++i) raw[i] = __ldg(src + i);
        const uint32_t *rw = reinterpret_cast<const uint32_t *>(raw);
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = __uint_as_float(rw[i] << 16);
            v[2 * i + 1] = __uint_as_float(rw[i] & 0xFFFF0000u);
        }
        uint32_t amax = 0;
#pragma unroll
        for (int i = 0; i < 16; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
        // pairs of lanes are wholly active or inactive (2 * nunits is even and
        // every thread's start is even)
        const unsigned mask = __activemask();
        amax = max(amax, __shfl_xor_sync(mask, amax, 1));
        const uint32_t sb = mx_scale_byte(__uint_as_float(amax), 8);
        const float iv = mx_inv_scale(sb);
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) c[i] = e4m3x4(v[4 * i] * iv, v[4 * i + 1] * iv, v[4 * i + 2] * iv, v[4 * i + 3] * iv);
        // the 4 scale bytes of blocks 4c .. 4c+3 (adjacent in the atom) go out as
        // one 32-bit store by the first lane of the group's 8: groups of 4
        // consecutive blocks are aligned (d / 32 and every thread's start are
        // multiples of 4 blocks), so a group is either wholly active or wholly
        // inactive
        uint32_t sb4 = sb;
        sb4 |= __shfl_down_sync(mask, sb, 2) << 8;
        sb4 |= __shfl_down_sync(mask, sb, 4) << 16;
        sb4 |= __shfl_down_sync(mask, sb, 6) << 24;
#pragma unroll
        for (int j = 0; j < SCATTER_KG; ++j) {
            if (j >= nj) break;
            if (rows[j] < 0) continue;
            if (b == 0 && h == 0) w_sorted[qs[j]] = __ldg(topk_w + p0 + j);
            const int64_t R = rows[j];
            *reinterpret_cast<uint4 *>(xq + int64_t(qs[j]) * d + b * 32 + h * 16) = make_uint4(c[0], c[1], c[2], c[3]);
            if ((b & 3) == 0 && h == 0) *reinterpret_cast<uint32_t *>(xs + tile_atom_off(R, b, KC, sc.NT)) = sb4;
        }
    }
}

// The same for large batches, one token at a time per CTA: the CTA rounds
// the token's row to MXFP8 once into shared memory (thread b: block b of 32
// elements), then one thread sends the row to each of the token's k token
// rows by bulk asynchronous copies (shared -> global, whole 3.5 KB rows);
// the scale bytes (4 blocks per 32-bit word of the atom layout) go out as
// plain stores.  Two row buffers: one token's copies run while the next
// token is rounded.
constexpr int SCATTER_ROWS_THREADS = 128;
__global__ void __launch_bounds__(SCATTER_ROWS_THREADS) k_quant_scatter_rows(
    const uint16_t *__restrict__ x, int T, int d, int k, const int32_t *__restrict__ dst_row,
    const int32_t *__restrict__ inv, const float *__restrict__ topk_w, uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
    float *__restrict__ w_sorted, FfnSched sc, int E)
{
    extern __shared__ __align__(128) uint8_t qrow_smem[];  // [2][d] e4m3 codes
    __shared__ int32_t rows_s[2][32], qrow_s[2][32];  // per slot: atom row, code row (permuted order)
    pdl_enter();
    fill_item_entries(sc, sc.tiles_gu[E], sc.tiles_dn[E], blockIdx.x * int64_t(blockDim.x) + threadIdx.x,
                      int64_t(gridDim.x) * blockDim.x);
    const int nb = d / 32, KC = d / 128;
    int it = 0;
    for (int t = blockIdx.x; t < T; t += gridDim.x, ++it) {
        uint8_t *buf = qrow_smem + (it & 1) * d;
        int32_t *rows = rows_s[it & 1], *qrows = qrow_s[it & 1];
        // the copies that read this buffer two tokens ago have read it
        if (threadIdx.x == 0) tc::bulk_wait_read<1>();
        if (threadIdx.x < k) {
            const int64_t p = int64_t(t) * k + threadIdx.x;
            const int32_t q = __ldg(inv + p);  // < 0: the permute rejected the pair
            rows[threadIdx.x] = q >= 0 ? __ldg(dst_row + p) : -1;
            qrows[threadIdx.x] = q;
            if (q >= 0) w_sorted[q] = __ldg(topk_w + p);
        }
        __syncthreads();
        for (int b0 = 0; b0 < nb; b0 += blockDim.x) {
            const int b = b0 + threadIdx.x;
            uint32_t sb = 0;
            if (b < nb) {
                const uint4 *src = reinterpret_cast<const uint4 *>(x + int64_t(t) * d + b * 32);
                uint4 raw[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) raw[i] = __ldg(src + i);
                const uint32_t *rw = reinterpret_cast<const uint32_t *>(raw);
                float v[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    v[2 * i] = __uint_as_float(rw[i] << 16);
                    v[2 * i + 1] = __uint_as_float(rw[i] & 0xFFFF0000u);
                }
                uint32_t amax = 0;
#pragma unroll
                for (int i = 0; i < 32; ++i) amax = max(amax, __float_as_uint(v[i]) & 0x7FFFFFFFu);
                sb = mx_scale_byte(__uint_as_float(amax), 8);
                const float iv = mx_inv_scale(sb);
                uint32_t c[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    c[i] = e4m3x4(v[4 * i] * iv, v[4 * i + 1] * iv, v[4 * i + 2] * iv, v[4 * i + 3] * iv);
                uint4 *dst = reinterpret_cast<uint4 *>(buf + b * 32);
                dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
                dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
            }
            // blocks 4c .. 4c+3 sit in adjacent lanes (nb and b0 are multiples of 4)
            uint32_t sb4 = sb;
            sb4 |= __shfl_down_sync(0xFFFFFFFFu, sb, 1) << 8;
            sb4 |= __shfl_down_sync(0xFFFFFFFFu, sb, 2) << 16;
            sb4 |= __shfl_down_sync(0xFFFFFFFFu, sb, 3) << 24;
            if (b < nb && (b & 3) == 0) {
                for (int j = 0; j < k; ++j) {
                    const int32_t R = rows[j];
                    if (R >= 0) *reinterpret_cast<uint32_t *>(xs + tile_atom_off(R, b, KC, sc.NT)) = sb4;
                }
            }
        }
        tc::fence_async_shared();  // the row's generic-proxy writes, before the async copies read it
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int j = 0; j < k; ++j)
                if (rows[j] >= 0) tc::bulk_store(xq + int64_t(qrows[j]) * d, buf, uint32_t(d));
            tc::bulk_commit();
        }
    }
    if (threadIdx.x == 0) tc::bulk_wait<0>();  // the copies are complete before the grid is
}

// MXFP8 rows xq/xs [T][d] (canonical) -> tiled layout, row q of perm taking token perm[q]/k.
__global__ void k_gather_pad(const uint8_t *__restrict__ xq, const uint8_t *__restrict__ xs, int64_t P, int d, int k,
                             int E, const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
                             const float *__restrict__ topk_w, const int32_t *__restrict__ pad_off, int NT, int SLOT,
                             uint8_t *__restrict__ q_pad, uint8_t *__restrict__ s_pad, float *__restrict__ w_sorted)
{
    pdl_enter();
    const int cq = d / 16, nb = d / 32, KC = d / 128;
    const int per_row = cq + nb;
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < P * per_row; g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t qrow = g / per_row;
        const int c = int(g - qrow * per_row);
        int lo = 0, hi = E;  // offsets[lo] <= qrow < offsets[hi]
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (__ldg(offsets + mid) <= qrow) lo = mid;
            else hi = mid;
        }
        const int64_t R = pad_row(int(qrow - __ldg(offsets + lo)), __ldg(pad_off + lo), NT, SLOT);
        const int64_t pr = __ldg(perm + qrow), t = pr / k;
        if (c == 0) w_sorted[qrow] = __ldg(topk_w + pr);
        if (c < cq) {
            reinterpret_cast<uint4 *>(q_pad + qrow * d)[c] = __ldg(reinterpret_cast<const uint4 *>(xq + t * d) + c);
        } else {
            const int b = c - cq;
            s_pad[tile_atom_off(R, b, KC, NT)] = __ldg(xs + t * nb + b);
        }
    }
}

// ---- host side --------------------------------------------------------------------------
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// rows x K 2-D tensor map with 128-element x box_rows boxes, 128-byte swizzle.
bool make_map(CUtensorMap *m, const void *base, bool fp4, uint64_t K, uint64_t rows, uint64_t row_bytes,
              uint32_t box_rows)
{
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {128, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return enc(m, fp4 ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
               const_cast<void *>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms()
{
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

// Deepest pipeline that fits the per-block shared-memory limit (dynamic part
// after the kernel's static shared memory) and the TMEM column budget.
template <int MODE, int NT, bool SPLIT>
int gemm_stages(int E, size_t &smem)
{
    using C = Cfg<MODE, NT>;
    int dev = 0, optin = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    cudaFuncAttributes fa{};
    cudaFuncGetAttributes(&fa, k_moe_gemm<MODE, NT, SPLIT>);
    const size_t fixed = 1024 + C::EPI_BYTES + (2 * 16 + 2 * C::ACC_STAGES + 2) * 8 + 16 + size_t(2) * (E + 1) * 4;
    const long avail = long(optin) - long(fa.sharedSizeBytes) - long(fixed);
    int st = int(avail / long(C::STAGE_BYTES));
    if (st > C::MAX_STAGES) st = C::MAX_STAGES;
    smem = fixed + size_t(st > 0 ? st : 0) * C::STAGE_BYTES;
    return st;
}

// One GEMM (MODE GATEUP / DOWN: maps a0, a1, b and `args`), or both in the
// fused kernel (a0, a1, b and `args` the gate/up GEMM; d, h and `args2` the
// down GEMM).
template <int MODE, int NT, bool SPLIT = false>
cudaError_t launch_gemm(const CUtensorMap &a0, const CUtensorMap &a1, const CUtensorMap &b, GemmArgs args,
                        cudaStream_t st, const CUtensorMap *d = nullptr, const CUtensorMap *h = nullptr,
                        const GemmArgs *args2 = nullptr)
{
    size_t smem = 0;
    args.stages = gemm_stages<MODE, NT, SPLIT>(args.E, smem);
    if (args.stages < 2) return cudaErrorInvalidConfiguration;
    if (MODE == FUSED && (!d || !h || !args2)) return cudaErrorInvalidValue;
    cudaError_t e =
        cudaFuncSetAttribute(k_moe_gemm<MODE, NT, SPLIT>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    GemmArgs q = args2 ? *args2 : args;
    q.stages = args.stages;
    {
        const cudaError_t le_ = launch_pdl(k_moe_gemm<MODE, NT, SPLIT>, dim3(num_sms()), dim3(Cfg<MODE, NT>::THREADS), smem, st,
                                           a0, a1, b, d ? *d : a0, h ? *h : b, args, q);
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

}  // namespace

// Output-column bands of the fused-combine down GEMM: only 1/kDownBands of
// the per-token fp32 rows take reductions at a time.
constexpr int kDownBands = 2;

// 128-row weight tiles per down-GEMM item (Cfg<DOWN, NT>::MATS).
static int down_tiles_per_item(int NT) { return NT <= 96 ? 2 : 1; }

// Whether a batch of P pairs over E experts can have at most half as many
// gate/up work items (MT weight tiles per token tile) as the grid has CTAs,
// so that the fused kernel's split-K instance may run it: the token tiles
// sum_e ceil(n_e / NT) over the touched experts are at most
// (P + touched (NT - 1)) / NT.  The kernel checks the actual count again.
static bool ksplit_possible(int64_t P, int E, int NT, int MT, int KC)
{
    const int64_t touched = P < E ? P : E;
    const int64_t items = (P + touched * (NT - 1)) / NT * MT;
    return KC >= 2 && items <= KSPLIT_MAX_ITEMS && 2 * items <= num_sms();
}

FfnLayout ffn_layout(int64_t P, int d, int E, int I)
{
    FfnLayout L{};
    L.NT = P <= 4 * int64_t(E) ? 16 : (P <= 16 * int64_t(E) ? 32 : 96);
    L.fused = L.NT >= 64;  // Cfg<DOWN, NT>::STAGED
    L.SLOT = L.NT;  // packed tiles
    const int64_t touched = P < E ? P : E;
    const int64_t tiles = ceil_div(P, L.NT) + touched;  // bounds sum_e ceil(n_e / NT)
    // code rows: one per pair in permuted order, plus one tile's worth that
    // the last expert's last tile may read past the end (those columns of its
    // products are dropped); scale factors: one atom per tile and 128 columns
    L.rows = P + L.NT;
    const int64_t atoms = tiles;
    const int Ip = int(round_up(I, 128));
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t o = off;
        off += size_t(round_up(int64_t(bytes), 256));
        return o;
    };
    L.pad_off = take(size_t(E + 1) * 4);
    L.tiles_gu = take(size_t(E + 1) * 4);
    L.tiles_dn = take(size_t(E + 1) * 4);
    const int64_t max_tiles = tiles;
    L.items_gu = take(size_t(max_tiles * ceil_div(I, 128)) * sizeof(int2));
    L.items_dn = take(size_t(max_tiles * ceil_div(d / 128, down_tiles_per_item(L.NT))) * sizeof(int2));
    L.tile_info = take(size_t(max_tiles) * sizeof(int2));
    L.xq = take(size_t(L.rows) * d);
    L.xs = take(size_t(atoms) * (d / 128) * 512);
    L.hq = take(size_t(L.rows) * I);
    L.hs = take(size_t(atoms) * (Ip / 128) * 512);
    L.hs_bytes = size_t(atoms) * (Ip / 128) * 512;
    L.w_sorted = take(size_t(P) * 4);
    L.dst_row = take(size_t(P) * 4);
    L.tile_done = take(size_t(max_tiles) * 4);
    // split-K gate/up halves (the fused kernel at 16-token tiles): per item
    // and half the fp32 accumulators of both matrices (4 warps x 2 x 16 x 32),
    // per item one arrival counter per epilogue warp
    const bool ks = L.NT == 16;
    L.kpart = take(ks ? size_t(KSPLIT_MAX_ITEMS) * 2 * kKsplitHalfBytes : 0);
    L.kcnt = take(ks ? size_t(KSPLIT_MAX_ITEMS) * 4 * sizeof(int32_t) : 0);
    L.total = off;
    return L;
}

cudaError_t launch_ffn_schedule(const int32_t *offsets, int E, int d, int I, const FfnLayout &L, char *scratch,
                                cudaStream_t st)
{
    {
        const cudaError_t le_ =
            launch_pdl(k_ffn_schedule, dim3(1), dim3(1024), 0, st, offsets, E, ffn_sched(L, d, I, scratch));
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

FfnSched ffn_sched(const FfnLayout &L, int d, int I, char *scratch)
{
    FfnSched sc;
    sc.NT = L.NT;
    sc.SLOT = L.SLOT;
    sc.MT_gu = int(ceil_div(I, 128));
    sc.MT_dn = int(ceil_div(d / 128, down_tiles_per_item(L.NT)));
    sc.pad_off = reinterpret_cast<int32_t *>(scratch + L.pad_off);
    sc.tiles_gu = reinterpret_cast<int32_t *>(scratch + L.tiles_gu);
    sc.tiles_dn = reinterpret_cast<int32_t *>(scratch + L.tiles_dn);
    sc.items_gu = reinterpret_cast<int2 *>(scratch + L.items_gu);
    sc.items_dn = reinterpret_cast<int2 *>(scratch + L.items_dn);
    sc.tile_info = reinterpret_cast<int2 *>(scratch + L.tile_info);
    sc.band = L.NT >= 64 ? kDownBands : 0;  // Cfg<DOWN, NT>::STAGED: the fused combine
    sc.dst_row = reinterpret_cast<int32_t *>(scratch + L.dst_row);
    sc.tile_done = reinterpret_cast<int32_t *>(scratch + L.tile_done);
    sc.kcnt = L.NT == 16 ? reinterpret_cast<int32_t *>(scratch + L.kcnt) : nullptr;
    return sc;
}

// Batches from this many tokens take the whole-row scatter (k_quant_scatter_rows).
constexpr int kScatterRowsMinTokens = 1024;

cudaError_t launch_quant_scatter_pad(const uint16_t *x, int T, int d, int k, int E, int I, const int32_t *inv,
                                     const float *topk_w, const FfnLayout &L, char *scratch, cudaStream_t st)
{
    const int64_t nunits = int64_t(T) * ceil_div(k, SCATTER_KG) * (d / 32);
    if (nunits == 0) return cudaSuccess;
    if (T >= kScatterRowsMinTokens) {
        // one token per CTA at a time, whole rows by bulk copies
        const int grid = T < 16 * num_sms() ? T : 16 * num_sms();
        const size_t smem = size_t(2) * d;
        if (smem > 48 * 1024) {
            cudaError_t e = cudaFuncSetAttribute(k_quant_scatter_rows, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 int(smem));
            if (e != cudaSuccess) return e;
        }
        const cudaError_t le_ = launch_pdl(
            k_quant_scatter_rows, dim3(grid), dim3(SCATTER_ROWS_THREADS), smem, st, x, T, d, k,
            reinterpret_cast<const int32_t *>(scratch + L.dst_row), inv, topk_w, reinterpret_cast<uint8_t *>(scratch + L.xq),
            reinterpret_cast<uint8_t *>(scratch + L.xs), reinterpret_cast<float *>(scratch + L.w_sorted),
            ffn_sched(L, d, I, scratch), E);
        if (le_ != cudaSuccess) return le_;
        return cudaGetLastError();
    }
    const int grid = int(ceil_div(2 * nunits, 128) < 152 * 32 ? ceil_div(2 * nunits, 128) : 152 * 32);
    {
        const cudaError_t le_ = launch_pdl(k_quant_scatter_pad, dim3(grid), dim3(128), 0, st, x, nunits, d, k, reinterpret_cast<const int32_t *>(scratch + L.dst_row), inv, topk_w, reinterpret_cast<uint8_t *>(scratch + L.xq), reinterpret_cast<uint8_t *>(scratch + L.xs), reinterpret_cast<float *>(scratch + L.w_sorted), ffn_sched(L, d, I, scratch), E);
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

cudaError_t launch_gather_pad(const uint8_t *xq, const uint8_t *xs, int T, int d, int k, int E, const int32_t *offsets,
                              const int32_t *perm, const float *topk_w, const FfnLayout &L, char *scratch,
                              cudaStream_t st)
{
    const int64_t P = int64_t(T) * k;
    const int64_t n = P * (d / 16 + d / 32);
    if (n == 0) return cudaSuccess;
    const int grid = int(ceil_div(n, 256) < 152 * 64 ? ceil_div(n, 256) : 152 * 64);
    {
        const cudaError_t le_ = launch_pdl(k_gather_pad, dim3(grid), dim3(256), 0, st, xq, xs, P, d, k, E, offsets, perm, topk_w, reinterpret_cast<const int32_t *>(scratch + L.pad_off), L.NT, L.SLOT, reinterpret_cast<uint8_t *>(scratch + L.xq), reinterpret_cast<uint8_t *>(scratch + L.xs), reinterpret_cast<float *>(scratch + L.w_sorted));
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

cudaError_t launch_expert_gemms(const FfnArgs &a, const FfnLayout &L, char *scratch, cudaStream_t st, cudaEvent_t mid)
{
    if (a.P == 0) return cudaSuccess;
    if (a.yacc && !L.fused) return cudaErrorInvalidValue;  // the fused combine needs the staged epilogue
    const int Ip = int(round_up(a.I, 128));
    uint8_t *xq = reinterpret_cast<uint8_t *>(scratch + L.xq);
    uint8_t *xs = reinterpret_cast<uint8_t *>(scratch + L.xs);
    uint8_t *hq = reinterpret_cast<uint8_t *>(scratch + L.hq);
    uint8_t *hs = reinterpret_cast<uint8_t *>(scratch + L.hs);
    if (a.I % 128 != 0) {
        // scale blocks past I in the last K chunk of h must be finite (the
        // matching A codes and B values are zero)
        cudaError_t e = cudaMemsetAsync(hs, 0, L.hs_bytes, st);
        if (e != cudaSuccess) return e;
    }
    CUtensorMap mg, mu, mx, md, mh;
    const bool ok = make_map(&mg, a.W->gate_q, true, uint64_t(a.d), uint64_t(a.E) * a.I, uint64_t(a.d) / 2, 128) &&
                    make_map(&mu, a.W->up_q, true, uint64_t(a.d), uint64_t(a.E) * a.I, uint64_t(a.d) / 2, 128) &&
                    make_map(&md, a.W->down_q, true, uint64_t(Ip), uint64_t(a.E) * a.d, uint64_t(Ip) / 2, 128) &&
                    make_map(&mx, xq, false, uint64_t(a.d), uint64_t(L.rows), uint64_t(a.d), uint32_t(L.NT)) &&
                    make_map(&mh, hq, false, uint64_t(a.I), uint64_t(L.rows), uint64_t(a.I), uint32_t(L.NT));
    if (!ok) return cudaErrorInvalidValue;
    GemmArgs g{};
    g.offsets = a.offsets;
    g.w_sorted = reinterpret_cast<const float *>(scratch + L.w_sorted);
    g.E = a.E;
    g.status = a.status;
    g.wait_limit = a.wait_limit > 0 ? a.wait_limit : 4000000000LL;  // ~2 s of SM clocks
    g.stall_first_fill = a.stall_first_fill;
    // gate/up
    g.sfa0 = a.W->gate_s;
    g.sfa1 = a.W->up_s;
    g.sfb = xs;
    g.tiles = reinterpret_cast<const int32_t *>(scratch + L.tiles_gu);
    g.pad_off = reinterpret_cast<const int32_t *>(scratch + L.pad_off);
    g.items = reinterpret_cast<const int2 *>(scratch + L.items_gu);
    g.hq = hq;
    g.hs = hs;
    g.hcap = a.hcap;
    g.Mtot = a.I;
    g.MTA = int(ceil_div(a.I, 128));
    g.KC = a.d / 128;
    g.KCh = Ip / 128;
    g.Ih = a.I;
    g.tile_done = reinterpret_cast<int32_t *>(scratch + L.tile_done);
    g.kpart = L.NT == 16 ? reinterpret_cast<float *>(scratch + L.kpart) : nullptr;
    g.kcnt = L.NT == 16 ? reinterpret_cast<int32_t *>(scratch + L.kcnt) : nullptr;
    // the fused combine's sums start at zero: the gate/up epilogue clears them
    g.zero = a.yacc ? reinterpret_cast<float4 *>(a.yacc) : nullptr;
    g.zero_n4 = a.yacc ? int64_t(a.P / a.k) * a.d / 4 : 0;
    // down
    GemmArgs gd = g;
    gd.zero = nullptr;
    gd.zero_n4 = 0;
    gd.sfa0 = a.W->down_s;
    gd.sfa1 = a.W->down_s;  // the second tile of a down item is the next tile of the same matrix
    gd.sfb = hs;
    gd.tiles = reinterpret_cast<const int32_t *>(scratch + L.tiles_dn);
    gd.items = reinterpret_cast<const int2 *>(scratch + L.items_dn);
    gd.hcap = nullptr;
    gd.yp = a.yp;
    gd.yacc = a.yacc;
    gd.perm = a.perm;
    gd.k = a.k;
    gd.Mtot = a.d;
    gd.MTA = a.d / 128;
    gd.KC = Ip / 128;
    if (ffn_fused(L)) {
        // both GEMMs in one persistent kernel (the stage-boundary event, if
        // asked for, follows it)
        const bool split = L.NT == 16 && g.kpart && ksplit_possible(a.P, a.E, L.NT, g.MTA, g.KC);
        cudaError_t e = split        ? launch_gemm<FUSED, 16, true>(mg, mu, mx, g, st, &md, &mh, &gd)
                        : L.NT == 16 ? launch_gemm<FUSED, 16>(mg, mu, mx, g, st, &md, &mh, &gd)
                        : L.NT == 32 ? launch_gemm<FUSED, 32>(mg, mu, mx, g, st, &md, &mh, &gd)
                                     : launch_gemm<FUSED, 96>(mg, mu, mx, g, st, &md, &mh, &gd);
        if (e == cudaSuccess && mid) e = cudaEventRecord(mid, st);
        return e;
    }
    cudaError_t e = launch_gemm<GATEUP, 96>(mg, mu, mx, g, st);
    if (e != cudaSuccess) return e;
    if (mid) {
        e = cudaEventRecord(mid, st);
        if (e != cudaSuccess) return e;
    }
    return launch_gemm<DOWN, 96>(md, md, mh, gd, st);
}

}  // namespace lmoe
