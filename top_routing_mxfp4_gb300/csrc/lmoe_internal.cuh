// Internal declarations shared by the lmoe CUDA translation units.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/lmoe.h"

namespace lmoe {

// ---- programmatic dependent launch -------------------------------------------------------
// Every kernel of the library is launched with programmatic stream
// serialisation: it may be scheduled while the previous kernel of the stream
// drains.  Before reading that kernel's outputs or writing global memory it
// calls pdl_wait() (returns once the previous grid has completed and its
// writes are visible), and only then allows its own dependents to be
// scheduled (pdl_trigger), so at most the immediately preceding kernel can
// still be running while a kernel does its pre-wait work; outputs of earlier
// kernels are complete.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait();
    pdl_trigger();
}
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args... args)
{
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- status word (first 4 bytes of a workspace) ---------------------------------
// Kernels record the first error they see; the host reads it back with
// lmoe_last_device_status.
__device__ __forceinline__ void set_status(int32_t *status, int32_t code)
{
    if (status) atomicCAS(status, 0, code);
}

// ---- small numeric helpers ----------------------------------------------------------
__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

// Shared block exponent as an E8M0 byte: clamp(floor(log2 amax) - emax + 127, 0, 254),
// 0 for amax == 0.  floor(log2) is read from the fp32 bit pattern (normals:
// exponent field - 127; subnormals: position of the leading mantissa bit).
__device__ __forceinline__ uint32_t mx_scale_byte(float amax, int emax)
{
    uint32_t u = __float_as_uint(amax) & 0x7FFFFFFFu;
    if (u == 0) return 0;
    int ex = int(u >> 23);
    int fl = ex ? ex - 127 : (31 - __clz(u)) - 149;
    int b = fl - emax + 127;
    return uint32_t(b < 0 ? 0 : (b > 254 ? 254 : b));
}

// 2^(127 - byte) as fp32 (byte in [0, 254] -> exponent in [-127, 127]); the
// multiplier that divides a block by its scale.  2^-127 is a subnormal.
__device__ __forceinline__ float mx_inv_scale(uint32_t byte)
{
    int e = 127 - int(byte);  // in [-127, 127]
    return e >= -126 ? __uint_as_float(uint32_t(e + 127) << 23) : __uint_as_float(0x00400000u);
}

// 2^(byte - 127) as fp32 (decode of an E8M0 byte in [0, 254]).
__device__ __forceinline__ float e8m0_to_f32(uint32_t byte)
{
    return byte ? __uint_as_float(byte << 23) : __uint_as_float(0x00400000u);
}

// Eight fp32 values (already divided by the block scale) -> eight e2m1 codes
// packed in a 32-bit word, element i in nibble i.  Hardware conversion:
// round to nearest even, saturate to the largest finite value.
__device__ __forceinline__ uint32_t e2m1x8(const float *v)
{
    uint32_t out;
    asm("{\n\t.reg .b8 b0, b1, b2, b3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n\t"
        "mov.b32 %0, {b0, b1, b2, b3};\n\t}"
        : "=r"(out)
        : "f"(v[0]), "f"(v[1]), "f"(v[2]), "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7]));
    return out;
}

// Two fp32 values -> two e4m3 codes (lo in the low byte), round to nearest
// even, saturate to +-448.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t out;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %2, %1;" : "=h"(out) : "f"(lo), "f"(hi));
    return out;
}

// Four fp32 -> four e4m3 codes in one word (element i in byte i).
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    return e4m3x2(a, b) | (e4m3x2(c, d) << 16);
}

// e4m3 byte -> fp32 via the hardware f16x2 conversion (exact).
__device__ __forceinline__ float e4m3_to_f32(uint32_t code)
{
    uint32_t h2;
    uint16_t in = uint16_t(code & 0xFF);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(in));
    return __half2float(__ushort_as_half(uint16_t(h2 & 0xFFFF)));
}

__host__ __device__ constexpr int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Scale byte of (token row R, block b) in the expert GEMMs' token layout:
// tiles of NT rows packed one after another, each tile's scale factors one
// 512-byte atom per 128 columns (KC atoms per tile); row rr = R % NT of the
// tile at byte 16*(rr % 32) + 4*(rr / 32) + b % 4 of atom (tile * KC + b / 4).
__host__ __device__ __forceinline__ int64_t tile_atom_off(int64_t R, int b, int KC, int NT)
{
    const int64_t tile = R / NT;
    const int rr = int(R - tile * NT);
    return (tile * KC + (b >> 2)) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + (b & 3);
}
__host__ __device__ constexpr int64_t round_up(int64_t a, int64_t b) { return ceil_div(a, b) * b; }

// ---- host-side launch wrappers (each returns cudaError_t of the launch) --------------
cudaError_t launch_quant_mxfp4(const float *w, int64_t nmat, int rows, int K, uint8_t *q, uint8_t *s, int layout,
                               cudaStream_t st);
cudaError_t launch_quant_mxfp8(const uint16_t *x, int64_t rows, int K, uint8_t *q, uint8_t *s, cudaStream_t st);
// canonical MXFP4 bytes -> the tensor-core layout (a byte rearrangement)
cudaError_t launch_repack_mxfp4(const uint8_t *q, const uint8_t *s, int64_t nmat, int rows, int K, uint8_t *q_tc,
                                uint8_t *s_tc, cudaStream_t st);
// per-matrix counts of each E8M0 scale byte, hist[nmat][256]
cudaError_t launch_scale_histogram(const uint8_t *s, int64_t nmat, int rows, int K, int layout, uint32_t *hist,
                                   cudaStream_t st);
// Router logits on the tensor cores (fp32 weights split into three bf16 parts).
size_t router_scratch_bytes(int T, int d, int E);
int router_kernel_count(int T, int d, int E);  // kernels of launch_route, top-k included
int permute_kernel_count(int64_t P);
// out[t][n] = bf16(sum_c x[t][c] W[n][c]), bf16 operands, fp32 accumulation.
size_t linear_scratch_bytes(int T, int K, int N);
cudaError_t launch_linear_bf16(const uint16_t *x, const uint16_t *W, int T, int K, int N, uint16_t *out, void *scratch,
                               int32_t *status, cudaStream_t st);
// Top-k + softmax of fp32 logits [T][E].
// status: the workspace's status word (the staged large-batch kernel's
// bounded waits report there); null selects the unstaged kernel.
cudaError_t launch_topk_softmax(const float *logits, int T, int E, int k, int32_t *idx, float *w, cudaStream_t st,
                                int32_t *status = nullptr);

// Optional by-products of the permute for the expert GEMMs: per expert the
// first atom row of its token tiles (pad_off = first tile * NT, E+1) and the
// first work item of each GEMM (tiles_gu / tiles_dn, E+1), the expert of each
// token tile (tile_info; the activation scatter turns it into the GEMMs'
// work-item tables items_gu / items_dn), and per pair p its atom row (dst_row,
// T*k: tile * NT + row in tile, which locates its scale factors; its codes sit
// at its permuted position).  pad_off == nullptr disables them.
struct FfnSched {
    int NT = 0, SLOT = 0, MT_gu = 0, MT_dn = 0;
    int band = 0;  // the down GEMM runs its items in this many output-column bands (0 or 1: one)
    int32_t *pad_off = nullptr, *tiles_gu = nullptr, *tiles_dn = nullptr, *dst_row = nullptr;
    int2 *items_gu = nullptr, *items_dn = nullptr;
    int2 *tile_info = nullptr;  // per token tile: {expert, token tile within the expert}
    int32_t *tile_done = nullptr;  // per token tile: the fused GEMM kernel's h-complete counter (zeroed here)
    int32_t *kcnt = nullptr;  // per gate/up item (the first KSPLIT_MAX_ITEMS): 4 split-K arrival counters (zeroed here)
};
// Gate/up items of one fused-kernel launch that may run as two K halves
// (the halves' fp32 accumulators have room for this many items).
constexpr int KSPLIT_MAX_ITEMS = 128;

// Work-item tables of the two expert GEMMs, in execution order: entry i is
// item i as {expert | weight tile << 16, token tile within the expert}.
// gate/up: items in (token tile, weight tile) order, weight tile fastest.
// down: the same, or with `band`, every item of the first half of the weight
// tiles before the second half (each half in that order), so that only half
// of the per-token output rows take reductions at a time.
// Two steps: tile_info[R] = {expert, token tile within the expert} for every
// token tile R (from the scan of token tiles per expert, E + 1 entries; one
// block), then any grid writes the entries, consecutive threads consecutive
// entries (the table sizes are tiles_gu[E] and tiles_dn[E]).
__device__ __forceinline__ void fill_tile_info(const int32_t *scan, int E, const FfnSched &sc, int nthreads)
{
    for (int e = threadIdx.x; e < E; e += nthreads)
        for (int R = scan[e]; R < scan[e + 1]; ++R) {
            sc.tile_info[R] = make_int2(e, R - scan[e]);
            if (sc.tile_done) sc.tile_done[R] = 0;
        }
}
// Entries [g0, n_gu + n_dn) with stride `step` (gate/up entries first).
// Down entries in bands: band b holds weight tiles [b*MT/NB, (b+1)*MT/NB) of
// every token tile, bands one after another.
__device__ __forceinline__ void fill_item_entries(const FfnSched &sc, int n_gu, int n_dn, int64_t g0, int64_t step)
{
    const int TT = n_gu / sc.MT_gu;
    const int NBd = sc.band > 1 ? sc.band : 1;
    for (int64_t g = g0; g < int64_t(n_gu) + n_dn; g += step) {
        int R, m;
        int2 *dst;
        if (g < n_gu) {
            R = int(g) / sc.MT_gu;
            m = int(g) - R * sc.MT_gu;
            dst = sc.items_gu + g;
            if (sc.kcnt && g < KSPLIT_MAX_ITEMS) reinterpret_cast<int4 *>(sc.kcnt)[g] = make_int4(0, 0, 0, 0);
        } else {
            const int it = int(g - n_gu);
            // band b starts at item TT * m_lo(b), m_lo(b) = b * MT / NBd
            int b = 0;
            while (b + 1 < NBd && it >= TT * ((b + 1) * sc.MT_dn / NBd)) ++b;
            const int m_lo = b * sc.MT_dn / NBd, m_len = (b + 1) * sc.MT_dn / NBd - m_lo;
            const int r = it - TT * m_lo;
            R = r / m_len;
            m = m_lo + (r - R * m_len);
            dst = sc.items_dn + it;
        }
        const int2 ti = sc.tile_info[R];
        *dst = make_int2(ti.x | (m << 16), ti.y);
    }
}
// Small batches (T <= 64): the permute done by the routing kernel.  Each
// token's CTA sets bit t of mask[e] for its selected experts; the last CTA to
// finish derives counts, offsets, the FFN schedule and, per pair p = t*k + j
// with expert e, its sorted position offsets[e] + popcount(mask[e] & (2^t - 1))
// (the stable counting sort's order: within an expert, pairs by token) into
// inv[p], perm[pos] and the pair's atom row.  mask and counter are zero when
// the call starts.  mask == null: not used.
struct PermByMask {
    unsigned long long *mask = nullptr;  // [E]
    int32_t *counter = nullptr;          // CTAs done
    int32_t *counts = nullptr, *offsets = nullptr, *perm = nullptr, *inv = nullptr;
    FfnSched sc;
};
// split-K partial logits [KS][T][E] -> logits (+ bias) and their top-k + softmax, one launch
cudaError_t launch_reduce_topk(const float *part, int KS, int T, int E, const float *bias, float *logits, int k,
                               int32_t *idx, float *w, cudaStream_t st, const PermByMask &pm = PermByMask());
// Router logits + top-k + softmax (split, GEMM, split-K reduction, selection).
// fp32 router weights [E][d] -> three bf16 planes [3][E][d] whose sum is exact
cudaError_t launch_split_router(const float *Wr, int E, int d, uint16_t *Wr3, cudaStream_t st);
cudaError_t launch_route(const uint16_t *x, const uint16_t *Wr3, const float *bias, int T, int d, int E, int k,
                         float *logits, int32_t *idx, float *w, void *scratch, int32_t *status, cudaStream_t st,
                         const PermByMask &pm = PermByMask());
// whether launch_route can also do the permute (PermByMask) for these dims
bool route_can_permute(int T, int d, int E, int k);
// pairs per block of the multi-block permute (its scratch: one histogram of
// E counts per block)
constexpr int PERMUTE_CHUNK = 2048;
size_t permute_scratch_bytes(int64_t P, int E);
cudaError_t launch_permute(const int32_t *idx, int64_t P, int E, int32_t *counts, int32_t *offsets, int32_t *perm,
                           int32_t *inv, void *scratch, int32_t *status, cudaStream_t st,
                           const FfnSched &sched = FfnSched());

// Expert FFN (tensor cores).  Activation codes live one row per pair in
// permuted order inside the FFN scratch, their scale factors in one atom per
// NT-row token tile (tiles numbered per expert from pad_off[e] / NT); see
// k_ffn_tc.cu.
struct FfnLayout {
    int NT, SLOT;      // token tile and the rows a tile occupies (SLOT == NT: tiles are packed)
    int64_t rows;      // code rows reserved: one per pair (permuted order) + one tile past the end
    size_t pad_off, tiles_gu, tiles_dn, items_gu, items_dn, tile_info, xq, xs, hq, hs, hs_bytes, w_sorted, dst_row,
        tile_done, kpart, kcnt, total;  // byte offsets / sizes (kpart, kcnt: 16-token tiles only, else empty)
    bool fused;  // large token tiles: the down GEMM can accumulate into the per-token output (FfnArgs::yacc)
};
FfnLayout ffn_layout(int64_t P, int d, int E, int I);
// Whether the two expert GEMMs of this layout run as one fused kernel: for
// decode-sized token tiles (at 96-token tiles the fused kernel measured
// slower than two kernels).
inline bool ffn_fused(const FfnLayout &L) { return L.NT <= 32; }
// The permute by-products the forward asks for, pointing into the FFN scratch.
FfnSched ffn_sched(const FfnLayout &L, int d, int I, char *scratch);

struct FfnArgs {
    const lmoe_expert_weights *W;
    const int32_t *offsets, *perm;
    const float *topk_w;
    int P, d, E, k, I;
    float *yp;    // [P][d] in permuted order
    float *yacc;  // when set (FfnLayout::fused only): [T][d] fp32 sums over the k pairs instead of yp (the gate/up kernel zeroes it)
    int32_t *status;
    float *hcap = nullptr;  // diagnostics: fp32 h before its MXFP8 rounding, [FfnLayout::rows][I]
    long long wait_limit = 0;   // bounded-wait limit in SM clocks (0: the default, ~2 s)
    int stall_first_fill = 0;   // failure-path test: the GEMMs' first stage never fills
};
// slot starts and per-GEMM work-item prefixes from the segment offsets
cudaError_t launch_ffn_schedule(const int32_t *offsets, int E, int d, int I, const FfnLayout &L, char *scratch,
                                cudaStream_t st);
// bf16 x[T][d] -> MXFP8 codes at each routed pair's permuted row (inv) and
// scales at its atom row (dst_row, from the permute); also the gate weights
// in permuted order.
// (also writes the expert GEMMs' work-item tables from the permute's tile_info)
cudaError_t launch_quant_scatter_pad(const uint16_t *x, int T, int d, int k, int E, int I, const int32_t *inv,
                                     const float *topk_w, const FfnLayout &L, char *scratch, cudaStream_t st);
// MXFP8 rows in token order -> tiled layout (row q of perm takes token perm[q]/k)
cudaError_t launch_gather_pad(const uint8_t *xq, const uint8_t *xs, int T, int d, int k, int E, const int32_t *offsets,
                              const int32_t *perm, const float *topk_w, const FfnLayout &L, char *scratch,
                              cudaStream_t st);
// gate/up GEMM (+ SwiGLU, MXFP8 of h), event `mid` (if set), down GEMM (x gate weight)
cudaError_t launch_expert_gemms(const FfnArgs &a, const FfnLayout &L, char *scratch, cudaStream_t st,
                                cudaEvent_t mid = nullptr);

// ---- small batches (k_small.cu): three weight-streaming kernels ----------------------
constexpr int SMALL_MAX_TOKENS = 8;
constexpr int SMALL_MAX_PAIRS = 256;
struct SmallLayout {
    size_t n_touched, seg_expert, seg_start, seg_pair, xq, xs, hq, hs, total;  // byte offsets / size
};
SmallLayout small_layout(int T, int d, int E, int k, int I);
// whether a batch of these dims can take the small-batch path (shared-memory
// limits), given the largest pair count the caller allows on it
bool small_path_fits(int T, int d, int E, int k, int I, int max_pairs);
// route + top-k + pair lists + MXFP8 (or, act == LMOE_ACT_MXFP4, MXFP4) x;
// gate/up + SwiGLU + the same rounding of h; down + combine.  `counter` (an int32 that is zero when the call starts) counts the
// routing CTAs; stage_events (optional, LMOE_NUM_STAGE_EVENTS of them): [1..3]
// are recorded after the routing kernel, [4] after gate/up.
cudaError_t launch_small_forward(const uint16_t *x, const uint16_t *Wr3, const float *bias, const lmoe_expert_weights *W,
                                 int T, int d, int E, int k, int I, int act, float *logits, int32_t *idx, float *w,
                                 uint16_t *y, const SmallLayout &L, char *scratch, int32_t *status, int32_t *counter,
                                 float *hcap, cudaStream_t st, const cudaEvent_t *stage_events);

// inv_early: inv is complete before the kernel preceding the combine starts
// (true inside lmoe_forward; false for the standalone entry point).
cudaError_t launch_combine(const float *yp, const int32_t *inv, int T, int d, int k, uint16_t *y, cudaStream_t st,
                           bool inv_early);
// y = bf16(acc), n elements (n % 4 == 0)
cudaError_t launch_acc_to_bf16(const float *acc, int64_t n, uint16_t *y, cudaStream_t st);

}  // namespace lmoe
