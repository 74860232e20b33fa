// Dense bf16 GEMMs on the tensor cores (tcgen05.mma kind::f16, fp32
// accumulation in TMEM): out[t][n] = sum_c x[t][c] * W[n][c].
//
// Two users:
//  * the router ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
//    "MoE 稀疏激活": scores = token embeddings x router weights).  The router
//    weights are fp32; they are split once per call into three bf16 parts
//    W = W_hi + W_mid + W_lo (8 + 8 + 8 significand bits), and the three
//    bf16 x bf16 products, exact in fp32, accumulate into one fp32
//    accumulator, so the logits carry fp32-level accuracy;
//  * the hidden <-> latent projections around the layer ("从Kimi K3到
//    MiniMax-H3" section 一: LatentMoE compresses the hidden state to the
//    3584-wide latent space first), bf16 weights, bf16 output.
//
// Weights are the M = 128 operand (A), tokens the N operand (B, N = NB per
// tile), both K-major, 64 bf16 (one 128-byte swizzle row) per K chunk.  With
// few tokens the K dimension is split over CTAs (fp32 partials, then a fixed-
// order reduction), so the weight stream is spread over the whole GPU.
// Same warp roles as the expert GEMMs: TMA producer, single-thread MMA issuer,
// four epilogue warps; every wait bounded.
#include <cuda.h>
#include <cuda_bf16.h>

#include "lmoe_internal.cuh"
#include "tc_ptx.cuh"

namespace lmoe {
namespace {

using namespace tc;

enum { OUT_F32 = 0, OUT_BF16 = 1, OUT_PARTIAL = 2 };

struct DenseArgs {
    int M, T, K;        // weight rows, tokens, reduction length
    int MT, NTL, KS;    // m tiles, token tiles, K slices
    int kc_per_slice;   // 64-wide K chunks per slice
    const float *bias;  // [M] (OUT_F32) or null
    void *out;          // [T][M] fp32 / bf16, or partials [KS][T][M] fp32
    int32_t *status;
};

template <int NPARTS, int NB>
struct DCfg {
    static constexpr uint32_t A_TILE = 128 * 128;  // 128 rows x 64 bf16
    static constexpr uint32_t B_TILE = NB * 128;
    static constexpr uint32_t STAGE_BYTES = NPARTS * A_TILE + B_TILE;
    static constexpr uint32_t TX_BYTES = STAGE_BYTES;
    static constexpr int STAGES_RAW = (200 * 1024) / int(STAGE_BYTES);
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr int ACC_STAGES = 2;
    static_assert(ACC_STAGES * NB <= 512, "TMEM columns");
    static_assert(STAGES >= 2, "pipeline depth");
};

// kind::f16 instruction descriptor: fp32 accumulator, A and B bf16, both
// K-major, M = 128, N given.
__device__ __forceinline__ uint32_t idesc_bf16(uint32_t N)
{
    return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((128u >> 4) << 24);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate)
{
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
                 "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate));
}

template <int NPARTS, int NB, int OUT>
__global__ void __launch_bounds__(192, 1)
    k_gemm_bf16(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const DenseArgs p)
{
    using C = DCfg<NPARTS, NB>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *stages = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t *full = reinterpret_cast<uint64_t *>(stages + C::STAGES * C::STAGE_BYTES);
    uint64_t *empty = full + C::STAGES;
    uint64_t *acc_full = empty + C::STAGES;
    uint64_t *acc_empty = acc_full + C::ACC_STAGES;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(acc_empty + C::ACC_STAGES);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < C::STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < C::ACC_STAGES; ++a) {
            mbar_init(&acc_full[a], 1);
            mbar_init(&acc_empty[a], 128);
        }
        mbar_init_fence();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tensormap(&tmA);
        prefetch_tensormap(&tmB);
    }
    if (warp == 1) tmem_alloc(tmem_slot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const int total = p.MT * p.NTL * p.KS;
    pdl_enter();

    // item -> (k slice, token tile, m tile); m fastest so neighbouring CTAs share the token tile
    if (warp == 0) {
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
                const int mt = it % p.MT, rest = it / p.MT, nt = rest % p.NTL, ks = rest / p.NTL;
                for (int c = 0; c < p.kc_per_slice; ++c) {
                    const int kx = (ks * p.kc_per_slice + c) * 64;
                    if (!mbar_wait(&empty[stage], phase ^ 1)) {
                        set_status(p.status, LMOE_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    uint8_t *sb = stages + stage * C::STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], C::TX_BYTES);
#pragma unroll
                    for (int part = 0; part < NPARTS; ++part)
                        tma_load_2d(sb + part * C::A_TILE, &tmA, kx, part * p.M + mt * 128, &full[stage]);
                    tma_load_2d(sb + NPARTS * C::A_TILE, &tmB, kx, nt * NB, &full[stage]);
                    if (++stage == C::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
                const int nt = (it / p.MT) % p.NTL;
                const int nv = min(NB, p.T - nt * NB);
                const uint32_t N = uint32_t((nv + 15) & ~15);
                const uint32_t id = idesc_bf16(N);
                if (!mbar_wait(&acc_empty[acc], acc_phase ^ 1)) {
                    set_status(p.status, LMOE_ERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const uint32_t d = tmem + uint32_t(acc * NB);
                for (int c = 0; c < p.kc_per_slice; ++c) {
                    if (!mbar_wait(&full[stage], phase)) {
                        set_status(p.status, LMOE_ERR_TIMEOUT);
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint8_t *sb = stages + stage * C::STAGE_BYTES;
                    const uint64_t bd = sdesc_k128(smem_u32(sb + NPARTS * C::A_TILE));
#pragma unroll
                    for (int part = 0; part < NPARTS; ++part) {
                        const uint64_t ad = sdesc_k128(smem_u32(sb + part * C::A_TILE));
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // 4 x K=16 per 128-byte row
                            mma_bf16(d, ad + 2 * kk, bd + 2 * kk, id, (c | part | kk) ? 1u : 0u);
                    }
                    tc_commit(&empty[stage]);
                    if (++stage == C::STAGES) {
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
        }
    } else {
        const int q = warp & 3;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int it = blockIdx.x; it < total; it += gridDim.x) {
            const int mt = it % p.MT, rest = it / p.MT, nt = rest % p.NTL, ks = rest / p.NTL;
            const int nv = min(NB, p.T - nt * NB);
            if (!mbar_wait(&acc_full[acc], acc_phase)) {
                set_status(p.status, LMOE_ERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const int row = mt * 128 + 32 * q + lane;
            const uint32_t tb = tmem + (uint32_t(32 * q) << 16) + uint32_t(acc * NB);
            const float b = (OUT == OUT_F32 && p.bias && row < p.M) ? __ldg(p.bias + row) : 0.f;
            for (int c0 = 0; c0 < nv; c0 += 16) {
                uint32_t v[16];
                tmem_ld16(tb + c0, v);
                tmem_ld_wait();
                if (row < p.M) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) {
                        const int t = nt * NB + c0 + j;
                        if (c0 + j >= nv) break;
                        const float y = __uint_as_float(v[j]);
                        if (OUT == OUT_F32) {
                            reinterpret_cast<float *>(p.out)[int64_t(t) * p.M + row] = p.bias ? y + b : y;
                        } else if (OUT == OUT_PARTIAL) {
                            reinterpret_cast<float *>(p.out)[(int64_t(ks) * p.T + t) * p.M + row] = y;
                        } else {
                            reinterpret_cast<__nv_bfloat16 *>(p.out)[int64_t(t) * p.M + row] = __float2bfloat16_rn(y);
                        }
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&acc_empty[acc]);
            if (++acc == C::ACC_STAGES) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, 512);
}

// fp32 -> three bf16 parts (hi, mid, lo), each part a contiguous [n] block.
__global__ void k_split_bf16x3(const float *__restrict__ w, int64_t n, __nv_bfloat16 *__restrict__ out)
{
    pdl_enter();
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n / 4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(w) + i);
        const float a[4] = {v.x, v.y, v.z, v.w};
        __nv_bfloat16 h[4], m[4], l[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            h[j] = __float2bfloat16_rn(a[j]);
            const float r1 = a[j] - __bfloat162float(h[j]);
            m[j] = __float2bfloat16_rn(r1);
            l[j] = __float2bfloat16_rn(r1 - __bfloat162float(m[j]));
        }
        reinterpret_cast<uint2 *>(out)[i] = *reinterpret_cast<uint2 *>(h);
        reinterpret_cast<uint2 *>(out + n)[i] = *reinterpret_cast<uint2 *>(m);
        reinterpret_cast<uint2 *>(out + 2 * n)[i] = *reinterpret_cast<uint2 *>(l);
    }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

bool make_bf16_map(CUtensorMap *m, const void *base, uint64_t K, uint64_t rows, uint32_t box_rows)
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return false;
        fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    const cuuint64_t dims[2] = {K, rows};
    const cuuint64_t strides[1] = {K * 2};
    const cuuint32_t box[2] = {64, box_rows};
    const cuuint32_t es[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int sm_count()
{
    int dev = 0, n = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    return n > 0 ? n : 148;
}

template <int NPARTS, int NB, int OUT>
cudaError_t run(const CUtensorMap &a, const CUtensorMap &b, const DenseArgs &args, cudaStream_t st)
{
    using C = DCfg<NPARTS, NB>;
    const size_t smem = 1024 + size_t(C::STAGES) * C::STAGE_BYTES + (2 * C::STAGES + 2 * C::ACC_STAGES) * 8 + 16;
    cudaError_t e = cudaFuncSetAttribute(k_gemm_bf16<NPARTS, NB, OUT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         int(smem));
    if (e != cudaSuccess) return e;
    const int total = args.MT * args.NTL * args.KS;
    const int grid = total < sm_count() ? total : sm_count();
    {
        const cudaError_t le_ = launch_pdl(k_gemm_bf16<NPARTS, NB, OUT>, dim3(grid), dim3(192), smem, st, a, b, args);
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

// Token tile and K split for T tokens, M weight rows, K reduction.
void plan(int T, int M, int K, int &NB, int &KS)
{
    NB = T <= 16 ? 16 : T <= 32 ? 32 : T <= 64 ? 64 : 128;
    const int items = int(ceil_div(M, 128) * ceil_div(T, NB));
    const int chunks = K / 64;
    // split K over the largest divisor of the chunk count that keeps the grid
    // within one wave and every slice at >= 2 chunks
    KS = 1;
    for (int ks = 2; ks <= chunks / 2; ++ks)
        if (chunks % ks == 0 && items * ks <= sm_count()) KS = ks;
}

template <int NPARTS, int OUT>
cudaError_t dispatch(int NB, const CUtensorMap &a, const CUtensorMap &b, const DenseArgs &args, cudaStream_t st)
{
    switch (NB) {
    case 16: return run<NPARTS, 16, OUT>(a, b, args, st);
    case 32: return run<NPARTS, 32, OUT>(a, b, args, st);
    case 64: return run<NPARTS, 64, OUT>(a, b, args, st);
    default: return run<NPARTS, 128, OUT>(a, b, args, st);
    }
}

}  // namespace

int router_kernel_count(int T, int d, int E)
{
    int NB, KS;
    plan(T, E, d, NB, KS);
    return 2;  // GEMM, top-k (with the split-K reduction when K is split)
}

size_t router_scratch_bytes(int T, int d, int E)
{
    int NB, KS;
    plan(T, E, d, NB, KS);
    return KS > 1 ? size_t(round_up(int64_t(KS) * T * E * 4, 256)) : 0;
}

cudaError_t launch_split_router(const float *Wr, int E, int d, uint16_t *Wr3, cudaStream_t st)
{
    const int64_t n = int64_t(E) * d;
    const int64_t blocks = ceil_div(n / 4, 256);
    return launch_pdl(k_split_bf16x3, dim3(unsigned(blocks < 152 * 16 ? blocks : 152 * 16)), dim3(256), 0, st, Wr, n,
                      reinterpret_cast<__nv_bfloat16 *>(Wr3));
}

cudaError_t launch_route(const uint16_t *x, const uint16_t *Wr3, const float *bias, int T, int d, int E, int k,
                         float *logits, int32_t *idx, float *w, void *scratch, int32_t *status, cudaStream_t st,
                         const PermByMask &pm)
{
    if (T == 0) return cudaSuccess;
    const __nv_bfloat16 *w3 = reinterpret_cast<const __nv_bfloat16 *>(Wr3);
    float *partial = static_cast<float *>(scratch);
    cudaError_t e = cudaSuccess;
    int NB, KS;
    plan(T, E, d, NB, KS);
    CUtensorMap ma, mb;
    if (!make_bf16_map(&ma, w3, uint64_t(d), uint64_t(3) * E, 128) ||
        !make_bf16_map(&mb, x, uint64_t(d), uint64_t(T), uint32_t(NB)))
        return cudaErrorInvalidValue;
    DenseArgs a{E, T, d, int(ceil_div(E, 128)), int(ceil_div(T, NB)), KS, d / 64 / KS, bias, logits, status};
    if (KS == 1) {
        if (pm.mask) return cudaErrorInvalidValue;  // the permute rides on the split-K top-k kernel only
        e = dispatch<3, OUT_F32>(NB, ma, mb, a, st);
        if (e != cudaSuccess) return e;
        return launch_topk_softmax(logits, T, E, k, idx, w, st, status);
    }
    a.out = partial;
    a.bias = nullptr;
    e = dispatch<3, OUT_PARTIAL>(NB, ma, mb, a, st);
    if (e != cudaSuccess) return e;
    return launch_reduce_topk(partial, KS, T, E, bias, logits, k, idx, w, st, pm);
}

bool route_can_permute(int T, int d, int E, int k)
{
    int NB, KS;
    plan(T, E, d, NB, KS);
    return KS > 1 && T >= 1 && T <= 64 && E <= 896 && k <= 32;
}

size_t linear_scratch_bytes(int T, int K, int N)
{
    int NB, KS;
    plan(T, N, K, NB, KS);
    return KS > 1 ? size_t(round_up(int64_t(KS) * T * N * 4, 256)) : 0;
}

cudaError_t launch_linear_bf16(const uint16_t *x, const uint16_t *W, int T, int K, int N, uint16_t *out, void *scratch,
                               int32_t *status, cudaStream_t st)
{
    if (T == 0) return cudaSuccess;
    int NB, KS;
    plan(T, N, K, NB, KS);
    KS = 1;  // bf16 output: no split
    CUtensorMap ma, mb;
    if (!make_bf16_map(&ma, W, uint64_t(K), uint64_t(N), 128) ||
        !make_bf16_map(&mb, x, uint64_t(K), uint64_t(T), uint32_t(NB)))
        return cudaErrorInvalidValue;
    (void)scratch;
    DenseArgs a{N, T, K, int(ceil_div(N, 128)), int(ceil_div(T, NB)), 1, K / 64, nullptr, out, status};
    return dispatch<1, OUT_BF16>(NB, ma, mb, a, st);
}

}  // namespace lmoe
