// Expert FFN on CUDA cores: one warp per (expert, output row), lanes over the
// K blocks, MXFP4 weights and MXFP8 activations decoded in registers, fp32
// accumulation ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "MXFP4 原生支持": dequantisation fused into the matrix product).
//   gate/up: h[q][i] = silu(g) * u  (fp32 scratch), then MXFP8 along I;
//   down:    yp[q][o] = topk_w[perm[q]] * (Wd[e][o] . h^[q]).
#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

__device__ __forceinline__ void decode_e2m1x32(const uint4 codes, float scale, const float *lut, float *out)
{
    const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int n = 0; n < 8; ++n) out[8 * i + n] = lut[(w[i] >> (4 * n)) & 15] * scale;
}

__device__ __forceinline__ float dot_e4m3x32(const uint8_t *codes, float scale, const float *wv)
{
    const uint4 *p = reinterpret_cast<const uint4 *>(codes);
    const uint4 a = __ldg(p), b = __ldg(p + 1);
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float acc = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int n = 0; n < 4; ++n) acc = fmaf(wv[4 * i + n], e4m3_to_f32((w[i] >> (8 * n)) & 0xFF), acc);
    return acc * scale;
}

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}

__device__ __forceinline__ int64_t tc_scale_offset(int64_t m, int r, int b, int RT, int KC)
{
    int rt = r >> 7, rr = r & 127, kc = b >> 2, kb = b & 3;
    return ((m * RT + rt) * KC + kc) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + kb;
}

constexpr int TG = 4;  // tokens per pass

__global__ void __launch_bounds__(256) k_gateup_simt(const uint8_t *__restrict__ xq, const uint8_t *__restrict__ xs,
                                                     const uint8_t *__restrict__ gq, const uint8_t *__restrict__ gs,
                                                     const uint8_t *__restrict__ uq, const uint8_t *__restrict__ us,
                                                     const int32_t *__restrict__ offsets, int E, int d, int I,
                                                     float *__restrict__ h)
{
    __shared__ float lut[16];
    if (threadIdx.x < 16) {
        const int c = threadIdx.x, ex = (c >> 1) & 3, man = c & 1;
        const float mag = ex == 0 ? 0.5f * man : ldexpf(1.f + 0.5f * man, ex - 1);
        lut[c] = (c & 8) ? -mag : mag;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t item = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (item >= int64_t(E) * I) return;
    const int e = int(item / I), i = int(item - int64_t(e) * I);
    const int q0 = offsets[e], q1 = offsets[e + 1];
    if (q0 == q1) return;
    const int Kp = int(round_up(d, 128)), RT = int(ceil_div(I, 128)), KC = Kp / 128, nb = d / 32;
    const int64_t row = int64_t(e) * I + i;
    for (int qb = q0; qb < q1; qb += TG) {
        float ag[TG], au[TG];
#pragma unroll
        for (int n = 0; n < TG; ++n) ag[n] = au[n] = 0.f;
        for (int b = lane; b < nb; b += 32) {
            float wg[32], wu[32];
            decode_e2m1x32(__ldg(reinterpret_cast<const uint4 *>(gq + row * (Kp / 2) + b * 16)),
                           e8m0_to_f32(gs[tc_scale_offset(e, i, b, RT, KC)]), lut, wg);
            decode_e2m1x32(__ldg(reinterpret_cast<const uint4 *>(uq + row * (Kp / 2) + b * 16)),
                           e8m0_to_f32(us[tc_scale_offset(e, i, b, RT, KC)]), lut, wu);
#pragma unroll
            for (int n = 0; n < TG; ++n) {
                const int q = qb + n;
                if (q < q1) {
                    const float sx = e8m0_to_f32(xs[int64_t(q) * nb + b]);
                    ag[n] += dot_e4m3x32(xq + int64_t(q) * d + b * 32, sx, wg);
                    au[n] += dot_e4m3x32(xq + int64_t(q) * d + b * 32, sx, wu);
                }
            }
        }
#pragma unroll
        for (int n = 0; n < TG; ++n) {
            const float g = warp_sum(ag[n]), u = warp_sum(au[n]);
            const int q = qb + n;
            if (lane == 0 && q < q1) h[int64_t(q) * I + i] = g / (1.f + expf(-g)) * u;
        }
    }
}

// MXFP8 of fp32 rows (one thread per 32-block).
__global__ void k_quant_f32_mxfp8(const float *__restrict__ h, int64_t nblocks, int K, uint8_t *__restrict__ q,
                                  uint8_t *__restrict__ s)
{
    const int nb = K / 32;
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < nblocks; g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = g / nb;
        const int b = int(g - row * nb);
        const float *src = h + row * K + b * 32;
        float v[32];
        uint32_t amax_bits = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            v[i] = src[i];
            amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7FFFFFFFu);
        }
        const uint32_t sb = mx_scale_byte(__uint_as_float(amax_bits), 8);
        const float inv = mx_inv_scale(sb);
        uint32_t c[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) c[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
        uint4 *dst = reinterpret_cast<uint4 *>(q + row * K + b * 32);
        dst[0] = make_uint4(c[0], c[1], c[2], c[3]);
        dst[1] = make_uint4(c[4], c[5], c[6], c[7]);
        s[row * nb + b] = uint8_t(sb);
    }
}

__global__ void __launch_bounds__(256) k_down_simt(const uint8_t *__restrict__ hq, const uint8_t *__restrict__ hs,
                                                   const uint8_t *__restrict__ dq, const uint8_t *__restrict__ ds,
                                                   const int32_t *__restrict__ offsets, const int32_t *__restrict__ perm,
                                                   const float *__restrict__ topk_w, int E, int d, int I,
                                                   float *__restrict__ yp)
{
    __shared__ float lut[16];
    if (threadIdx.x < 16) {
        const int c = threadIdx.x, ex = (c >> 1) & 3, man = c & 1;
        const float mag = ex == 0 ? 0.5f * man : ldexpf(1.f + 0.5f * man, ex - 1);
        lut[c] = (c & 8) ? -mag : mag;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int64_t item = int64_t(blockIdx.x) * 8 + (threadIdx.x >> 5);
    if (item >= int64_t(E) * d) return;
    const int e = int(item / d), o = int(item - int64_t(e) * d);
    const int q0 = offsets[e], q1 = offsets[e + 1];
    if (q0 == q1) return;
    const int Kp = int(round_up(I, 128)), RT = int(ceil_div(d, 128)), KC = Kp / 128, nb = I / 32;
    const int64_t row = int64_t(e) * d + o;
    for (int qb = q0; qb < q1; qb += TG) {
        float acc[TG];
#pragma unroll
        for (int n = 0; n < TG; ++n) acc[n] = 0.f;
        for (int b = lane; b < nb; b += 32) {
            float wd[32];
            decode_e2m1x32(__ldg(reinterpret_cast<const uint4 *>(dq + row * (Kp / 2) + b * 16)),
                           e8m0_to_f32(ds[tc_scale_offset(e, o, b, RT, KC)]), lut, wd);
#pragma unroll
            for (int n = 0; n < TG; ++n) {
                const int q = qb + n;
                if (q < q1) acc[n] += dot_e4m3x32(hq + int64_t(q) * I + b * 32, e8m0_to_f32(hs[int64_t(q) * nb + b]), wd);
            }
        }
#pragma unroll
        for (int n = 0; n < TG; ++n) {
            const float v = warp_sum(acc[n]);
            const int q = qb + n;
            if (lane == 0 && q < q1) yp[int64_t(q) * d + o] = topk_w[perm[q]] * v;
        }
    }
}

}  // namespace

size_t ffn_scratch_bytes(int64_t P, int d, int E, int I)
{
    (void)d; (void)E;
    return size_t(round_up(P * I * 4, 256) + round_up(P * I, 256) + round_up(P * (I / 32), 256));
}

cudaError_t launch_expert_ffn(const FfnArgs &a, cudaStream_t st, cudaEvent_t mid)
{
    if (a.P == 0) return cudaSuccess;
    char *ws = static_cast<char *>(a.scratch);
    float *h = reinterpret_cast<float *>(ws);
    uint8_t *hq = reinterpret_cast<uint8_t *>(ws + round_up(int64_t(a.P) * a.I * 4, 256));
    uint8_t *hs = hq + round_up(int64_t(a.P) * a.I, 256);
    const int64_t n1 = int64_t(a.E) * a.I;
    k_gateup_simt<<<unsigned(ceil_div(n1, 8)), 256, 0, st>>>(a.xq_sorted, a.xs_sorted, a.W->gate_q, a.W->gate_s,
                                                            a.W->up_q, a.W->up_s, a.offsets, a.E, a.d, a.I, h);
    const int64_t nb = int64_t(a.P) * (a.I / 32);
    k_quant_f32_mxfp8<<<unsigned(ceil_div(nb, 256)), 256, 0, st>>>(h, nb, a.I, hq, hs);
    if (mid) {
        cudaError_t e = cudaEventRecord(mid, st);
        if (e != cudaSuccess) return e;
    }
    const int64_t n2 = int64_t(a.E) * a.d;
    k_down_simt<<<unsigned(ceil_div(n2, 8)), 256, 0, st>>>(hq, hs, a.W->down_q, a.W->down_s, a.offsets, a.perm,
                                                          a.topk_w, a.E, a.d, a.I, a.yp);
    return cudaGetLastError();
}

}  // namespace lmoe
