// MX block quantisation kernels: fp32 weights -> MXFP4 (load-time conversion,
// "Kimi K3 Day-0 适配剖析" section 三) and bf16 activations -> MXFP8
// ("从Kimi K3到MiniMax-H3" section 二, first layer: 4-bit weights meet
// higher-precision activations).  One thread per block of 32 elements: it
// reads the block with 16-byte loads, takes amax, derives the E8M0 byte and
// converts with the hardware round-to-nearest-even instructions.
#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

// Scale byte position of (matrix m, row r, block b) in the tensor-core layout:
// 512-byte atoms of 128 rows x 4 blocks; inside an atom row 32*j + i, block
// kb sits at byte 16*i + 4*j + kb.
__device__ __forceinline__ int64_t tc_scale_offset(int64_t m, int r, int b, int RT, int KC)
{
    int rt = r >> 7, rr = r & 127, kc = b >> 2, kb = b & 3;
    return ((m * RT + rt) * KC + kc) * 512 + (rr & 31) * 16 + (rr >> 5) * 4 + kb;
}

__global__ void k_quant_mxfp4(const float *__restrict__ w, int64_t nblocks, int rows, int K, uint8_t *__restrict__ q,
                              uint8_t *__restrict__ s, int layout, int Kp, int RT, int KC)
{
    pdl_enter();
    const int nb = K / 32;
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < nblocks; g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = g / nb;  // row over all matrices
        const int b = int(g - row * nb);
        const float4 *src = reinterpret_cast<const float4 *>(w + row * K + b * 32);
        float v[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float4 t = __ldg(src + i);
            v[4 * i] = t.x; v[4 * i + 1] = t.y; v[4 * i + 2] = t.z; v[4 * i + 3] = t.w;
        }
        uint32_t amax_bits = 0;
#pragma unroll
        for (int i = 0; i < 32; ++i) amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7FFFFFFFu);
        const uint32_t sb = mx_scale_byte(__uint_as_float(amax_bits), 2);
        const float inv = mx_inv_scale(sb);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] *= inv;
        uint4 codes;
        codes.x = e2m1x8(v);
        codes.y = e2m1x8(v + 8);
        codes.z = e2m1x8(v + 16);
        codes.w = e2m1x8(v + 24);
        if (layout == LMOE_LAYOUT_TC) {
            const int64_t m = row / rows;
            const int r = int(row - m * rows);
            *reinterpret_cast<uint4 *>(q + row * (Kp / 2) + b * 16) = codes;
            s[tc_scale_offset(m, r, b, RT, KC)] = uint8_t(sb);
        } else {
            *reinterpret_cast<uint4 *>(q + row * (K / 2) + b * 16) = codes;
            s[row * nb + b] = uint8_t(sb);
        }
    }
}

// One MXFP8 block: 32 bf16 -> 32 e4m3 codes (two uint4) + scale byte.
__device__ __forceinline__ uint32_t quant_block_e4m3(const uint16_t *src, uint4 &lo, uint4 &hi)
{
    const uint4 *p = reinterpret_cast<const uint4 *>(src);
    uint4 raw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) raw[i] = __ldg(p + i);
    float v[32];
    const uint32_t *rw = reinterpret_cast<const uint32_t *>(raw);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        v[2 * i] = __uint_as_float(rw[i] << 16);
        v[2 * i + 1] = __uint_as_float(rw[i] & 0xFFFF0000u);
    }
    uint32_t amax_bits = 0;
#pragma unroll
    for (int i = 0; i < 32; ++i) amax_bits = max(amax_bits, __float_as_uint(v[i]) & 0x7FFFFFFFu);
    const uint32_t sb = mx_scale_byte(__uint_as_float(amax_bits), 8);
    const float inv = mx_inv_scale(sb);
    uint32_t c[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) c[i] = e4m3x4(v[4 * i] * inv, v[4 * i + 1] * inv, v[4 * i + 2] * inv, v[4 * i + 3] * inv);
    lo = make_uint4(c[0], c[1], c[2], c[3]);
    hi = make_uint4(c[4], c[5], c[6], c[7]);
    return sb;
}

__global__ void k_quant_mxfp8(const uint16_t *__restrict__ x, int64_t nblocks, int K, uint8_t *__restrict__ q,
                              uint8_t *__restrict__ s)
{
    pdl_enter();
    const int nb = K / 32;
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < nblocks; g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = g / nb;
        const int b = int(g - row * nb);
        uint4 lo, hi;
        const uint32_t sb = quant_block_e4m3(x + row * K + b * 32, lo, hi);
        uint4 *dst = reinterpret_cast<uint4 *>(q + row * K + b * 32);
        dst[0] = lo;
        dst[1] = hi;
        s[row * nb + b] = uint8_t(sb);
    }
}

int grid_for(int64_t n, int threads)
{
    int64_t g = ceil_div(n, threads);
    return int(g < 1 ? 1 : (g > 152 * 64 ? 152 * 64 : g));
}

}  // namespace

cudaError_t launch_quant_mxfp4(const float *w, int64_t nmat, int rows, int K, uint8_t *q, uint8_t *s, int layout,
                               cudaStream_t st)
{
    const int64_t nblocks = nmat * rows * (K / 32);
    const int Kp = int(round_up(K, 128)), RT = int(ceil_div(rows, 128)), KC = Kp / 128;
    if (layout == LMOE_LAYOUT_TC) {
        // padding codes and padding / out-of-matrix scale bytes are zero
        cudaError_t e = cudaSuccess;
        if (Kp != K) e = cudaMemsetAsync(q, 0, size_t(nmat) * rows * (Kp / 2), st);
        if (e == cudaSuccess && (Kp != K || RT * 128 != rows))
            e = cudaMemsetAsync(s, 0, size_t(nmat) * RT * KC * 512, st);
        if (e != cudaSuccess) return e;
    }
    if (nblocks == 0) return cudaSuccess;
    {
        const cudaError_t le_ = launch_pdl(k_quant_mxfp4, dim3(grid_for(nblocks, 256)), dim3(256), 0, st, w, nblocks, rows, K, q, s, layout, Kp, RT, KC);
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

cudaError_t launch_quant_mxfp8(const uint16_t *x, int64_t rows, int K, uint8_t *q, uint8_t *s, cudaStream_t st)
{
    const int64_t nblocks = rows * (K / 32);
    if (nblocks == 0) return cudaSuccess;
    {
        const cudaError_t le_ = launch_pdl(k_quant_mxfp8, dim3(grid_for(nblocks, 256)), dim3(256), 0, st, x, nblocks, K, q, s);
        if (le_ != cudaSuccess) return le_;
    }
    return cudaGetLastError();
}

}  // namespace lmoe
