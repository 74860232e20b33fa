// Load-time conversion of an MXFP4 checkpoint ("Kimi K3 Day-0 适配剖析"
// section 三: the checkpoint is converted to the hardware's form layer by
// layer while it loads) and the per-matrix distribution of its E8M0 block
// scales ("SGLang 0.5.17: Kimi K3 原生 MXFP4 推理架构解析", section
// "精度与速度的平衡": the scale factors of each expert block are logged).
//
// The checkpoint's canonical MXFP4 bytes (codes[r][K/2], scales[r][K/32])
// are rearranged, not re-quantised, into the tensor-core layout the expert
// GEMMs read: codes keep their bytes with each row padded to Kp =
// roundup(K, 128) by zero codes; scales move into 512-byte atoms of 128 rows
// x 4 blocks (row 32*j + i, block b at byte 16*i + 4*j + b).  Both kernels
// write every output byte (padding included), so the destination needs no
// clearing, and they are plain streaming copies: one 16-byte code chunk or
// one 4-byte scale word per thread, grid-stride.
#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

// Output code chunk g (16 bytes = 32 elements) of row `row` (over all
// matrices): chunk c < K/32 copies input chunk c, the rest are zero.
__global__ void k_repack_codes(const uint8_t *__restrict__ q, int64_t nchunks, int K, int Kp,
                               uint8_t *__restrict__ q_tc)
{
    pdl_enter();
    const int cin = K / 32, cout = Kp / 32;
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < nchunks; g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t row = g / cout;
        const int c = int(g - row * cout);
        uint4 v = make_uint4(0, 0, 0, 0);
        if (c < cin) v = __ldg(reinterpret_cast<const uint4 *>(q + row * (K / 2)) + c);
        reinterpret_cast<uint4 *>(q_tc + row * (Kp / 2))[c] = v;
    }
}

// Output scale word g: atom a = g / 128 (matrix m, row tile rt, K chunk kc),
// word w = 4*i + j of the atom holds blocks kc*4 .. kc*4+3 of row rt*128 +
// 32*j + i (0 outside the matrix).
__global__ void k_repack_scales(const uint8_t *__restrict__ s, int64_t nwords, int rows, int nb, int RT, int KC,
                                uint32_t *__restrict__ s_tc)
{
    pdl_enter();
    for (int64_t g = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; g < nwords; g += int64_t(gridDim.x) * blockDim.x) {
        const int64_t a = g >> 7;
        const int w = int(g & 127), i = w >> 2, j = w & 3;
        const int64_t m = a / (int64_t(RT) * KC);
        const int rem = int(a - m * RT * KC);
        const int rt = rem / KC, kc = rem - rt * KC;
        const int r = rt * 128 + 32 * j + i;
        uint32_t word = 0;
        if (r < rows) {
            const uint8_t *src = s + (m * rows + r) * nb;
#pragma unroll
            for (int b = 0; b < 4; ++b) {
                const int blk = kc * 4 + b;
                if (blk < nb) word |= uint32_t(__ldg(src + blk)) << (8 * b);
            }
        }
        s_tc[g] = word;
    }
}

// Per matrix, the count of each scale byte value over its rows x K/32
// blocks (one block of threads per matrix, counts in shared memory).
__global__ void __launch_bounds__(256) k_scale_hist(const uint8_t *__restrict__ s, int rows, int nb, int layout, int RT,
                                                    int KC, uint32_t *__restrict__ hist)
{
    pdl_enter();
    __shared__ uint32_t h[256];
    h[threadIdx.x] = 0;
    __syncthreads();
    const int64_t m = blockIdx.x;
    const int64_t n = int64_t(rows) * nb;
    for (int64_t g = threadIdx.x; g < n; g += blockDim.x) {
        const int r = int(g / nb), b = int(g - int64_t(r) * nb);
        int64_t off;
        if (layout == LMOE_LAYOUT_TC)
            off = ((m * RT + (r >> 7)) * KC + (b >> 2)) * 512 + (r & 31) * 16 + ((r & 127) >> 5) * 4 + (b & 3);
        else
            off = m * n + g;
        atomicAdd(&h[__ldg(s + off)], 1u);
    }
    __syncthreads();
    hist[m * 256 + threadIdx.x] = h[threadIdx.x];
}

int grid_for(int64_t n, int threads)
{
    const int64_t g = ceil_div(n, threads);
    return int(g < 1 ? 1 : (g > 152 * 32 ? 152 * 32 : g));
}

}  // namespace

cudaError_t launch_repack_mxfp4(const uint8_t *q, const uint8_t *s, int64_t nmat, int rows, int K, uint8_t *q_tc,
                                uint8_t *s_tc, cudaStream_t st)
{
    const int Kp = int(round_up(K, 128)), RT = int(ceil_div(rows, 128)), KC = Kp / 128;
    const int64_t nchunks = nmat * rows * (Kp / 32), nwords = nmat * RT * KC * 128;
    cudaError_t e = launch_pdl(k_repack_codes, dim3(grid_for(nchunks, 256)), dim3(256), 0, st, q, nchunks, K, Kp, q_tc);
    if (e == cudaSuccess)
        e = launch_pdl(k_repack_scales, dim3(grid_for(nwords, 256)), dim3(256), 0, st, s, nwords, rows, K / 32, RT, KC,
                       reinterpret_cast<uint32_t *>(s_tc));
    return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_scale_histogram(const uint8_t *s, int64_t nmat, int rows, int K, int layout, uint32_t *hist,
                                   cudaStream_t st)
{
    const int Kp = int(round_up(K, 128)), RT = int(ceil_div(rows, 128)), KC = Kp / 128;
    cudaError_t e = launch_pdl(k_scale_hist, dim3(unsigned(nmat)), dim3(256), 0, st, s, rows, K / 32, layout, RT, KC,
                               hist);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace lmoe
