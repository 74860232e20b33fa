// Combine ("Kimi K3 Day-0 适配剖析" section 四: collect the expert results back
// by weight): y[t] = bf16( sum_j yp[inv[t*k + j]] ), slot order, fp32 sums.
// The gate weight was already applied by the down-projection epilogue.
#include <cuda_bf16.h>

#include "lmoe_internal.cuh"

namespace lmoe {
namespace {

__global__ void __launch_bounds__(128) k_combine(const float *__restrict__ yp, const int32_t *__restrict__ inv, int T,
                                                 int d, int k, uint16_t *__restrict__ y, int inv_early)
{
    __shared__ int32_t rows[32];
    const int t = blockIdx.x;
    // inv_early: inv was complete before the kernel this one follows started
    // (inside the layer call), so it is read before waiting for that kernel
    if (inv_early && threadIdx.x < k) rows[threadIdx.x] = __ldg(inv + int64_t(t) * k + threadIdx.x);
    pdl_enter();
    if (!inv_early && threadIdx.x < k) rows[threadIdx.x] = __ldg(inv + int64_t(t) * k + threadIdx.x);
    __syncthreads();
    const int nv = d / 4;
    for (int c = threadIdx.x + blockIdx.y * blockDim.x; c < nv; c += blockDim.x * gridDim.y) {
        // the k rows' loads go out in batches of 16 before they are summed (in
        // slot order), so each batch costs one memory latency, not sixteen
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int j0 = 0; j0 < k; j0 += 16) {
            float4 v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                v[j] = j0 + j < k ? __ldcg(reinterpret_cast<const float4 *>(yp + int64_t(rows[j0 + j]) * d) + c)
                                  : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                if (j0 + j < k) {
                    acc.x += v[j].x;
                    acc.y += v[j].y;
                    acc.z += v[j].z;
                    acc.w += v[j].w;
                }
            }
        }
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 out;
        out.x = *reinterpret_cast<uint32_t *>(&lo);
        out.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(y + int64_t(t) * d)[c] = out;
    }
}

// fused combine's last step: the fp32 per-token sums rounded to bf16
__global__ void __launch_bounds__(256) k_acc_to_bf16(const float4 *__restrict__ acc, int64_t n4, uint2 *__restrict__ y)
{
    pdl_enter();
    for (int64_t i = blockIdx.x * int64_t(blockDim.x) + threadIdx.x; i < n4; i += int64_t(gridDim.x) * blockDim.x) {
        const float4 v = __ldg(acc + i);
        __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y);
        __nv_bfloat162 hi = __floats2bfloat162_rn(v.z, v.w);
        uint2 out;
        out.x = *reinterpret_cast<uint32_t *>(&lo);
        out.y = *reinterpret_cast<uint32_t *>(&hi);
        y[i] = out;
    }
}

}  // namespace

cudaError_t launch_acc_to_bf16(const float *acc, int64_t n, uint16_t *y, cudaStream_t st)
{
    const int64_t n4 = n / 4;
    if (n4 == 0) return cudaSuccess;
    const int64_t blocks = ceil_div(n4, 256);
    return launch_pdl(k_acc_to_bf16, dim3(unsigned(blocks < 152 * 16 ? blocks : 152 * 16)), dim3(256), 0, st,
                      reinterpret_cast<const float4 *>(acc), n4, reinterpret_cast<uint2 *>(y));
}

cudaError_t launch_combine(const float *yp, const int32_t *inv, int T, int d, int k, uint16_t *y, cudaStream_t st,
                           bool inv_early)
{
    if (T == 0) return cudaSuccess;
    const int ysplit = T >= 1024 ? 1 : (T >= 128 ? 2 : 7);  // enough CTAs for small T
    return launch_pdl(k_combine, dim3(T, ysplit), dim3(128), 0, st, yp, inv, T, d, k, y, inv_early ? 1 : 0);
}

}  // namespace lmoe
