// lmoe_permute_noalloc: the dispatch permute without any caller-provided
// scratch buffer and without any device allocation.
//
// Who needs this: some callers cannot hand the library a workspace or let it
// allocate.  Examples are plugin or callback code that runs inside another
// runtime whose device memory pool it does not own, and serving loops whose
// device memory is planned once at start-up, where any allocation during a
// step is an error.  For them the permute keeps its block histograms in a
// fixed array that lives in the library itself.
//
// The array below is file-scope device memory, so every GPU that loads the
// library holds it until the process exits.  Its host-side name is not a
// device address: the device address is looked up once per device with
// cudaGetSymbolAddress (the first call on a device does that look-up, and
// the first call after a device reset repeats it; make that call before any
// stream capture).  All calls share the array and
// it keeps the last call's contents, so calls that overlap on the GPU (two
// streams, or two threads) race with each other and must be serialised by the
// caller.
#include <cuda.h>

#include <mutex>

#include "lmoe_internal.cuh"

namespace {

// status word (256 bytes) + block histograms for up to
// LMOE_PERMUTE_NOALLOC_MAX_PAIRS pairs and 2048 experts
constexpr size_t kStatusBytes = 256;
constexpr size_t kScratchBytes =
    kStatusBytes + size_t((LMOE_PERMUTE_NOALLOC_MAX_PAIRS + lmoe::PERMUTE_CHUNK - 1) / lmoe::PERMUTE_CHUNK) * 2048 *
                       sizeof(int32_t);

static __device__ __align__(256) uint8_t g_permute_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void *g_scratch_ptr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};  // the context the address belongs to

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    if (!fn) {
        cudaDriverEntryPointQueryResult q;
        void *f = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(f);
    }
    return fn;
}

// Device address of the array on the current device: looked up once per
// device and context (a device reset makes a new context, in which the
// module may be loaded at another address; the look-up is then repeated).
lmoe_status scratch_on_current_device(uint8_t **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return LMOE_ERR_CUDA;
    CUcontext ctx = nullptr;  // null until the runtime has made the device's context current
    CtxGetCurrentFn get = ctx_get_current();
    if (!get || get(&ctx) != CUDA_SUCCESS) return LMOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!g_scratch_ptr[dev] || !ctx || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_permute_scratch) != cudaSuccess || !p) return LMOE_ERR_CUDA;
        if (get(&ctx) != CUDA_SUCCESS) return LMOE_ERR_CUDA;  // current now
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = static_cast<uint8_t *>(g_scratch_ptr[dev]);
    return LMOE_OK;
}

}  // namespace

extern "C" lmoe_status lmoe_permute_noalloc(const int32_t *topk_idx, const lmoe_dims *dims, int32_t *counts,
                                            int32_t *offsets, int32_t *perm, int32_t *inv, int32_t *device_status,
                                            void *stream)
{
    if (!dims || dims->T < 0 || dims->E <= 0 || dims->E > 2048 || dims->k <= 0 || dims->k > 32 || dims->k > dims->E)
        return LMOE_ERR_INVALID_ARG;
    const int64_t P = int64_t(dims->T) * dims->k;
    if (P > LMOE_PERMUTE_NOALLOC_MAX_PAIRS) return LMOE_ERR_INVALID_ARG;  // beyond the fixed array
    if (!counts || !offsets || (P > 0 && (!topk_idx || !perm || !inv))) return LMOE_ERR_INVALID_ARG;
    uint8_t *scratch = nullptr;
    lmoe_status s = scratch_on_current_device(&scratch);
    if (s != LMOE_OK) return s;
    cudaStream_t st = cudaStream_t(stream);
    int32_t *status = reinterpret_cast<int32_t *>(scratch);
    // the status word must start at zero; the histograms are fully rewritten by every call
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int32_t), st);
    if (e == cudaSuccess)
        e = lmoe::launch_permute(topk_idx, P, dims->E, counts, offsets, perm, inv, scratch + kStatusBytes, status, st);
    if (e == cudaSuccess && device_status)
        e = cudaMemcpyAsync(device_status, status, sizeof(int32_t), cudaMemcpyDeviceToDevice, st);
    if (e != cudaSuccess) return LMOE_ERR_CUDA;
    return LMOE_OK;
}
