// ssd_prefill_varlen_noalloc: the CUDA-core prefill with its scratch in a
// fixed device array of this library instead of caller-provided workspace.
//
// It is for callers that cannot allocate device memory when they call us: a
// serving engine that reserved all free device memory up front (for its state
// cache) and hands none out afterwards, or a host that only has this C ABI and
// no device allocator of its own.  The scratch lives in one file-scope
// __device__ array of SSD_NOALLOC_SCRATCH_BYTES; every GPU that loads the
// library holds it until the process exits.
#include <cuda.h>

#include <mutex>

#include "common.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_ctx[kMaxDevices];      // context the address below was looked up in
void *g_scratch_addr[kMaxDevices];     // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch array on the current device.  The name of a
// __device__ variable is only a host-side stand-in, so its address is asked
// from the runtime (with that device current) and kept, together with the
// context it belongs to: after a device reset the device has a new primary
// context with the module loaded anew, and the address is looked up again.
cudaError_t scratch_on_current_device(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *ctx = nullptr;  // null until the runtime has made the device's context current
    if (!ssd::current_context(&ctx)) return cudaErrorDeviceUninitialized;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!ctx || !g_scratch_addr[dev] || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);  // sets the primary context up if needed
        if (e != cudaSuccess) return e;
        if (!ssd::current_context(&ctx) || !ctx) return cudaErrorDeviceUninitialized;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

namespace ssd {
// cuCtxGetCurrent, reached through the runtime (the library does not link the driver itself)
bool current_context(void **ctx) {
    using Fn = CUresult (*)(CUcontext *);
    static Fn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        return cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
                       q == cudaDriverEntryPointSuccess
                   ? reinterpret_cast<Fn>(p)
                   : nullptr;
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return false;
    *ctx = c;
    return true;
}
}  // namespace ssd

extern "C" ssd_status_t ssd_prefill_varlen_noalloc(const ssd_prefill_args *a, ssd_stream_t stream) {
    // the same host checks as ssd_prefill_varlen, through its public size query
    if (!a) return SSD_ERR_INVALID_ARG;
    if (ssd_prefill_kernel_count(a) < 0) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens == 0) return SSD_OK;
    if (!ssd::simt_prefill_supported(*a)) return SSD_ERR_UNSUPPORTED;
    const size_t need = ssd::simt_prefill_workspace(*a, nullptr, nullptr);
    if (need > (size_t)SSD_NOALLOC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
    void *base = nullptr;
    if (scratch_on_current_device(&base) != cudaSuccess) return SSD_ERR_CUDA;
    // Every element of the scratch the kernels read is written earlier in the
    // same call, so the previous call's contents need no clearing.
    ssd::PrefillWorkspace ws;
    ssd::simt_prefill_workspace(*a, &ws, base);
    return ssd::simt_prefill_launch(*a, ws, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SSD_OK
               : SSD_ERR_CUDA;
}
