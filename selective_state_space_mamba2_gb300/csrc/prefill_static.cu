// ssd_prefill_varlen_noalloc: the CUDA-core prefill with its scratch in a
// fixed device array of this library instead of caller-provided workspace.
//
// It is for callers that cannot allocate device memory when they call us: a
// serving engine that reserved all free device memory up front (for its state
// cache) and hands none out afterwards, or a host that only has this C ABI and
// no device allocator of its own.  The scratch lives in one file-scope
// __device__ array of SSD_NOALLOC_SCRATCH_BYTES; every GPU that loads the
// library holds it until the process exits.
#include <mutex>

#include "common.cuh"

namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[SSD_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void *g_scratch_addr[kMaxDevices];  // device address of g_noalloc_scratch, per device ordinal

// Device address of the scratch array on the current device.  The name of a
// __device__ variable is only a host-side stand-in, so its address is asked
// from the runtime once per device (with that device current) and kept.
cudaError_t scratch_on_current_device(void **addr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

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
