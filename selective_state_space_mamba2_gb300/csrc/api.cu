// C-ABI entry points: host-side argument checks, workspace carving, dispatch.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "common.cuh"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

ssd_status_t from_cuda(cudaError_t e) { return e == cudaSuccess ? SSD_OK : SSD_ERR_CUDA; }

bool dtype_ok(int32_t d) { return d == SSD_F32 || d == SSD_BF16; }

bool limits_ok(float lo, float hi) { return !std::isnan(lo) && !std::isnan(hi) && lo <= hi; }

// sizes shared by prefill and decode
bool dims_ok(int32_t H, int32_t P, int32_t N, int32_t G) {
    return H > 0 && P > 0 && N > 0 && G > 0 && H % G == 0 && P <= 256 && N <= 256;
}

ssd_status_t check_prefill(const ssd_prefill_args *a) {
    if (!a) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens < 0 || a->num_seqs < 0 || a->num_chunks < 0) return SSD_ERR_INVALID_ARG;
    if (!dims_ok(a->nheads, a->headdim, a->dstate, a->ngroups)) return SSD_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype) || !limits_ok(a->dt_min, a->dt_max)) return SSD_ERR_INVALID_ARG;
    if (a->wait_limit_cycles < 0) return SSD_ERR_INVALID_ARG;
    if (a->num_chunks > 0 && (a->total_tokens == 0 || a->num_seqs == 0)) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens > 0 && a->num_chunks == 0) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens == 0) return SSD_OK;
    if (!a->x || !a->dt || !a->B || !a->C || !a->A || !a->y || !a->cu_seqlens ||
        !a->cu_chunk_seqlens || !a->last_chunk_indices)
        return SSD_ERR_INVALID_ARG;
    if (!aligned16(a->x) || !aligned16(a->B) || !aligned16(a->C) || !aligned16(a->y) || (a->z && !aligned16(a->z)))
        return SSD_ERR_INVALID_ARG;
    if ((a->init_slot || a->chunk_slot) && (!a->state_cache || a->num_slots <= 0 || !aligned16(a->state_cache)))
        return SSD_ERR_INVALID_ARG;
    return SSD_OK;
}

}  // namespace

extern "C" const char *ssd_status_string(ssd_status_t s) {
    switch (s) {
        case SSD_OK: return "SSD_OK";
        case SSD_ERR_INVALID_ARG: return "SSD_ERR_INVALID_ARG";
        case SSD_ERR_UNSUPPORTED: return "SSD_ERR_UNSUPPORTED";
        case SSD_ERR_WORKSPACE: return "SSD_ERR_WORKSPACE";
        case SSD_ERR_CUDA: return "SSD_ERR_CUDA";
    }
    return "SSD_ERR_UNKNOWN";
}

extern "C" int32_t ssd_abi_version(void) { return SSD_ABI_VERSION; }

extern "C" size_t ssd_prefill_workspace_size(const ssd_prefill_args *a) {
    if (check_prefill(a) != SSD_OK) return 0;
    if (a->total_tokens == 0) return 0;
    if (ssd::tc_prefill_supported(*a)) return ssd::tc_prefill_workspace(*a);
    return ssd::simt_prefill_workspace(*a, nullptr, nullptr);
}

extern "C" int32_t ssd_prefill_kernel_count(const ssd_prefill_args *a) {
    if (check_prefill(a) != SSD_OK) return -1;
    if (a->total_tokens == 0) return 0;
    return ssd::tc_prefill_supported(*a) ? (ssd::tc_prefill_segments(*a) > 1 ? 3 : 2) : 4;
}

namespace {

ssd_status_t check_decode(const ssm_decode_args *a) {
    if (!a) return SSD_ERR_INVALID_ARG;
    if (a->batch < 0 || a->tokens_per_req < 1 || a->state_indices_cols < a->tokens_per_req)
        return SSD_ERR_INVALID_ARG;
    if (!dims_ok(a->nheads, a->headdim, a->dstate, a->ngroups)) return SSD_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype) || !limits_ok(a->dt_min, a->dt_max)) return SSD_ERR_INVALID_ARG;
    if (a->batch == 0) return SSD_OK;
    if (!a->x || !a->dt || !a->B || !a->C || !a->A || !a->y || !a->state_cache || !a->state_indices ||
        a->num_slots <= 0)
        return SSD_ERR_INVALID_ARG;
    if (!aligned16(a->state_cache) || a->dstate % 4 != 0) return SSD_ERR_INVALID_ARG;
    if (!ssd::decode_supported(*a)) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

// The prefill's workspace check and launch.  after_prep and before_fused as for
// tc_prefill_launch; on the CUDA-core path before_fused is recorded before its first kernel and
// after_prep not at all.
ssd_status_t prefill_checked_launch(const ssd_prefill_args *a, void *workspace, size_t workspace_bytes,
                                    cudaStream_t cs, cudaEvent_t after_prep, cudaEvent_t before_fused = nullptr) {
    // bf16 with headdim 64 and dstate 128: the fused tensor-core kernel
    if (ssd::tc_prefill_supported(*a)) {
        if (!workspace || workspace_bytes < ssd::tc_prefill_workspace(*a) ||
            (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return SSD_ERR_WORKSPACE;
        return from_cuda(ssd::tc_prefill_launch(*a, workspace, cs, after_prep, before_fused));
    }
    if (!ssd::simt_prefill_supported(*a)) return SSD_ERR_UNSUPPORTED;
    const size_t need = ssd::simt_prefill_workspace(*a, nullptr, nullptr);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
        return SSD_ERR_WORKSPACE;
    ssd::PrefillWorkspace ws;
    ssd::simt_prefill_workspace(*a, &ws, workspace);
    if (before_fused && cudaEventRecord(before_fused, cs) != cudaSuccess) return SSD_ERR_CUDA;
    return from_cuda(ssd::simt_prefill_launch(*a, ws, cs));
}

// ssd_mixed_step's streams and events, one set per device, made in the context current at the
// time and made again when a later call finds another context there (after a device reset).
struct MixedSet {
    void *ctx = nullptr;
    cudaStream_t hi = nullptr, lo = nullptr;  // prefill (greatest priority), decode (least)
    cudaEvent_t fork = nullptr, prep = nullptr, hi_done = nullptr, lo_done = nullptr;
};
constexpr int kMaxDevices = 64;
std::mutex g_mixed_mutex;  // held from the lookup to the last event of a call
MixedSet g_mixed[kMaxDevices];

cudaError_t mixed_set(MixedSet **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    void *ctx = nullptr;
    if (!ssd::current_context(&ctx)) return cudaErrorDeviceUninitialized;
    if (!ctx) {  // no context current on this thread yet: make the device's primary one current
        e = cudaFree(nullptr);
        if (e != cudaSuccess) return e;
        if (!ssd::current_context(&ctx) || !ctx) return cudaErrorDeviceUninitialized;
    }
    MixedSet &m = g_mixed[dev];
    if (m.ctx != ctx) {  // first call here, or the old context is gone: its handles went with it
        MixedSet n;
        int least = 0, greatest = 0;
        e = cudaDeviceGetStreamPriorityRange(&least, &greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&n.hi, cudaStreamNonBlocking, greatest);
        if (e == cudaSuccess) e = cudaStreamCreateWithPriority(&n.lo, cudaStreamNonBlocking, least);
        for (cudaEvent_t *ev : {&n.fork, &n.prep, &n.hi_done, &n.lo_done})
            if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        n.ctx = ctx;
        m = n;
    }
    *out = &m;
    return cudaSuccess;
}

}  // namespace

extern "C" ssd_status_t ssd_prefill_varlen(const ssd_prefill_args *a, void *workspace,
                                           size_t workspace_bytes, ssd_stream_t stream) {
    const ssd_status_t st = check_prefill(a);
    if (st != SSD_OK || a->total_tokens == 0) return st;
    return prefill_checked_launch(a, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

extern "C" ssd_status_t ssd_prefill_varlen_marked(const ssd_prefill_args *a, void *workspace, size_t workspace_bytes,
                                                  ssd_stream_t stream, void *event_before_fused) {
    const ssd_status_t st = check_prefill(a);
    if (st != SSD_OK || a->total_tokens == 0) return st;
    return prefill_checked_launch(a, workspace, workspace_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr,
                                  static_cast<cudaEvent_t>(event_before_fused));
}

extern "C" ssd_status_t ssm_decode_update(const ssm_decode_args *a, ssd_stream_t stream) {
    const ssd_status_t st = check_decode(a);
    if (st != SSD_OK || a->batch == 0) return st;
    return from_cuda(ssd::decode_launch(*a, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" ssd_status_t ssd_mixed_step(const ssd_prefill_args *prefill, void *workspace, size_t workspace_bytes,
                                       const ssm_decode_args *decode, ssd_stream_t stream) {
    ssd_status_t st = check_prefill(prefill);
    if (st != SSD_OK) return st;
    st = check_decode(decode);
    if (st != SSD_OK) return st;
    const cudaStream_t cs = reinterpret_cast<cudaStream_t>(stream);
    const bool has_prefill = prefill->total_tokens > 0, has_decode = decode->batch > 0;
    if (has_prefill && !ssd::tc_prefill_supported(*prefill) && !ssd::simt_prefill_supported(*prefill))
        return SSD_ERR_UNSUPPORTED;
    if (has_prefill) {
        const size_t need = ssd::tc_prefill_supported(*prefill) ? ssd::tc_prefill_workspace(*prefill)
                                                                : ssd::simt_prefill_workspace(*prefill, nullptr, nullptr);
        if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
            return SSD_ERR_WORKSPACE;
    }
    if (!has_decode) return has_prefill ? prefill_checked_launch(prefill, workspace, workspace_bytes, cs, nullptr) : SSD_OK;
    if (!has_prefill) return from_cuda(ssd::decode_launch(*decode, cs));

    std::lock_guard<std::mutex> lock(g_mixed_mutex);
    MixedSet *m = nullptr;
    cudaError_t e = mixed_set(&m);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    // fork: both streams start after the work queued on `stream` so far
    e = cudaEventRecord(m->fork, cs);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(m->hi, m->fork, 0);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    // The decode starts once the prefill's prep kernel is done: the CUDA-core path records
    // nothing there, so it waits for the fork alone (recorded again on hi for the same effect).
    e = cudaEventRecord(m->prep, m->hi);
    if (e != cudaSuccess) return SSD_ERR_CUDA;
    st = prefill_checked_launch(prefill, workspace, workspace_bytes, m->hi, m->prep);
    // join the hi stream back even when the prefill failed to launch, so that `stream` is left
    // ordered after whatever did get queued
    e = cudaStreamWaitEvent(m->lo, m->prep, 0);
    if (e == cudaSuccess && st == SSD_OK) e = ssd::decode_launch(*decode, m->lo);
    cudaError_t j = cudaEventRecord(m->hi_done, m->hi);
    if (j == cudaSuccess) j = cudaEventRecord(m->lo_done, m->lo);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(cs, m->hi_done, 0);
    if (j == cudaSuccess) j = cudaStreamWaitEvent(cs, m->lo_done, 0);
    if (st != SSD_OK) return st;
    return e == cudaSuccess && j == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}

namespace {

ssd_status_t check_conv(const ssd_conv1d_args *a, bool decode) {
    if (!a) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens < 0 || a->num_seqs < 0 || a->num_chunks < 0) return SSD_ERR_INVALID_ARG;
    if (a->dim_x < 0 || a->dim_bc < 0 || a->dim_x % 8 != 0 || a->dim_bc % 8 != 0 || a->dim_x + a->dim_bc == 0)
        return SSD_ERR_INVALID_ARG;
    if (a->width < 2 || a->width > 4 || (a->activation != 0 && a->activation != 1)) return SSD_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return SSD_ERR_INVALID_ARG;
    if (decode && (a->tokens_per_req < 1 || (int64_t)a->num_seqs * a->tokens_per_req != a->total_tokens))
        return SSD_ERR_INVALID_ARG;
    if (a->total_tokens == 0 && a->num_seqs == 0) return SSD_OK;
    if (!a->xbc || !a->weight || !aligned16(a->xbc) || !aligned16(a->weight)) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens > 0 && (!a->x_out || !a->B_out || !a->C_out || !aligned16(a->x_out) ||
                                !aligned16(a->B_out) || !aligned16(a->C_out)))
        return SSD_ERR_INVALID_ARG;
    if (!decode) {
        if (!a->cu_seqlens) return SSD_ERR_INVALID_ARG;
        if (a->chunk_slot && (!a->cu_chunk_seqlens || !a->last_chunk_indices || a->num_chunks <= 0))
            return SSD_ERR_INVALID_ARG;
    } else if (!a->init_slot) {
        return SSD_ERR_INVALID_ARG;
    }
    const bool uses_state = a->init_slot || (!decode && (a->out_slot || a->chunk_slot));
    if (uses_state && (!a->conv_state || a->num_slots <= 0 || !aligned16(a->conv_state))) return SSD_ERR_INVALID_ARG;
    return SSD_OK;
}

}  // namespace

extern "C" ssd_status_t ssd_conv1d_varlen(const ssd_conv1d_args *a, ssd_stream_t stream) {
    const ssd_status_t st = check_conv(a, false);
    if (st != SSD_OK || a->num_seqs == 0) return st;
    return from_cuda(ssd::conv1d_launch(*a, false, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" ssd_status_t ssd_conv1d_update(const ssd_conv1d_args *a, ssd_stream_t stream) {
    const ssd_status_t st = check_conv(a, true);
    if (st != SSD_OK || a->num_seqs == 0) return st;
    return from_cuda(ssd::conv1d_launch(*a, true, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

ssd_status_t check_mamba1(const mamba1_args *a, bool decode) {
    if (!a) return SSD_ERR_INVALID_ARG;
    if (a->total_tokens < 0 || a->num_seqs < 0 || a->num_chunks < 0) return SSD_ERR_INVALID_ARG;
    if (a->dim <= 0 || a->ngroups <= 0 || a->dim % a->ngroups != 0) return SSD_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype) || !limits_ok(a->dt_min, a->dt_max)) return SSD_ERR_INVALID_ARG;
    if (a->dim % 64 != 0 || (a->dim / a->ngroups) % 64 != 0 || (a->dstate != 8 && a->dstate != 16))
        return SSD_ERR_UNSUPPORTED;
    if (decode) {
        if (a->tokens_per_req < 1 || a->state_indices_cols < a->tokens_per_req ||
            (int64_t)a->num_seqs * a->tokens_per_req != a->total_tokens)
            return SSD_ERR_INVALID_ARG;
    } else {
        if (a->num_chunks > 0 && (a->total_tokens == 0 || a->num_seqs == 0)) return SSD_ERR_INVALID_ARG;
        if (a->total_tokens > 0 && a->num_chunks == 0) return SSD_ERR_INVALID_ARG;
    }
    if (a->total_tokens == 0) return SSD_OK;
    if (!a->x || !a->dt || !a->B || !a->C || !a->A || !a->y) return SSD_ERR_INVALID_ARG;
    if (!aligned16(a->x) || !aligned16(a->dt) || !aligned16(a->B) || !aligned16(a->C) || !aligned16(a->y) ||
        !aligned16(a->A) || (a->z && !aligned16(a->z)))
        return SSD_ERR_INVALID_ARG;
    if (decode) {
        if (!a->state_indices || !a->state_cache || a->num_slots <= 0 || !aligned16(a->state_cache))
            return SSD_ERR_INVALID_ARG;
    } else {
        if (!a->cu_seqlens || !a->cu_chunk_seqlens || !a->last_chunk_indices) return SSD_ERR_INVALID_ARG;
        if ((a->init_slot || a->chunk_slot) && (!a->state_cache || a->num_slots <= 0 || !aligned16(a->state_cache)))
            return SSD_ERR_INVALID_ARG;
    }
    if (a->num_seqs > 0 && (int64_t)a->dim / 64 > 65535) return SSD_ERR_UNSUPPORTED;
    return SSD_OK;
}

}  // namespace

extern "C" ssd_status_t mamba1_scan_varlen(const mamba1_args *a, ssd_stream_t stream) {
    const ssd_status_t st = check_mamba1(a, false);
    if (st != SSD_OK || a->total_tokens == 0 || a->num_seqs == 0) return st;
    return from_cuda(ssd::mamba1_launch(*a, false, reinterpret_cast<cudaStream_t>(stream)));
}

extern "C" ssd_status_t mamba1_state_update(const mamba1_args *a, ssd_stream_t stream) {
    const ssd_status_t st = check_mamba1(a, true);
    if (st != SSD_OK || a->num_seqs == 0) return st;
    return from_cuda(ssd::mamba1_launch(*a, true, reinterpret_cast<cudaStream_t>(stream)));
}
