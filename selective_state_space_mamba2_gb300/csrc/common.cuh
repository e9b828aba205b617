// Shared device helpers of the SSD library (internal header).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ssd.h"

namespace ssd {

// ---- element access -------------------------------------------------------
__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float v) {
    return __float2bfloat16_rn(v);
}

template <typename T> __device__ __forceinline__ float ldg_f32(const T *p) { return to_f32(__ldg(p)); }

// Output gate: y * silu(z) = y * z * sigmoid(z) (the optional z argument of the
// chunk-scan call on "[vllm] vLLM Mamba2 SSD 커널 웜업", section
// "mamba_mixer2.py 변경 사항 (핵심)").  The quotient uses the fast approximate
// divide (reciprocal times numerator, about 2 ulp): for z below about -88,
// __expf(-z) is +inf, its reciprocal 0, and the result the right limit, 0.
__device__ __forceinline__ float silu(float v) { return __fdividef(v, 1.f + __expf(-v)); }
__device__ __forceinline__ float silu_gate(float y, float z) { return y * silu(z); }

// ---- the per-token step size ----------------------------------------------
// delta = clamp(softplus(dt + dt_bias), dt_min, dt_max).  softplus(v) is taken
// as v itself above 20, where log1p(exp(v)) - v < 2.1e-9 * v (below fp32
// resolution); CUDA's expf / log1pf are called, not re-derived.
__device__ __forceinline__ float step_delta(float dt_plus_bias, int dt_softplus, float dt_min,
                                            float dt_max) {
    float d = dt_plus_bias;
    if (dt_softplus) d = d > 20.f ? d : log1pf(__expf(d));
    return fminf(fmaxf(d, dt_min), dt_max);
}

// delta = clamp(softplus(v), lo, hi) from the fast exp/log intrinsics:
// softplus(v) = v above 15 (the rest is below e^-15 relative); e - e^2/2 with
// e = exp(v) below -5 (log1p's series; the next term is under 2e-5
// relative there); log(1 + e) in between, where 1 + e >= 1.0067 keeps the
// rounding of the sum under 1e-5 relative.
__device__ __forceinline__ float fast_delta(float v, int dt_softplus, float lo, float hi) {
    float d = v;
    if (dt_softplus && v <= 15.f) {
        const float e = __expf(v);
        d = v < -5.f ? e * (1.f - 0.5f * e) : __logf(1.f + e);
    }
    return fminf(fmaxf(d, lo), hi);
}

// ---- device error word ------------------------------------------------------
__device__ __forceinline__ void report(uint32_t *err, uint32_t bits) {
    if (err) atomicOr(err, bits);
}

// true when `slot` may be accessed; reports out-of-range ids (null is not an error)
__device__ __forceinline__ bool slot_usable(int32_t slot, int32_t null_id, int32_t num_slots,
                                            uint32_t *err) {
    if (slot == null_id) return false;
    if (slot < 0 || slot >= num_slots) {
        report(err, SSD_DEVERR_SLOT);
        return false;
    }
    return true;
}

}  // namespace ssd

// ---- internal launchers (C++ linkage, not part of the ABI) -------------------
namespace ssd {
struct PrefillWorkspace {
    float *delta;        // [H, T]
    double *cumlog;      // [H, T] inclusive in-chunk cumsum of delta * A (fp64: decays are
                         // exponentials of its differences)
    float *chunk_state;  // [K, H, P, N]
    float *state_in;     // [K, H, P, N]
};
size_t simt_prefill_workspace(const ssd_prefill_args &a, PrefillWorkspace *ws, void *base);
cudaError_t simt_prefill_launch(const ssd_prefill_args &a, const PrefillWorkspace &ws,
                                cudaStream_t s);
bool simt_prefill_supported(const ssd_prefill_args &a);

bool tc_prefill_supported(const ssd_prefill_args &a);
int tc_prefill_segments(const ssd_prefill_args &a);
size_t tc_prefill_workspace(const ssd_prefill_args &a);
// after_prep: recorded on s once the prep kernel is queued (before the segment pass and the
// fused kernel), or nullptr; before_fused: recorded right before the fused kernel (after the
// segment pass, if any), or nullptr
cudaError_t tc_prefill_launch(const ssd_prefill_args &a, void *workspace, cudaStream_t s,
                              cudaEvent_t after_prep = nullptr, cudaEvent_t before_fused = nullptr);

bool decode_supported(const ssm_decode_args &a);
cudaError_t decode_launch(const ssm_decode_args &a, cudaStream_t s);

cudaError_t conv1d_launch(const ssd_conv1d_args &a, bool decode, cudaStream_t s);

cudaError_t mamba1_launch(const mamba1_args &a, bool decode, cudaStream_t s);

// The current context (CUcontext) as an opaque handle: false when the driver entry point is
// unavailable; *ctx is null until the runtime has made a context current on this thread.
bool current_context(void **ctx);
}  // namespace ssd
