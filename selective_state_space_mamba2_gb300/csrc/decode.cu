// Decode state update: one CTA per (request, head), state held in registers.
//
// "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링": decode is a sequential
// update ("왜 이 설계인가" item 2) through the state-index table of
// "MetadataBuilder 초기화"; padded CUDA-graph rows hold NULL_BLOCK_ID
// ("CUDA Graph 지원") and are skipped; with speculative tokens,
// num_accepted_tokens selects the checkpoint to resume from ("왜 이 설계인가"
// item 4) and every token's state is stored to its own column.
//
// Memory behaviour: per live (request, head) the fp32 state [P, N] is read
// once (float4, a warp covers 512 contiguous bytes) and written once per
// token whose column slot is not null.  That traffic is the whole algorithmic
// cost, so the kernel is HBM-bound as long as the arithmetic per state element
// (one FMA pair for the update, one for y) stays a few instructions: the
// dstate = 128 instance has fixed indexing, reads B and C once per token and
// reduces a warp's rows for y in one transposing shuffle pass; the general
// instance serves the other dstate values.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;
constexpr int kTokBatch = 8;  // tokens whose inputs are staged together

// Shared memory of one CTA: per staged token, x and y [P], B and C [N] and delta.
__host__ __device__ inline size_t decode_smem_bytes(int P, int N) {
    return (size_t)kTokBatch * (2 * P + 2 * N + 1) * sizeof(float);
}

// At least 4 resident CTAs per SM (at most 64 registers) while the state takes up to 32
// floats per thread: the kernel is HBM-bound, and occupancy is what keeps enough state loads
// in flight.  The 64-float case keeps its registers (2 CTAs per SM).
//
// The tokens of a request are taken in batches of up to kTokBatch: their x, B, C and delta are
// loaded together (one memory latency per batch, not per token), and each token reduces into its
// own y row, so the tokens of a batch follow each other with no barrier in between.
template <typename Tin, int VPT, bool kGate>
__global__ void __launch_bounds__(kThreads, VPT >= 16 ? 2 : 4)
    ssm_decode_kernel(const ssm_decode_args a) {
    const int r = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x;
    const int H = a.nheads, P = a.headdim, N = a.dstate;
    const int g = h / (H / a.ngroups);
    const int tpr = a.tokens_per_req;

    const int col = a.num_accepted_tokens ? a.num_accepted_tokens[r] : 0;
    if (col < 0 || col >= a.state_indices_cols) {
        if (tid == 0 && h == 0) report(a.err_word, SSD_DEVERR_COLUMN);
        return;
    }
    const int32_t *row_slots = a.state_indices + (size_t)r * a.state_indices_cols;
    const int32_t rs = row_slots[col];
    if (rs == a.null_block_id) return;  // CUDA-graph padding row
    if (rs < 0 || rs >= a.num_slots) {
        if (tid == 0 && h == 0) report(a.err_word, SSD_DEVERR_SLOT);
        return;
    }

    extern __shared__ __align__(16) float dsm[];
    float *sx = dsm;                   // [kTokBatch][P]
    float *sy = sx + kTokBatch * P;    // [kTokBatch][P]
    float *sB = sy + kTokBatch * P;    // [kTokBatch][N]
    float *sC = sB + kTokBatch * N;    // [kTokBatch][N]
    float *sD = sC + kTokBatch * N;    // [kTokBatch] delta

    const int PN = P * N;
    const int nvec = PN >> 2;  // float4 chunks; N % 4 == 0
    const size_t head_off = (size_t)h * PN;
    float4 s[VPT];
    {
        const float4 *src = reinterpret_cast<const float4 *>(a.state_cache + (size_t)rs * H * PN + head_off);
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int e = tid + i * kThreads;
            s[i] = e < nvec ? src[e] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    // rows of dstate/4 chunks: a segment of `seg` lanes shares one p
    const int quads = N >> 2;
    const int seg = quads < 32 ? quads : 32;

    const float A = a.A[h];
    const float Dh = a.D ? a.D[h] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *dtp = static_cast<const Tin *>(a.dt);
    const Tin *Bp = static_cast<const Tin *>(a.B);
    const Tin *Cp = static_cast<const Tin *>(a.C);
    const Tin *z = static_cast<const Tin *>(a.z);  // output gate or NULL
    Tin *y = static_cast<Tin *>(a.y);

    for (int k0 = 0; k0 < tpr; k0 += kTokBatch) {
        const int kb = min(kTokBatch, tpr - k0);
        __syncthreads();  // the previous batch's readers of the staging arrays are done
        for (int j = tid; j < kb * P; j += kThreads) {
            const int kk = j / P, pp = j - kk * P;
            const size_t row = (size_t)r * tpr + k0 + kk;
            sx[kk * P + pp] = ldg_f32(x + (row * H + h) * P + pp);
            sy[kk * P + pp] = 0.f;
        }
        for (int j = tid; j < kb * N; j += kThreads) {
            const int kk = j / N, nn = j - kk * N;
            const size_t row = (size_t)r * tpr + k0 + kk;
            sB[kk * N + nn] = ldg_f32(Bp + (row * a.ngroups + g) * N + nn);
            sC[kk * N + nn] = ldg_f32(Cp + (row * a.ngroups + g) * N + nn);
        }
        if (tid < kb) {
            const size_t row = (size_t)r * tpr + k0 + tid;
            sD[tid] = step_delta(ldg_f32(dtp + row * H + h) + bias, a.dt_softplus, a.dt_min, a.dt_max);
        }
        __syncthreads();
        for (int kk = 0; kk < kb; ++kk) {
            const float delta = sD[kk];
            const float decay = __expf(delta * A);
            const float *xk = sx + kk * P, *Bk = sB + kk * N, *Ck = sC + kk * N;
#pragma unroll
            for (int i = 0; i < VPT; ++i) {
                const int e = tid + i * kThreads;
                float part = 0.f;
                int p = 0;
                if (e < nvec) {
                    p = e / quads;
                    const int n = (e - p * quads) << 2;
                    const float dx = delta * xk[p];
                    const float4 b4 = *reinterpret_cast<const float4 *>(Bk + n);
                    const float4 c4 = *reinterpret_cast<const float4 *>(Ck + n);
                    s[i].x = fmaf(decay, s[i].x, dx * b4.x);
                    s[i].y = fmaf(decay, s[i].y, dx * b4.y);
                    s[i].z = fmaf(decay, s[i].z, dx * b4.z);
                    s[i].w = fmaf(decay, s[i].w, dx * b4.w);
                    part = s[i].x * c4.x + s[i].y * c4.y + s[i].z * c4.z + s[i].w * c4.w;
                }
                // segmented reduction over the lanes that share p
                for (int off = seg >> 1; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
                if (e < nvec && (threadIdx.x & (seg - 1)) == 0) atomicAdd(&sy[kk * P + p], part);
            }
            const int32_t ws = row_slots[k0 + kk];
            if (slot_usable(ws, a.null_block_id, a.num_slots, tid == 0 ? a.err_word : nullptr)) {
                float4 *dst = reinterpret_cast<float4 *>(a.state_cache + (size_t)ws * H * PN + head_off);
#pragma unroll
                for (int i = 0; i < VPT; ++i) {
                    const int e = tid + i * kThreads;
                    if (e < nvec) dst[e] = s[i];
                }
            }
        }
        __syncthreads();
        for (int j = tid; j < kb * P; j += kThreads) {
            const int kk = j / P, pp = j - kk * P;
            const size_t o = (((size_t)r * tpr + k0 + kk) * H + h) * P + pp;
            const float v = sy[j] + Dh * sx[j];
            y[o] = from_f32<Tin>(kGate ? silu_gate(v, ldg_f32(z + o)) : v);
        }
    }
}

// Sum of K per-row partials over the 32 lanes of a warp, transposing as it goes: each halving
// step trades half of the lane's rows with the partner lane `o` away, so K values need log2(K)
// shuffles for the first steps instead of K each.  On return, lane l holds in v[0] the full sum of
// row (l >> (5 - log2 K)) & (K - 1).
template <int K>
__device__ __forceinline__ void warp_transpose_sum(float (&v)[K], int lane) {
    int o = 16;
#pragma unroll
    for (int k = K; k > 1; k >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int q = 0; q < k / 2; ++q) {
            const float send = up ? v[q] : v[q + k / 2];
            const float keep = up ? v[q + k / 2] : v[q];
            v[q] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
#pragma unroll
    for (; o > 0; o >>= 1) v[0] += __shfl_xor_sync(0xffffffffu, v[0], o);
}

template <int K> struct Log2 { static constexpr int v = 1 + Log2<K / 2>::v; };
template <> struct Log2<1> { static constexpr int v = 0; };

// dstate = 128: a state row of one headdim index p is 128 floats, one float4 per lane of a warp,
// so warp w owns the rows p = w + 8 i (i < RPW = headdim / 8) with fixed indexing.  B and C are
// read once per token (lane l's four dstate entries), and the warp's RPW row sums for y come out of
// one transposing reduction, each written by a single lane: no atomics, no zeroing of y.
template <typename Tin, int RPW, bool kGate>
__global__ void __launch_bounds__(kThreads, RPW >= 16 ? 2 : 4)
    ssm_decode_n128_kernel(const ssm_decode_args a) {
    const int r = blockIdx.x;
    const int h = blockIdx.y;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    constexpr int P = 8 * RPW, N = 128;
    const int H = a.nheads;
    const int g = h / (H / a.ngroups);
    const int tpr = a.tokens_per_req;

    const int col = a.num_accepted_tokens ? a.num_accepted_tokens[r] : 0;
    if (col < 0 || col >= a.state_indices_cols) {
        if (tid == 0 && h == 0) report(a.err_word, SSD_DEVERR_COLUMN);
        return;
    }
    const int32_t *row_slots = a.state_indices + (size_t)r * a.state_indices_cols;
    const int32_t rs = row_slots[col];
    if (rs == a.null_block_id) return;  // CUDA-graph padding row
    if (rs < 0 || rs >= a.num_slots) {
        if (tid == 0 && h == 0) report(a.err_word, SSD_DEVERR_SLOT);
        return;
    }

    extern __shared__ __align__(16) float dsm[];
    float *sx = dsm;                   // [kTokBatch][8][RPW]: x of row w + 8 i at [w][i]
    float *sy = sx + kTokBatch * P;    // [kTokBatch][P]
    float *sB = sy + kTokBatch * P;    // [kTokBatch][N]
    float *sC = sB + kTokBatch * N;    // [kTokBatch][N]
    float *sD = sC + kTokBatch * N;    // [kTokBatch] delta

    constexpr int PN = P * N;
    const size_t head_off = (size_t)h * PN;
    float4 s[RPW];
    {
        const float4 *src = reinterpret_cast<const float4 *>(a.state_cache + (size_t)rs * H * PN + head_off);
#pragma unroll
        for (int i = 0; i < RPW; ++i) s[i] = src[(warp + 8 * i) * 32 + lane];
    }
    const float A = a.A[h];
    const float Dh = a.D ? a.D[h] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *dtp = static_cast<const Tin *>(a.dt);
    const Tin *Bp = static_cast<const Tin *>(a.B);
    const Tin *Cp = static_cast<const Tin *>(a.C);
    const Tin *z = static_cast<const Tin *>(a.z);  // output gate or NULL
    Tin *y = static_cast<Tin *>(a.y);
    constexpr int kShift = 5 - Log2<RPW>::v;  // lanes below this bit share a reduced row
    const int my_row = (lane >> kShift) & (RPW - 1);
    const bool writer = (lane & ((1 << kShift) - 1)) == 0;

    for (int k0 = 0; k0 < tpr; k0 += kTokBatch) {
        const int kb = min(kTokBatch, tpr - k0);
        if (k0 > 0) __syncthreads();  // the previous batch's readers of the staging arrays are done
        for (int j = tid; j < kb * P; j += kThreads) {
            const int kk = j / P, pp = j - kk * P;
            const size_t row = (size_t)r * tpr + k0 + kk;
            sx[kk * P + (pp & 7) * RPW + (pp >> 3)] = ldg_f32(x + (row * H + h) * P + pp);
        }
        for (int j = tid; j < kb * N; j += kThreads) {
            const int kk = j / N, nn = j - kk * N;
            const size_t row = (size_t)r * tpr + k0 + kk;
            sB[kk * N + nn] = ldg_f32(Bp + (row * a.ngroups + g) * N + nn);
            sC[kk * N + nn] = ldg_f32(Cp + (row * a.ngroups + g) * N + nn);
        }
        if (tid < kb) {
            const size_t row = (size_t)r * tpr + k0 + tid;
            sD[tid] = step_delta(ldg_f32(dtp + row * H + h) + bias, a.dt_softplus, a.dt_min, a.dt_max);
        }
        __syncthreads();
        for (int kk = 0; kk < kb; ++kk) {
            const float delta = sD[kk];
            const float decay = __expf(delta * A);
            const float4 b4 = reinterpret_cast<const float4 *>(sB + kk * N)[lane];
            const float4 c4 = reinterpret_cast<const float4 *>(sC + kk * N)[lane];
            const float *xw = sx + kk * P + warp * RPW;
            float part[RPW];
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float dx = delta * xw[i];
                s[i].x = fmaf(decay, s[i].x, dx * b4.x);
                s[i].y = fmaf(decay, s[i].y, dx * b4.y);
                s[i].z = fmaf(decay, s[i].z, dx * b4.z);
                s[i].w = fmaf(decay, s[i].w, dx * b4.w);
                part[i] = s[i].x * c4.x + s[i].y * c4.y + s[i].z * c4.z + s[i].w * c4.w;
            }
            warp_transpose_sum<RPW>(part, lane);
            if (writer) sy[kk * P + warp + 8 * my_row] = part[0];
            const int32_t ws = row_slots[k0 + kk];
            if (slot_usable(ws, a.null_block_id, a.num_slots, tid == 0 ? a.err_word : nullptr)) {
                float4 *dst = reinterpret_cast<float4 *>(a.state_cache + (size_t)ws * H * PN + head_off);
#pragma unroll
                for (int i = 0; i < RPW; ++i) dst[(warp + 8 * i) * 32 + lane] = s[i];
            }
        }
        __syncthreads();
        for (int j = tid; j < kb * P; j += kThreads) {
            const int kk = j / P, pp = j - kk * P;
            const size_t o = (((size_t)r * tpr + k0 + kk) * H + h) * P + pp;
            const float v = sy[j] + Dh * sx[kk * P + (pp & 7) * RPW + (pp >> 3)];
            y[o] = from_f32<Tin>(kGate ? silu_gate(v, ldg_f32(z + o)) : v);
        }
    }
}

template <typename Tin, bool kGate>
bool launch_n128(const ssm_decode_args &a, cudaStream_t st) {
    dim3 grid(a.batch, a.nheads);
    const size_t sm = decode_smem_bytes(a.headdim, a.dstate);
    switch (a.headdim) {
    case 8: ssm_decode_n128_kernel<Tin, 1, kGate><<<grid, kThreads, sm, st>>>(a); return true;
    case 16: ssm_decode_n128_kernel<Tin, 2, kGate><<<grid, kThreads, sm, st>>>(a); return true;
    case 32: ssm_decode_n128_kernel<Tin, 4, kGate><<<grid, kThreads, sm, st>>>(a); return true;
    case 64: ssm_decode_n128_kernel<Tin, 8, kGate><<<grid, kThreads, sm, st>>>(a); return true;
    case 128: ssm_decode_n128_kernel<Tin, 16, kGate><<<grid, kThreads, sm, st>>>(a); return true;
    default: return false;
    }
}

template <typename Tin>
cudaError_t launch_typed(const ssm_decode_args &a, cudaStream_t st) {
    const int nvec = a.headdim * a.dstate / 4;
    const int vpt = (nvec + kThreads - 1) / kThreads;
    if (a.dstate == 128 && (a.z ? launch_n128<Tin, true>(a, st) : launch_n128<Tin, false>(a, st)))
        return cudaGetLastError();
    dim3 grid(a.batch, a.nheads);
    const size_t sm = decode_smem_bytes(a.headdim, a.dstate);
    if (a.z) {  // gated instances: y * silu(z)
        if (vpt <= 1) ssm_decode_kernel<Tin, 1, true><<<grid, kThreads, sm, st>>>(a);
        else if (vpt <= 2) ssm_decode_kernel<Tin, 2, true><<<grid, kThreads, sm, st>>>(a);
        else if (vpt <= 4) ssm_decode_kernel<Tin, 4, true><<<grid, kThreads, sm, st>>>(a);
        else if (vpt <= 8) ssm_decode_kernel<Tin, 8, true><<<grid, kThreads, sm, st>>>(a);
        else ssm_decode_kernel<Tin, 16, true><<<grid, kThreads, sm, st>>>(a);
    } else {
        if (vpt <= 1) ssm_decode_kernel<Tin, 1, false><<<grid, kThreads, sm, st>>>(a);
        else if (vpt <= 2) ssm_decode_kernel<Tin, 2, false><<<grid, kThreads, sm, st>>>(a);
        else if (vpt <= 4) ssm_decode_kernel<Tin, 4, false><<<grid, kThreads, sm, st>>>(a);
        else if (vpt <= 8) ssm_decode_kernel<Tin, 8, false><<<grid, kThreads, sm, st>>>(a);
        else ssm_decode_kernel<Tin, 16, false><<<grid, kThreads, sm, st>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace

bool decode_supported(const ssm_decode_args &a) {
    const int N = a.dstate;
    const bool n_ok = (N % 128 == 0) || (N >= 4 && (N & (N - 1)) == 0);
    return n_ok && a.headdim <= 256 && N <= 256 && a.headdim * N <= 16 * 4 * kThreads;
}

cudaError_t decode_launch(const ssm_decode_args &a, cudaStream_t s) {
    if (a.dtype == SSD_BF16) return launch_typed<__nv_bfloat16>(a, s);
    return launch_typed<float>(a, s);
}

}  // namespace ssd
