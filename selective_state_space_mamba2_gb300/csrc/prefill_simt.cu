// Chunked SSD prefill on the CUDA cores (fp32 arithmetic).
//
// Serves fp32 inputs (where bf16 tensor-core operands would miss a 1e-4
// tolerance) and any shape the tensor-core path does not take.  Four kernels,
// one per step of the chunked scan of "[vllm] vLLM Mamba2 SSD 커널 웜업"
// (section "mamba_mixer2.py 변경 사항 (핵심)": a state-passing kernel and a
// chunk-scan kernel, with and without initial states):
//   1. delta and the in-chunk inclusive cumsum of delta*A       -> workspace
//   2. chunk state  S_k = sum_s exp(c_end - c_s) delta_s x_s (outer) B_s
//   3. state passing over the chunks of each sequence, fp32; stores every
//      chunk's end state to its cache slot and keeps the state entering
//      each chunk for step 4
//   4. chunk scan  y_t = sum_{s<=t} exp(c_t - c_s) delta_s (C_t.B_s) x_s
//                        + exp(c_t) C_t . state_in + D x_t
// Decays are always formed as exp of a non-positive difference c_t - c_s
// (s <= t), never as a ratio of exponentials, so they cannot overflow.  The
// cumsums are kept in fp64 and differenced there before an accurate expf, so
// the fp32 path's decays carry no cancellation error from large |c|.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kThreads = 256;

struct SeqRange {
    int first, last;  // chunk range [first, last]; empty when last < first
};

__device__ __forceinline__ SeqRange chunks_of(const ssd_prefill_args &a, int r) {
    SeqRange s;
    s.first = r > 0 ? a.last_chunk_indices[r - 1] + 1 : 0;
    s.last = a.last_chunk_indices[r];
    return s;
}

// ---------------------------------------------------------------- step 1 ----
template <typename Tin>
__global__ void __launch_bounds__(kThreads) cumsum_kernel(const ssd_prefill_args a, PrefillWorkspace ws) {
    const int k = blockIdx.x;
    const int h = blockIdx.y * (kThreads / 32) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (h >= a.nheads) return;
    const int t0 = a.cu_chunk_seqlens[k], t1 = a.cu_chunk_seqlens[k + 1];
    if (t0 < 0 || t1 < t0 || t1 > a.total_tokens) {
        if (lane == 0) report(a.err_word, SSD_DEVERR_METADATA);
        return;
    }
    const Tin *dt = static_cast<const Tin *>(a.dt);
    const float A = a.A[h];
    const float bias = a.dt_bias ? a.dt_bias[h] : 0.f;
    const size_t row = (size_t)h * a.total_tokens;
    double carry = 0.0;
    for (int base = t0; base < t1; base += 32) {
        const int t = base + lane;
        float d = 0.f;
        double c = 0.0;
        if (t < t1) {
            d = step_delta(ldg_f32(dt + (size_t)t * a.nheads + h) + bias, a.dt_softplus, a.dt_min, a.dt_max);
            c = (double)d * (double)A;
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const double v = __shfl_up_sync(0xffffffffu, c, off);
            if (lane >= off) c += v;
        }
        c += carry;
        if (t < t1) {
            ws.delta[row + t] = d;
            ws.cumlog[row + t] = c;
        }
        carry = __shfl_sync(0xffffffffu, c, 31);
    }
}

// ---------------------------------------------------------------- step 2 ----
constexpr int kStateTile = 16;  // tokens staged per round

template <typename Tin, int OPT>
__global__ void __launch_bounds__(kThreads) chunk_state_kernel(const ssd_prefill_args a, PrefillWorkspace ws) {
    extern __shared__ float smem[];
    const int k = blockIdx.x, h = blockIdx.y;
    const int H = a.nheads, P = a.headdim, N = a.dstate, G = a.ngroups;
    const int g = h / (H / G);
    const int PN = P * N;
    const int t0 = a.cu_chunk_seqlens[k], t1 = a.cu_chunk_seqlens[k + 1];
    if (t0 < 0 || t1 < t0 || t1 > a.total_tokens) return;  // reported by step 1
    float *sx = smem;                        // [tile][P]
    float *sB = sx + kStateTile * P;         // [tile][N]
    float *sw = sB + kStateTile * N;         // [tile]
    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *B = static_cast<const Tin *>(a.B);
    const size_t hrow = (size_t)h * a.total_tokens;
    const double c_end = t1 > t0 ? ws.cumlog[hrow + t1 - 1] : 0.0;

    float acc[OPT];
    int pofs[OPT], nofs[OPT];
#pragma unroll
    for (int j = 0; j < OPT; ++j) {
        acc[j] = 0.f;
        const int e = threadIdx.x + j * kThreads;
        pofs[j] = e < PN ? e / N : 0;
        nofs[j] = e < PN ? e - pofs[j] * N : 0;
    }
    for (int base = t0; base < t1; base += kStateTile) {
        __syncthreads();
        for (int i = threadIdx.x; i < kStateTile * P; i += kThreads) {
            const int tt = i / P, p = i - tt * P, t = base + tt;
            sx[i] = t < t1 ? ldg_f32(x + ((size_t)t * H + h) * P + p) : 0.f;
        }
        for (int i = threadIdx.x; i < kStateTile * N; i += kThreads) {
            const int tt = i / N, n = i - tt * N, t = base + tt;
            sB[i] = t < t1 ? ldg_f32(B + ((size_t)t * G + g) * N + n) : 0.f;
        }
        if (threadIdx.x < kStateTile) {
            const int t = base + threadIdx.x;
            sw[threadIdx.x] = t < t1 ? expf((float)(c_end - ws.cumlog[hrow + t])) * ws.delta[hrow + t] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int tt = 0; tt < kStateTile; ++tt) {
            const float w = sw[tt];
#pragma unroll
            for (int j = 0; j < OPT; ++j)
                acc[j] = fmaf(w * sx[tt * P + pofs[j]], sB[tt * N + nofs[j]], acc[j]);
        }
    }
    float *out = ws.chunk_state + ((size_t)k * H + h) * PN;
#pragma unroll
    for (int j = 0; j < OPT; ++j) {
        const int e = threadIdx.x + j * kThreads;
        if (e < PN) out[e] = acc[j];
    }
}

// ---------------------------------------------------------------- step 3 ----
__global__ void __launch_bounds__(kThreads) state_pass_kernel(const ssd_prefill_args a, PrefillWorkspace ws) {
    const int r = blockIdx.x, h = blockIdx.y;
    const int H = a.nheads;
    const int PN = a.headdim * a.dstate;
    const int e = blockIdx.z * kThreads + threadIdx.x;
    const SeqRange cr = chunks_of(a, r);
    const bool reporter = threadIdx.x == 0 && blockIdx.z == 0 && h == 0;
    if (cr.last >= cr.first) {
        if (cr.first < 0 || cr.last >= a.num_chunks ||
            a.cu_chunk_seqlens[cr.first] != a.cu_seqlens[r] ||
            a.cu_chunk_seqlens[cr.last + 1] != a.cu_seqlens[r + 1]) {
            if (reporter) report(a.err_word, SSD_DEVERR_METADATA);
            return;
        }
    }
    if (e >= PN) return;
    const size_t head_off = (size_t)h * PN + e;
    float s = 0.f;
    const int32_t is = a.init_slot ? a.init_slot[r] : a.null_block_id;
    if (slot_usable(is, a.null_block_id, a.num_slots, reporter ? a.err_word : nullptr))
        s = a.state_cache[(size_t)is * H * PN + head_off];
    const size_t hrow = (size_t)h * a.total_tokens;
    for (int k = cr.first; k <= cr.last; ++k) {
        const int t0 = a.cu_chunk_seqlens[k], t1 = a.cu_chunk_seqlens[k + 1];
        if (t0 < 0 || t1 <= t0 || t1 > a.total_tokens) {
            if (reporter) report(a.err_word, SSD_DEVERR_METADATA);
            return;
        }
        ws.state_in[(size_t)k * H * PN + head_off] = s;
        const float decay = (float)exp(ws.cumlog[hrow + t1 - 1]);
        s = fmaf(decay, s, ws.chunk_state[(size_t)k * H * PN + head_off]);
        const int32_t cs = a.chunk_slot ? a.chunk_slot[k] : a.null_block_id;
        if (slot_usable(cs, a.null_block_id, a.num_slots, reporter ? a.err_word : nullptr))
            a.state_cache[(size_t)cs * H * PN + head_off] = s;
    }
}

// ---------------------------------------------------------------- step 4 ----
constexpr int kScanRows = 32;  // output tokens per CTA
constexpr int kScanCols = 32;  // source tokens per round

// floats in front of the two fp64 vectors of the scan kernel, rounded up to an
// even count so the fp64 part is 8-byte aligned
__host__ __device__ __forceinline__ size_t scan_float_slots(int P, int N) {
    const size_t nf = (size_t)P * (N + 1) + kScanRows * N + kScanCols * (N + 1) + kScanCols * P +
                      kScanRows * (kScanCols + 1) + kScanCols;
    return (nf + 1) & ~(size_t)1;
}

template <typename Tin>
__global__ void __launch_bounds__(kThreads) chunk_scan_kernel(const ssd_prefill_args a, PrefillWorkspace ws) {
    extern __shared__ float smem[];
    const int k = blockIdx.x, h = blockIdx.y;
    const int H = a.nheads, P = a.headdim, N = a.dstate, G = a.ngroups;
    const int g = h / (H / G);
    const int t0 = a.cu_chunk_seqlens[k], t1 = a.cu_chunk_seqlens[k + 1];
    if (t0 < 0 || t1 < t0 || t1 > a.total_tokens) return;
    const int Ns = N + 1;  // padded row stride of the state copy
    float *sh = smem;                         // [P][N+1]  state entering the chunk
    float *sC = sh + P * Ns;                  // [rows][N]
    float *sB = sC + kScanRows * N;           // [cols][N+1] (padded: column reads stride by row)
    float *sx = sB + kScanCols * Ns;          // [cols][P]
    float *sM = sx + kScanCols * P;           // [rows][cols+1]
    float *sds = sM + kScanRows * (kScanCols + 1);  // [cols] delta_s
    double *scr = reinterpret_cast<double *>(smem + scan_float_slots(P, N));  // [rows] c_t (8-byte aligned)
    double *scs = scr + kScanRows;            // [cols] c_s

    const Tin *x = static_cast<const Tin *>(a.x);
    const Tin *B = static_cast<const Tin *>(a.B);
    const Tin *C = static_cast<const Tin *>(a.C);
    const Tin *z = static_cast<const Tin *>(a.z);  // output gate or NULL
    Tin *y = static_cast<Tin *>(a.y);
    const size_t hrow = (size_t)h * a.total_tokens;
    const float Dh = a.D ? a.D[h] : 0.f;

    // the state entering this chunk
    const float *st = ws.state_in + ((size_t)k * H + h) * P * N;
    for (int i = threadIdx.x; i < P * N; i += kThreads) {
        const int p = i / N, n = i - p * N;
        sh[p * Ns + n] = st[i];
    }
    const int row_groups = kThreads / P;  // >= 1 because P <= 256
    const int my_p = threadIdx.x % P;
    const int my_r0 = threadIdx.x / P;
    const bool active = my_r0 < row_groups;

    for (int ta = t0 + blockIdx.z * kScanRows; ta < t1; ta += gridDim.z * kScanRows) {
        const int tb = min(ta + kScanRows, t1);
        __syncthreads();
        for (int i = threadIdx.x; i < kScanRows * N; i += kThreads) {
            const int rr = i / N, n = i - rr * N, t = ta + rr;
            sC[i] = t < tb ? ldg_f32(C + ((size_t)t * G + g) * N + n) : 0.f;
        }
        if (threadIdx.x < kScanRows) {
            const int t = ta + threadIdx.x;
            scr[threadIdx.x] = t < tb ? ws.cumlog[hrow + t] : 0.0;
        }
        __syncthreads();
        float acc[kScanRows];
#pragma unroll
        for (int i = 0; i < kScanRows; ++i) acc[i] = 0.f;
        // carried state: exp(c_t) * C_t . state_in[p, :]
        if (active) {
            for (int n = 0; n < N; ++n) {
                const float hv = sh[my_p * Ns + n];
#pragma unroll
                for (int i = 0; i < kScanRows; ++i)
                    if (my_r0 + i * row_groups < kScanRows) acc[i] = fmaf(sC[(my_r0 + i * row_groups) * N + n], hv, acc[i]);
            }
#pragma unroll
            for (int i = 0; i < kScanRows; ++i)
                if (my_r0 + i * row_groups < kScanRows) acc[i] *= (float)exp(scr[my_r0 + i * row_groups]);
        }
        // in-chunk contributions from source tokens s in [t0, tb)
        for (int sa = t0; sa < tb; sa += kScanCols) {
            __syncthreads();
            for (int i = threadIdx.x; i < kScanCols * N; i += kThreads) {
                const int cc = i / N, n = i - cc * N, s = sa + cc;
                sB[cc * Ns + n] = s < tb ? ldg_f32(B + ((size_t)s * G + g) * N + n) : 0.f;
            }
            for (int i = threadIdx.x; i < kScanCols * P; i += kThreads) {
                const int cc = i / P, p = i - cc * P, s = sa + cc;
                sx[i] = s < tb ? ldg_f32(x + ((size_t)s * H + h) * P + p) : 0.f;
            }
            if (threadIdx.x < kScanCols) {
                const int s = sa + threadIdx.x;
                scs[threadIdx.x] = s < tb ? ws.cumlog[hrow + s] : 0.0;
                sds[threadIdx.x] = s < tb ? ws.delta[hrow + s] : 0.f;
            }
            __syncthreads();
            // M[t, s] = exp(c_t - c_s) delta_s (C_t . B_s) for s <= t
            for (int i = threadIdx.x; i < kScanRows * kScanCols; i += kThreads) {
                const int rr = i / kScanCols, cc = i - rr * kScanCols;
                const int t = ta + rr, s = sa + cc;
                float m = 0.f;
                if (t < tb && s <= t) {
                    float dot = 0.f;
                    for (int n = 0; n < N; ++n) dot = fmaf(sC[rr * N + n], sB[cc * Ns + n], dot);
                    m = dot * expf((float)(scr[rr] - scs[cc])) * sds[cc];
                }
                sM[rr * (kScanCols + 1) + cc] = m;
            }
            __syncthreads();
            if (active) {
                for (int cc = 0; cc < kScanCols; ++cc) {
                    const float xv = sx[cc * P + my_p];
#pragma unroll
                    for (int i = 0; i < kScanRows; ++i)
                        if (my_r0 + i * row_groups < kScanRows)
                            acc[i] = fmaf(sM[(my_r0 + i * row_groups) * (kScanCols + 1) + cc], xv, acc[i]);
                }
            }
        }
        if (active) {
#pragma unroll
            for (int i = 0; i < kScanRows; ++i) {
                const int rr = my_r0 + i * row_groups;
                const int t = ta + rr;
                if (rr < kScanRows && t < tb) {
                    const size_t o = ((size_t)t * H + h) * P + my_p;
                    const float v = acc[i] + Dh * ldg_f32(x + o);
                    y[o] = from_f32<Tin>(z ? silu_gate(v, ldg_f32(z + o)) : v);
                }
            }
        }
    }
}

size_t scan_smem_bytes(const ssd_prefill_args &a) {
    const int P = a.headdim, N = a.dstate;
    return sizeof(float) * scan_float_slots(P, N) + sizeof(double) * (kScanRows + kScanCols);
}

size_t state_smem_bytes(const ssd_prefill_args &a) {
    return sizeof(float) * ((size_t)kStateTile * (a.headdim + a.dstate) + kStateTile);
}

template <typename Tin, int OPT>
cudaError_t launch_state(const ssd_prefill_args &a, const PrefillWorkspace &ws, cudaStream_t st) {
    const size_t smem = state_smem_bytes(a);
    auto kern = chunk_state_kernel<Tin, OPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    kern<<<dim3(a.num_chunks, a.nheads), kThreads, smem, st>>>(a, ws);
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_typed(const ssd_prefill_args &a, const PrefillWorkspace &ws, cudaStream_t st) {
    cumsum_kernel<Tin><<<dim3(a.num_chunks, (a.nheads + 7) / 8), kThreads, 0, st>>>(a, ws);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const int opt = (a.headdim * a.dstate + kThreads - 1) / kThreads;
    if (opt <= 4) e = launch_state<Tin, 4>(a, ws, st);
    else if (opt <= 8) e = launch_state<Tin, 8>(a, ws, st);
    else if (opt <= 16) e = launch_state<Tin, 16>(a, ws, st);
    else if (opt <= 32) e = launch_state<Tin, 32>(a, ws, st);
    else e = launch_state<Tin, 64>(a, ws, st);
    if (e != cudaSuccess) return e;
    const int pn = a.headdim * a.dstate;
    state_pass_kernel<<<dim3(a.num_seqs, a.nheads, (pn + kThreads - 1) / kThreads), kThreads, 0, st>>>(a, ws);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = scan_smem_bytes(a);
    e = cudaFuncSetAttribute(chunk_scan_kernel<Tin>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int zt = (a.chunk_size + kScanRows - 1) / kScanRows;
    chunk_scan_kernel<Tin><<<dim3(a.num_chunks, a.nheads, zt < 1 ? 1 : (zt > 64 ? 64 : zt)), kThreads, smem, st>>>(a, ws);
    return cudaGetLastError();
}

size_t align_up(size_t v) { return (v + 255) & ~(size_t)255; }

}  // namespace

bool simt_prefill_supported(const ssd_prefill_args &a) {
    return a.headdim >= 1 && a.headdim <= 256 && a.dstate >= 1 && a.dstate <= 256 &&
           a.headdim * a.dstate <= 64 * kThreads && scan_smem_bytes(a) <= 220 * 1024;
}

size_t simt_prefill_workspace(const ssd_prefill_args &a, PrefillWorkspace *ws, void *base) {
    const size_t per_tok = align_up(sizeof(float) * (size_t)a.nheads * a.total_tokens);
    const size_t per_tok64 = align_up(sizeof(double) * (size_t)a.nheads * a.total_tokens);
    const size_t per_chunk = align_up(sizeof(float) * (size_t)a.num_chunks * a.nheads * a.headdim * a.dstate);
    if (ws) {
        char *p = static_cast<char *>(base);
        ws->delta = reinterpret_cast<float *>(p);
        ws->cumlog = reinterpret_cast<double *>(p + per_tok);
        ws->chunk_state = reinterpret_cast<float *>(p + per_tok + per_tok64);
        ws->state_in = reinterpret_cast<float *>(p + per_tok + per_tok64 + per_chunk);
    }
    return per_tok + per_tok64 + 2 * per_chunk;
}

cudaError_t simt_prefill_launch(const ssd_prefill_args &a, const PrefillWorkspace &ws, cudaStream_t s) {
    if (a.dtype == SSD_BF16) return launch_typed<__nv_bfloat16>(a, ws, s);
    return launch_typed<float>(a, ws, s);
}

}  // namespace ssd
