// Mamba1 selective scan (S6): per-channel states, varlen prefill and decode.
//
// "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링", section "논문 핵심 내용":
// in S6, Delta, B and C are functions of the token.  Every channel d carries
// its own state vector s[d, 0..N-1] with its own decay rates A[d, :], so
// there is no head-level contraction to put on the tensor cores: the work is
// N exponentials and 2N FMAs per (token, channel), and its only data are the
// token's x, dt (and z) for the channel and the group's B and C rows.
//
// Prefill: one CTA per (sequence, 64 channels), one channel per thread, the
// N-vector state in registers for the whole sequence.  The sequence is walked
// in tiles of up to 32 tokens (16 for fp32) that never cross a chunk end; each tile's x, dt
// (and z) rows for the CTA's channels and the group's B and C rows are staged
// into shared memory with 16-byte cp.async copies, double-buffered so the
// next tile is in flight while this one is computed.  After a chunk's last
// token the state goes to the chunk's cache slot (prefix caching at the
// chunk size, 2048 by default for Mamba1: "[vllm] vLLM Mamba2 SSD 커널 웜업",
// "vllm/config/model.py 변경 사항").
//
// Bound: the exponentials.  N of them per (token, channel) against about
// 3 x 2 bytes of HBM traffic (x, dt, y in bf16), so the multi-function unit,
// not HBM, sets the time at N = 16.
//
// Decode: one CTA per (request, 64 channels), the request's state read from
// the slot its num_accepted_tokens column names, each token's state stored to
// its own column: the routing of ssm_decode_update.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kCh = 64;  // channels per CTA, one per thread
// tokens per staged tile: 32 of bf16, 16 of fp32 (both keep a stage at 14 KB)
template <typename Tin>
constexpr int tile_tokens() { return sizeof(Tin) == 2 ? 32 : 16; }

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

// N consecutive elements (16-byte aligned) -> fp32, in 16-byte loads
template <int N>
__device__ __forceinline__ void row_to_f32(const float *p, float (&o)[N]) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float4 v = reinterpret_cast<const float4 *>(p)[i];
        o[4 * i] = v.x; o[4 * i + 1] = v.y; o[4 * i + 2] = v.z; o[4 * i + 3] = v.w;
    }
}
template <int N>
__device__ __forceinline__ void row_to_f32(const __nv_bfloat16 *p, float (&o)[N]) {
#pragma unroll
    for (int i = 0; i < N / 8; ++i) {
        const uint4 v = reinterpret_cast<const uint4 *>(p)[i];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            o[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
            o[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
        }
    }
}
template <int N, typename Tin>
__device__ __forceinline__ void row_to_f32_ldg(const Tin *p, float (&o)[N]) {
    if constexpr (sizeof(Tin) == 4) {
#pragma unroll
        for (int i = 0; i < N / 4; ++i) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(p) + i);
            o[4 * i] = v.x; o[4 * i + 1] = v.y; o[4 * i + 2] = v.z; o[4 * i + 3] = v.w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < N / 8; ++i) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(p) + i);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                o[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                o[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        }
    }
}

template <int N>
__device__ __forceinline__ void state_load(const float *p, float (&h)[N]) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float4 v = reinterpret_cast<const float4 *>(p)[i];
        h[4 * i] = v.x; h[4 * i + 1] = v.y; h[4 * i + 2] = v.z; h[4 * i + 3] = v.w;
    }
}
template <int N>
__device__ __forceinline__ void state_store(float *p, const float (&h)[N]) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
        reinterpret_cast<float4 *>(p)[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
}

// One token of one channel: the state update and the output.
template <int N>
__device__ __forceinline__ float m1_step(float (&h)[N], const float (&Ad)[N], float delta, float xv,
                                         const float (&Bt)[N], const float (&Ct)[N], float Dd) {
    const float dx = delta * xv;
    float acc = 0.f;
#pragma unroll
    for (int n = 0; n < N; ++n) {
        h[n] = fmaf(__expf(delta * Ad[n]), h[n], dx * Bt[n]);
        acc = fmaf(Ct[n], h[n], acc);
    }
    return fmaf(Dd, xv, acc);
}

// Tiles of at most kTc tokens of one sequence, never crossing a chunk end.
template <int kTc>
struct TileCursor {
    const int32_t *cu_chunk;
    int k, last, tb, ce;
    __device__ void start(const int32_t *cc, int first, int last_) {
        cu_chunk = cc;
        k = first;
        last = last_;
        tb = cc[first];
        ce = cc[first + 1];
    }
    __device__ int len() const { return min(kTc, ce - tb); }
    __device__ bool ends_chunk() const { return tb + len() == ce; }
    __device__ void next() {
        tb += len();
        if (tb == ce && k < last) {
            ++k;
            ce = cu_chunk[k + 1];
        }
    }
};

template <typename Tin, int N, bool kGate>
__global__ void __launch_bounds__(kCh) mamba1_scan_kernel(const mamba1_args a) {
    constexpr int kTc = tile_tokens<Tin>();
    constexpr int kRow = kCh * (int)sizeof(Tin);  // one token's CTA channels, bytes
    constexpr int kBc = N * (int)sizeof(Tin);     // one token's B (or C) row, bytes
    constexpr int kTileX = kTc * kRow;
    constexpr int kTileBC = kTc * kBc;
    constexpr int kStage = (kGate ? 3 : 2) * kTileX + 2 * kTileBC;
    __shared__ __align__(16) uint8_t sm[2 * kStage];

    const int r = blockIdx.x, tid = threadIdx.x;
    const int Dc = a.dim, G = a.ngroups;
    const int d0 = blockIdx.y * kCh, d = d0 + tid;
    const int g = d0 / (Dc / G);  // (Dc / G) % kCh == 0: the CTA's channels share a group

    // the sequence's chunk range, validated before anything is read through it
    const int first = r > 0 ? a.last_chunk_indices[r - 1] + 1 : 0;
    const int last = a.last_chunk_indices[r];
    if (last < first) return;  // no new tokens
    int ntiles = 0;
    {
        bool bad = first < 0 || last >= a.num_chunks || a.cu_chunk_seqlens[first] != a.cu_seqlens[r] ||
                   a.cu_chunk_seqlens[last + 1] != a.cu_seqlens[r + 1];
        for (int k = first; !bad && k <= last; ++k) {
            const int lo = a.cu_chunk_seqlens[k], hi = a.cu_chunk_seqlens[k + 1];
            if (lo < 0 || hi <= lo || hi > a.total_tokens) bad = true;
            else ntiles += (hi - lo + kTc - 1) / kTc;
        }
        if (bad) {
            if (tid == 0 && blockIdx.y == 0) report(a.err_word, SSD_DEVERR_METADATA);
            return;
        }
    }

    float h[N], Ad[N];
    {
        const int32_t is = a.init_slot ? a.init_slot[r] : a.null_block_id;
        if (slot_usable(is, a.null_block_id, a.num_slots, (tid == 0) ? a.err_word : nullptr))
            state_load<N>(a.state_cache + ((size_t)is * Dc + d) * N, h);
        else
#pragma unroll
            for (int n = 0; n < N; ++n) h[n] = 0.f;
#pragma unroll
        for (int n = 0; n < N; ++n) Ad[n] = a.A[(size_t)d * N + n];
    }
    const float Dd = a.D ? a.D[d] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[d] : 0.f;
    const uint8_t *gx = static_cast<const uint8_t *>(a.x), *gdt = static_cast<const uint8_t *>(a.dt);
    const uint8_t *gz = static_cast<const uint8_t *>(a.z);
    const uint8_t *gB = static_cast<const uint8_t *>(a.B), *gC = static_cast<const uint8_t *>(a.C);
    Tin *y = static_cast<Tin *>(a.y);

    auto load_tile = [&](int buf, int tb, int L) {
        uint8_t *st = sm + buf * kStage;
        constexpr int kPieces = kRow / 16;
        for (int i = tid; i < L * kPieces; i += kCh) {
            const int row = i / kPieces, pc = i - row * kPieces;
            const size_t go = ((size_t)(tb + row) * Dc + d0) * sizeof(Tin) + pc * 16;
            const int so = row * kRow + pc * 16;
            cp_async16(st + so, gx + go);
            cp_async16(st + kTileX + so, gdt + go);
            if (kGate) cp_async16(st + 2 * kTileX + so, gz + go);
        }
        constexpr int kBcPieces = kBc / 16;
        uint8_t *sb = st + (kGate ? 3 : 2) * kTileX;
        for (int i = tid; i < L * kBcPieces; i += kCh) {
            const int row = i / kBcPieces, pc = i - row * kBcPieces;
            const size_t go = ((size_t)(tb + row) * G + g) * kBc + pc * 16;
            cp_async16(sb + row * kBc + pc * 16, gB + go);
            cp_async16(sb + kTileBC + row * kBc + pc * 16, gC + go);
        }
        cp_async_commit();
    };

    TileCursor<kTc> ld, cur;
    ld.start(a.cu_chunk_seqlens, first, last);
    cur.start(a.cu_chunk_seqlens, first, last);
    load_tile(0, ld.tb, ld.len());
    ld.next();
    int32_t cs = a.chunk_slot ? a.chunk_slot[first] : a.null_block_id;  // slot of the current chunk's end
    for (int i = 0; i < ntiles; ++i) {
        if (i + 1 < ntiles) {
            load_tile((i + 1) & 1, ld.tb, ld.len());  // that buffer's readers passed the barrier below
            ld.next();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // tile i has landed for every thread
        const uint8_t *st = sm + (i & 1) * kStage;
        const Tin *xs = reinterpret_cast<const Tin *>(st);
        const Tin *dts = reinterpret_cast<const Tin *>(st + kTileX);
        const Tin *zs = reinterpret_cast<const Tin *>(st + 2 * kTileX);
        const uint8_t *sb = st + (kGate ? 3 : 2) * kTileX;
        const Tin *Bs = reinterpret_cast<const Tin *>(sb);
        const Tin *Cs = reinterpret_cast<const Tin *>(sb + kTileBC);
        const int tb = cur.tb, L = cur.len();
        for (int t = 0; t < L; ++t) {
            float Bt[N], Ct[N];
            row_to_f32<N>(Bs + t * N, Bt);
            row_to_f32<N>(Cs + t * N, Ct);
            const float xv = to_f32(xs[t * kCh + tid]);
            const float delta = step_delta(to_f32(dts[t * kCh + tid]) + bias, a.dt_softplus, a.dt_min, a.dt_max);
            float yv = m1_step<N>(h, Ad, delta, xv, Bt, Ct, Dd);
            if (kGate) yv = silu_gate(yv, to_f32(zs[t * kCh + tid]));
            y[(size_t)(tb + t) * Dc + d] = from_f32<Tin>(yv);
        }
        if (cur.ends_chunk()) {
            if (slot_usable(cs, a.null_block_id, a.num_slots, (tid == 0) ? a.err_word : nullptr))
                state_store<N>(a.state_cache + ((size_t)cs * Dc + d) * N, h);
            if (a.chunk_slot) cs = a.chunk_slot[min(cur.k + 1, last)];
        }
        cur.next();
        __syncthreads();  // every thread is done with buffer (i & 1) before it is refilled
    }
}

template <typename Tin, int N, bool kGate>
__global__ void __launch_bounds__(kCh) mamba1_update_kernel(const mamba1_args a) {
    const int r = blockIdx.x, tid = threadIdx.x;
    const int Dc = a.dim, G = a.ngroups;
    const int d = blockIdx.y * kCh + tid;
    const int g = d / (Dc / G);
    const int tpr = a.tokens_per_req;
    const int col = a.num_accepted_tokens ? a.num_accepted_tokens[r] : 0;
    if (col < 0 || col >= a.state_indices_cols) {
        if (tid == 0 && blockIdx.y == 0) report(a.err_word, SSD_DEVERR_COLUMN);
        return;
    }
    const int32_t *row_slots = a.state_indices + (size_t)r * a.state_indices_cols;
    const int32_t rs = row_slots[col];
    if (rs == a.null_block_id) return;  // CUDA-graph padding row
    if (rs < 0 || rs >= a.num_slots) {
        if (tid == 0 && blockIdx.y == 0) report(a.err_word, SSD_DEVERR_SLOT);
        return;
    }
    float h[N], Ad[N];
    state_load<N>(a.state_cache + ((size_t)rs * Dc + d) * N, h);
#pragma unroll
    for (int n = 0; n < N; ++n) Ad[n] = a.A[(size_t)d * N + n];
    const float Dd = a.D ? a.D[d] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[d] : 0.f;
    const Tin *x = static_cast<const Tin *>(a.x), *dt = static_cast<const Tin *>(a.dt);
    const Tin *Bp = static_cast<const Tin *>(a.B), *Cp = static_cast<const Tin *>(a.C);
    const Tin *z = static_cast<const Tin *>(a.z);
    Tin *y = static_cast<Tin *>(a.y);
    for (int k = 0; k < tpr; ++k) {
        const size_t row = (size_t)r * tpr + k;
        float Bt[N], Ct[N];
        row_to_f32_ldg<N>(Bp + (row * G + g) * N, Bt);
        row_to_f32_ldg<N>(Cp + (row * G + g) * N, Ct);
        const float xv = ldg_f32(x + row * Dc + d);
        const float delta = step_delta(ldg_f32(dt + row * Dc + d) + bias, a.dt_softplus, a.dt_min, a.dt_max);
        float yv = m1_step<N>(h, Ad, delta, xv, Bt, Ct, Dd);
        if (kGate) yv = silu_gate(yv, ldg_f32(z + row * Dc + d));
        y[row * Dc + d] = from_f32<Tin>(yv);
        const int32_t ws = row_slots[k];
        if (slot_usable(ws, a.null_block_id, a.num_slots, tid == 0 ? a.err_word : nullptr))
            state_store<N>(a.state_cache + ((size_t)ws * Dc + d) * N, h);
    }
}

template <typename Tin, int N>
cudaError_t launch_n(const mamba1_args &a, bool decode, cudaStream_t st) {
    const dim3 grid(a.num_seqs, a.dim / kCh);
    if (decode) {
        if (a.z) mamba1_update_kernel<Tin, N, true><<<grid, kCh, 0, st>>>(a);
        else mamba1_update_kernel<Tin, N, false><<<grid, kCh, 0, st>>>(a);
    } else {
        if (a.z) mamba1_scan_kernel<Tin, N, true><<<grid, kCh, 0, st>>>(a);
        else mamba1_scan_kernel<Tin, N, false><<<grid, kCh, 0, st>>>(a);
    }
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const mamba1_args &a, bool decode, cudaStream_t st) {
    return a.dstate == 8 ? launch_n<Tin, 8>(a, decode, st) : launch_n<Tin, 16>(a, decode, st);
}

}  // namespace

cudaError_t mamba1_launch(const mamba1_args &a, bool decode, cudaStream_t st) {
    if (a.num_seqs == 0) return cudaSuccess;
    return a.dtype == SSD_BF16 ? launch_t<__nv_bfloat16>(a, decode, st) : launch_t<float>(a, decode, st);
}

}  // namespace ssd
