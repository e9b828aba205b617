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
// in tiles of up to 48 tokens (16 for fp32) that never cross a chunk end; each tile's x, dt
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
// Decode: one CTA per (two requests, 64 channels), each request's state read
// from the slot its num_accepted_tokens column names, each token's state
// stored to its own column: the routing of ssm_decode_update.
#include "common.cuh"

namespace ssd {
namespace {

constexpr int kCh = 64;  // channels per CTA, one per thread
// tokens per staged tile: 48 of bf16, 16 of fp32.  48 bf16 tokens (the gated instance's two
// stages then fill the 48 KB of static shared memory) beat 32 (2.04 vs 2.12 ms on 8 x 8192 tokens
// x 5120 channels) and 16 (2.14); 64 leaves too few CTAs per SM (2.63).
template <typename Tin>
constexpr int tile_tokens() { return sizeof(Tin) == 2 ? 48 : 16; }

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

// N consecutive elements (16-byte aligned) of global memory -> fp32, in 16-byte loads
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

// Packed fp32 pairs: one instruction does two lanes of work on the FMA pipe.
__device__ __forceinline__ uint64_t pk(float2 v) { return *reinterpret_cast<uint64_t *>(&v); }
__device__ __forceinline__ float2 upk(uint64_t v) { return *reinterpret_cast<float2 *>(&v); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)), "l"(pk(c)));
    return upk(r);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(pk(a)), "l"(pk(b)));
    return upk(r);
}
// 2^x on the multi-function unit; e^v is taken as 2^(v log2 e), with log2 e folded into A
__device__ __forceinline__ float exp2_fast(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// One token of one channel: the state update and the output.  A2 = A[d, :] log2 e, so the decay
// of state n is 2^(delta A2[n]) = exp(delta A[d, n]).
template <int N>
__device__ __forceinline__ float m1_step(float2 (&h)[N / 2], const float2 (&A2)[N / 2], float delta, float xv,
                                         const float (&Bt)[N], const float (&Ct)[N], float Dd) {
    const float2 dd = make_float2(delta, delta);
    const float dx = delta * xv;
    const float2 dx2 = make_float2(dx, dx);
    float2 acc0 = make_float2(0.f, 0.f), acc1 = make_float2(0.f, 0.f);
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
        const float2 e = mul2(dd, A2[i]);
        const float2 a = make_float2(exp2_fast(e.x), exp2_fast(e.y));
        h[i] = fma2(a, h[i], mul2(dx2, make_float2(Bt[2 * i], Bt[2 * i + 1])));
        if (i & 1) acc1 = fma2(make_float2(Ct[2 * i], Ct[2 * i + 1]), h[i], acc1);
        else acc0 = fma2(make_float2(Ct[2 * i], Ct[2 * i + 1]), h[i], acc0);
    }
    return fmaf(Dd, xv, (acc0.x + acc0.y) + (acc1.x + acc1.y));
}

template <typename Tin>
__device__ __forceinline__ float m1_delta(float v, const mamba1_args &a) {
    // bf16 tokens: the fast exp/log form (under 2e-5 relative); fp32 tokens: expf/log1pf
    if constexpr (sizeof(Tin) == 2) return fast_delta(v, a.dt_softplus, a.dt_min, a.dt_max);
    else return step_delta(v, a.dt_softplus, a.dt_min, a.dt_max);
}

template <int N>
__device__ __forceinline__ void smem_row(const float *p, float (&o)[N]) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float4 v = reinterpret_cast<const float4 *>(p)[i];
        o[4 * i] = v.x; o[4 * i + 1] = v.y; o[4 * i + 2] = v.z; o[4 * i + 3] = v.w;
    }
}

template <int N>
__device__ __forceinline__ void state_load2(const float *p, float2 (&h)[N / 2]) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i) {
        const float4 v = reinterpret_cast<const float4 *>(p)[i];
        h[2 * i] = make_float2(v.x, v.y);
        h[2 * i + 1] = make_float2(v.z, v.w);
    }
}
template <int N>
__device__ __forceinline__ void state_store2(float *p, const float2 (&h)[N / 2]) {
#pragma unroll
    for (int i = 0; i < N / 4; ++i)
        reinterpret_cast<float4 *>(p)[i] = make_float4(h[2 * i].x, h[2 * i].y, h[2 * i + 1].x, h[2 * i + 1].y);
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
    constexpr bool kConvert = sizeof(Tin) != 4;  // bf16 B/C rows are widened to fp32 once per tile
    __shared__ __align__(16) uint8_t sm[2 * kStage];
    __shared__ __align__(16) float sBCf[kConvert ? 2 * kTc * N : 4];

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

    constexpr float kLog2e = 1.4426950408889634f;
    float2 h[N / 2], A2[N / 2];
    {
        const int32_t is = a.init_slot ? a.init_slot[r] : a.null_block_id;
        if (slot_usable(is, a.null_block_id, a.num_slots, (tid == 0) ? a.err_word : nullptr))
            state_load2<N>(a.state_cache + ((size_t)is * Dc + d) * N, h);
        else
#pragma unroll
            for (int i = 0; i < N / 2; ++i) h[i] = make_float2(0.f, 0.f);
#pragma unroll
        for (int i = 0; i < N / 2; ++i)
            A2[i] = make_float2(a.A[(size_t)d * N + 2 * i] * kLog2e, a.A[(size_t)d * N + 2 * i + 1] * kLog2e);
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
        const int tb = cur.tb, L = cur.len();
        const float *Bf, *Cf;  // the tile's B and C rows in fp32, [kTc][N] each
        if constexpr (kConvert) {
            const uint4 *raw = reinterpret_cast<const uint4 *>(sb);  // B rows then C rows, 8 bf16 per uint4
            for (int i = tid; i < 2 * L * N / 8; i += kCh) {
                const int which = i / (L * N / 8), j = i - which * (L * N / 8);
                const uint4 v = raw[which * (kTc * N / 8) + j];
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
                float4 *o = reinterpret_cast<float4 *>(sBCf + which * kTc * N + 8 * j);
                o[0] = make_float4(__uint_as_float(w[0] << 16), __uint_as_float(w[0] & 0xFFFF0000u),
                                   __uint_as_float(w[1] << 16), __uint_as_float(w[1] & 0xFFFF0000u));
                o[1] = make_float4(__uint_as_float(w[2] << 16), __uint_as_float(w[2] & 0xFFFF0000u),
                                   __uint_as_float(w[3] << 16), __uint_as_float(w[3] & 0xFFFF0000u));
            }
            __syncthreads();
            Bf = sBCf;
            Cf = sBCf + kTc * N;
        } else {
            Bf = reinterpret_cast<const float *>(sb);
            Cf = reinterpret_cast<const float *>(sb + kTileBC);
        }
        // two tokens per step: the second token's loads, delta and decays do not depend on the
        // first token's state, so they overlap its update
        int t = 0;
        for (; t + 2 <= L; t += 2) {
            float B0[N], C0[N], B1[N], C1[N];
            smem_row<N>(Bf + t * N, B0);
            smem_row<N>(Cf + t * N, C0);
            smem_row<N>(Bf + (t + 1) * N, B1);
            smem_row<N>(Cf + (t + 1) * N, C1);
            const float x0 = to_f32(xs[t * kCh + tid]), x1 = to_f32(xs[(t + 1) * kCh + tid]);
            const float dl0 = m1_delta<Tin>(to_f32(dts[t * kCh + tid]) + bias, a);
            const float dl1 = m1_delta<Tin>(to_f32(dts[(t + 1) * kCh + tid]) + bias, a);
            float y0 = m1_step<N>(h, A2, dl0, x0, B0, C0, Dd);
            float y1 = m1_step<N>(h, A2, dl1, x1, B1, C1, Dd);
            if (kGate) {
                y0 = silu_gate(y0, to_f32(zs[t * kCh + tid]));
                y1 = silu_gate(y1, to_f32(zs[(t + 1) * kCh + tid]));
            }
            y[(size_t)(tb + t) * Dc + d] = from_f32<Tin>(y0);
            y[(size_t)(tb + t + 1) * Dc + d] = from_f32<Tin>(y1);
        }
        if (t < L) {
            float B0[N], C0[N];
            smem_row<N>(Bf + t * N, B0);
            smem_row<N>(Cf + t * N, C0);
            const float x0 = to_f32(xs[t * kCh + tid]);
            const float dl0 = m1_delta<Tin>(to_f32(dts[t * kCh + tid]) + bias, a);
            float y0 = m1_step<N>(h, A2, dl0, x0, B0, C0, Dd);
            if (kGate) y0 = silu_gate(y0, to_f32(zs[t * kCh + tid]));
            y[(size_t)(tb + t) * Dc + d] = from_f32<Tin>(y0);
        }
        if (cur.ends_chunk()) {
            if (slot_usable(cs, a.null_block_id, a.num_slots, (tid == 0) ? a.err_word : nullptr))
                state_store2<N>(a.state_cache + ((size_t)cs * Dc + d) * N, h);
            if (a.chunk_slot) cs = a.chunk_slot[min(cur.k + 1, last)];
        }
        cur.next();
        __syncthreads();  // every thread is done with buffer (i & 1) and the fp32 rows before reuse
    }
}

// Decode: one CTA per (kReq requests, 64 channels), one channel per thread.  A thread loads the
// states of its requests (and A once) before computing any of them, so kReq state loads are in
// flight per thread and the grid has kReq times fewer waves.
constexpr int kReq = 2;

template <typename Tin, int N, bool kGate>
__global__ void __launch_bounds__(kCh) mamba1_update_kernel(const mamba1_args a) {
    const int tid = threadIdx.x;
    const int Dc = a.dim, G = a.ngroups;
    const int d = blockIdx.y * kCh + tid;
    const int g = d / (Dc / G);
    const int tpr = a.tokens_per_req;
    int32_t rs[kReq];
    bool live[kReq];
    bool any = false;
#pragma unroll
    for (int q = 0; q < kReq; ++q) {
        const int r = blockIdx.x * kReq + q;
        live[q] = false;
        rs[q] = 0;
        if (r >= a.num_seqs) continue;
        const int col = a.num_accepted_tokens ? a.num_accepted_tokens[r] : 0;
        if (col < 0 || col >= a.state_indices_cols) {
            if (tid == 0 && blockIdx.y == 0) report(a.err_word, SSD_DEVERR_COLUMN);
            continue;
        }
        const int32_t s0 = a.state_indices[(size_t)r * a.state_indices_cols + col];
        if (s0 == a.null_block_id) continue;  // CUDA-graph padding row
        if (s0 < 0 || s0 >= a.num_slots) {
            if (tid == 0 && blockIdx.y == 0) report(a.err_word, SSD_DEVERR_SLOT);
            continue;
        }
        live[q] = true;
        rs[q] = s0;
        any = true;
    }
    if (!any) return;
    constexpr float kLog2e = 1.4426950408889634f;
    float2 h[kReq][N / 2], A2[N / 2];
#pragma unroll
    for (int q = 0; q < kReq; ++q)
        if (live[q]) state_load2<N>(a.state_cache + ((size_t)rs[q] * Dc + d) * N, h[q]);
    state_load2<N>(a.A + (size_t)d * N, A2);
#pragma unroll
    for (int i = 0; i < N / 2; ++i) A2[i] = make_float2(A2[i].x * kLog2e, A2[i].y * kLog2e);
    const float Dd = a.D ? a.D[d] : 0.f;
    const float bias = a.dt_bias ? a.dt_bias[d] : 0.f;
    const Tin *x = static_cast<const Tin *>(a.x), *dt = static_cast<const Tin *>(a.dt);
    const Tin *Bp = static_cast<const Tin *>(a.B), *Cp = static_cast<const Tin *>(a.C);
    const Tin *z = static_cast<const Tin *>(a.z);
    Tin *y = static_cast<Tin *>(a.y);
#pragma unroll
    for (int q = 0; q < kReq; ++q) {
        if (!live[q]) continue;
        const int r = blockIdx.x * kReq + q;
        const int32_t *row_slots = a.state_indices + (size_t)r * a.state_indices_cols;
        for (int k = 0; k < tpr; ++k) {
            const size_t row = (size_t)r * tpr + k;
            float Bt[N], Ct[N];
            row_to_f32_ldg<N>(Bp + (row * G + g) * N, Bt);
            row_to_f32_ldg<N>(Cp + (row * G + g) * N, Ct);
            const float xv = ldg_f32(x + row * Dc + d);
            const float delta = m1_delta<Tin>(ldg_f32(dt + row * Dc + d) + bias, a);
            float yv = m1_step<N>(h[q], A2, delta, xv, Bt, Ct, Dd);
            if (kGate) yv = silu_gate(yv, ldg_f32(z + row * Dc + d));
            y[row * Dc + d] = from_f32<Tin>(yv);
            const int32_t ws = row_slots[k];
            if (slot_usable(ws, a.null_block_id, a.num_slots, tid == 0 ? a.err_word : nullptr))
                state_store2<N>(a.state_cache + ((size_t)ws * Dc + d) * N, h[q]);
        }
    }
}

template <typename Tin, int N>
cudaError_t launch_n(const mamba1_args &a, bool decode, cudaStream_t st) {
    const dim3 grid(a.num_seqs, a.dim / kCh);
    if (decode) {
        const dim3 dgrid((a.num_seqs + kReq - 1) / kReq, a.dim / kCh);
        if (a.z) mamba1_update_kernel<Tin, N, true><<<dgrid, kCh, 0, st>>>(a);
        else mamba1_update_kernel<Tin, N, false><<<dgrid, kCh, 0, st>>>(a);
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
