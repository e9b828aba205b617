// Depthwise causal conv1d in front of the SSM, with a conv-state cache.
//
// The step that produces x, B and C ("get hidden_states, B and C after
// depthwise convolution", MambaMixer2 listing of "[vllm] vLLM Mamba2 SSD 커널
// 웜업"), with the per-block conv state of "vLLM v0.20.0 하이브리드 SSM 모델을
// 위한 분산 서빙 추가" ("전체 흐름": [num_blocks, 3, 3072]).  For channel c and
// token t of a sequence,
//   out[t, c] = act(bias[c] + sum_{k<W} weight[c, k] * in[t - (W-1) + k, c]),
// with the W-1 inputs before the sequence's first token taken from its conv
// state (zeros without one).
//
// HBM-bound streaming work, no contraction.  The varlen (prefill) form streams
// TMA-loaded token tiles through shared memory (conv1d_tiled_kernel below); a
// second, small kernel then writes the conv states at chunk ends and sequence
// ends, ordered after the first on the stream, so all state reads precede all
// state writes.  The decode form runs one thread per (request, 8 channels)
// that reads its slot's history, applies the request's tokens and writes the
// new window back (conv1d_decode_kernel).  The outputs go straight to three
// tensors (x, B, C), the layout the SSM calls take.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <algorithm>

namespace ssd {
namespace {
using namespace tc;

constexpr int kVec = 8;        // channels per thread (16 bytes of bf16)
constexpr int kConvThreads = 128;

struct ConvParams {
    int T, S, K, tpr, D, dim_x, dim_bc, num_slots, null_id, activation;
    bool decode;               // requests of tpr tokens; null slot = padding (skipped)
    const float *weight, *bias;
    const int32_t *cu_seqlens, *cu_chunk, *last_chunk, *init_slot, *out_slot, *chunk_slot;
    uint32_t *err;
};

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
    struct Raw { uint4 u; };
    static __device__ __forceinline__ Raw load_raw(const __nv_bfloat16 *p) { return {*reinterpret_cast<const uint4 *>(p)}; }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&v)[kVec]) {
        const uint32_t w[4] = {r.u.x, r.u.y, r.u.z, r.u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ void load(const __nv_bfloat16 *p, float (&v)[kVec]) {
        const uint4 u = *reinterpret_cast<const uint4 *>(p);
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
        }
    }
    static __device__ __forceinline__ void store(__nv_bfloat16 *p, const float (&v)[kVec]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<const uint32_t *>(&h);
        }
        *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
    }
    static __device__ __forceinline__ void store_raw(__nv_bfloat16 *p, const Raw &r) {
        *reinterpret_cast<uint4 *>(p) = r.u;
    }
    // exact copy of an input vector (states hold inputs bit for bit)
    static __device__ __forceinline__ void copy(__nv_bfloat16 *dst, const __nv_bfloat16 *src) {
        *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
    }
};
template <> struct Vec8<float> {
    struct Raw { float4 a, b; };
    static __device__ __forceinline__ Raw load_raw(const float *p) {
        return {reinterpret_cast<const float4 *>(p)[0], reinterpret_cast<const float4 *>(p)[1]};
    }
    static __device__ __forceinline__ void unpack(const Raw &r, float (&v)[kVec]) {
        v[0] = r.a.x; v[1] = r.a.y; v[2] = r.a.z; v[3] = r.a.w;
        v[4] = r.b.x; v[5] = r.b.y; v[6] = r.b.z; v[7] = r.b.w;
    }
    static __device__ __forceinline__ void load(const float *p, float (&v)[kVec]) {
        const float4 a = reinterpret_cast<const float4 *>(p)[0], b = reinterpret_cast<const float4 *>(p)[1];
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
        v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ void store(float *p, const float (&v)[kVec]) {
        reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
        reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
    }
    static __device__ __forceinline__ void store_raw(float *p, const Raw &r) {
        reinterpret_cast<float4 *>(p)[0] = r.a;
        reinterpret_cast<float4 *>(p)[1] = r.b;
    }
    static __device__ __forceinline__ void copy(float *dst, const float *src) {
        reinterpret_cast<float4 *>(dst)[0] = reinterpret_cast<const float4 *>(src)[0];
        reinterpret_cast<float4 *>(dst)[1] = reinterpret_cast<const float4 *>(src)[1];
    }
};

// sequence holding token t: the last r with cu_seqlens[r] <= t (empty sequences skipped)
__device__ __forceinline__ int seq_of(const int32_t *cu, int S, int t) {
    int lo = 0, hi = S - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (cu[mid] <= t) lo = mid;
        else hi = mid - 1;
    }
    while (lo + 1 < S && cu[lo + 1] <= t) ++lo;  // past empty sequences that start at t
    return lo;
}

__device__ __forceinline__ int seq_start(const ConvParams &p, int r) { return p.decode ? r * p.tpr : p.cu_seqlens[r]; }
__device__ __forceinline__ int seq_end(const ConvParams &p, int r) { return p.decode ? (r + 1) * p.tpr : p.cu_seqlens[r + 1]; }

// conv-state slot sequence r starts from: -1 for zeros, -2 for a skipped (padding) request
__device__ __forceinline__ int history_slot(const ConvParams &p, int r, bool report_errors) {
    const int32_t s = p.init_slot ? p.init_slot[r] : p.null_id;
    if (s == p.null_id) return p.decode ? -2 : -1;
    if (s < 0 || s >= p.num_slots) {
        if (report_errors) report(p.err, SSD_DEVERR_SLOT);
        return p.decode ? -2 : -1;
    }
    return s;
}

// ---- decode: one thread per (request, 8 channels) ------------------------------------------
// A request's W-1 history rows come from its slot, its tokens follow, and the window after its
// last token goes back to the same slot: the thread reads every row it writes before writing
// it, so no second kernel is needed.  One CTA row of threads per request keeps every request
// (and its slot's latency) in flight at once; padding requests (null slot) read and write nothing.
template <typename Tin, int W>
__global__ void __launch_bounds__(kConvThreads) conv1d_decode_kernel(const Tin *__restrict__ xbc, Tin *state,
                                                                     Tin *__restrict__ x_out, Tin *__restrict__ B_out,
                                                                     Tin *__restrict__ C_out, ConvParams p) {
    const int vec = blockIdx.x * kConvThreads + threadIdx.x;
    const int r = blockIdx.y;
    if (vec * kVec >= p.D) return;
    const int hslot = history_slot(p, r, vec == 0);
    if (hslot < 0) return;  // padding (or an out-of-range slot, reported)
    const int c0 = vec * kVec;
    Tin *out;
    int ocol, ostride;
    if (c0 < p.dim_x) {
        out = x_out, ocol = c0, ostride = p.dim_x;
    } else if (c0 < p.dim_x + p.dim_bc) {
        out = B_out, ocol = c0 - p.dim_x, ostride = p.dim_bc;
    } else {
        out = C_out, ocol = c0 - p.dim_x - p.dim_bc, ostride = p.dim_bc;
    }
    Tin *slot = state + (size_t)hslot * (W - 1) * p.D + c0;
    float win[W - 1][kVec];  // win[0] oldest
#pragma unroll
    for (int j = 0; j < W - 1; ++j) Vec8<Tin>::load(slot + (size_t)j * p.D, win[j]);
    // the thread's kVec x W weights are contiguous ([D, W] layout): W kVec / 4 16-byte loads
    float wf[W * kVec], w[W][kVec], b[kVec];
#pragma unroll
    for (int j = 0; j < W * kVec / 4; ++j) {
        const float4 v = reinterpret_cast<const float4 *>(p.weight + (size_t)c0 * W)[j];
        wf[4 * j] = v.x; wf[4 * j + 1] = v.y; wf[4 * j + 2] = v.z; wf[4 * j + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
#pragma unroll
        for (int k = 0; k < W; ++k) w[k][i] = wf[i * W + k];
        b[i] = p.bias ? p.bias[c0 + i] : 0.f;
    }
    for (int k = 0; k < p.tpr; ++k) {
        const int t = r * p.tpr + k;
        float cur[kVec], o[kVec];
        Vec8<Tin>::load(xbc + (size_t)t * p.D + c0, cur);
#pragma unroll
        for (int i = 0; i < kVec; ++i) {
            float acc = b[i];
#pragma unroll
            for (int kk = 0; kk < W - 1; ++kk) acc = fmaf(w[kk][i], win[kk][i], acc);
            acc = fmaf(w[W - 1][i], cur[i], acc);
            o[i] = p.activation ? silu(acc) : acc;
        }
        Vec8<Tin>::store(out + (size_t)t * ostride + ocol, o);
#pragma unroll
        for (int jj = 0; jj + 1 < W - 1; ++jj)
#pragma unroll
            for (int i = 0; i < kVec; ++i) win[jj][i] = win[jj + 1][i];
#pragma unroll
        for (int i = 0; i < kVec; ++i) win[W - 2][i] = cur[i];
    }
    // the window holds exact input values (widened from the token dtype), so storing them back
    // reproduces the inputs bit for bit
#pragma unroll
    for (int j = 0; j < W - 1; ++j) Vec8<Tin>::store(slot + (size_t)j * p.D, win[j]);
}

// ---- prefill: token tiles staged in shared memory ---------------------------------------
// The varlen (prefill) form streams tiles of kTileTok tokens x 512 bytes of channels (256 bf16
// or 128 fp32), plus the W-1 rows before them, into shared memory, one TMA box per tile.
// About two 256-thread CTAs per SM, each owning one channel tile and walking token tiles, keep
// the next tile of each CTA in flight while this one is computed (about 100 KB of loads per
// SM).  96-token tiles in two stages beat 64-token tiles in three (3.45 vs 3.60 ms on 524,288
// tokens x 10,240 channels): fewer halo rows and tile hand-offs per token.  Each thread then
// computes 8 channels x (96 / groups) tokens from shared memory with a sliding window of the W-1
// previous inputs in registers, restarted from the history at every sequence start.
constexpr int kTileTok = 96;
constexpr int kTileRowBytes = 512;
constexpr int kTiledThreads = 256;
constexpr int kTiledStages = 2;

template <int W>
constexpr int tiled_smem_bytes() { return kTiledStages * (kTileTok + W - 1) * kTileRowBytes; }

template <typename Tin, int W>
__global__ void __launch_bounds__(kTiledThreads, 2) conv1d_tiled_kernel(const __grid_constant__ CUtensorMap tmx,
                                                                     const Tin *__restrict__ xbc,
                                                                     const Tin *__restrict__ state,
                                                                     Tin *__restrict__ x_out, Tin *__restrict__ B_out,
                                                                     Tin *__restrict__ C_out, ConvParams p) {
    constexpr int kChT = kTileRowBytes / (int)sizeof(Tin);  // channels per tile
    constexpr int kThrVec = kChT / kVec;                    // thread vectors across a tile row
    constexpr int kGroups = kTiledThreads / kThrVec;        // token groups
    constexpr int kRunT = kTileTok / kGroups;               // tokens per thread
    constexpr int kRows = kTileTok + W - 1;
    constexpr int kStageBytes = kRows * kTileRowBytes;
    extern __shared__ __align__(128) uint8_t tsm[];
    __shared__ uint64_t full[kTiledStages];  // TMA completion of each stage

    // CTA b keeps one channel tile, ct = b % nct, and walks token tiles tt0, tt0 + step, ...: its
    // weights are loaded once, and the sequence of its tokens only moves forward
    const int tid = threadIdx.x;
    const int nct = (p.D + kChT - 1) / kChT;
    const int ntt = (p.T + kTileTok - 1) / kTileTok;
    const int step = gridDim.x / nct;
    const int ct = blockIdx.x % nct, tt0 = blockIdx.x / nct;
    if (step < 1 || tt0 >= step) return;  // grid is a multiple of nct (host); CTA-uniform
    const int ntiles = tt0 < ntt ? (ntt - tt0 + step - 1) / step : 0;  // this CTA's tiles

    if (tid == 0) {
        for (int s = 0; s < kTiledStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    // one TMA box per tile: kRows rows (the W-1 before the tile included; rows outside the
    // tensor read as zeros and are never used) x 512 bytes of channels
    auto load_tile = [&](int k, int stage) {
        if (tid == 0 && k < ntiles) {
            fence_proxy_async_smem();  // this stage's earlier readers are ordered before the copy
            mbar_arrive_expect_tx(&full[stage], kStageBytes);
            tma_load_2d(tsm + stage * kStageBytes, &tmx, ct * kChT, (tt0 + k * step) * kTileTok - (W - 1), &full[stage]);
        }
    };

    const int v = tid % kThrVec, grp = tid / kThrVec;
    const int c0 = ct * kChT + v * kVec;
    const bool active = c0 < p.D;
    float w[W][kVec], b[kVec];
#pragma unroll
    for (int i = 0; i < kVec; ++i) {
#pragma unroll
        for (int k = 0; k < W; ++k) w[k][i] = active ? __ldg(p.weight + (size_t)(c0 + i) * W + k) : 0.f;
        b[i] = active && p.bias ? __ldg(p.bias + c0 + i) : 0.f;
    }
    Tin *out;
    int ocol, ostride;
    if (c0 < p.dim_x) {
        out = x_out, ocol = c0, ostride = p.dim_x;
    } else if (c0 < p.dim_x + p.dim_bc) {
        out = B_out, ocol = c0 - p.dim_x, ostride = p.dim_bc;
    } else {
        out = C_out, ocol = c0 - p.dim_x - p.dim_bc, ostride = p.dim_bc;
    }
    // the sequence of this thread's first token in its first tile; it only moves forward
    int r = seq_of(p.cu_seqlens, p.S, min(tt0 * kTileTok + grp * kRunT, p.T - 1));
    int s0 = p.cu_seqlens[r], e0 = p.cu_seqlens[r + 1];
    int hslot = history_slot(p, r, c0 == 0 && grp == 0 && tt0 == 0);
    bool bad = false;

#pragma unroll
    for (int s = 0; s < kTiledStages - 1; ++s) load_tile(s, s);
    for (int k = 0; k < ntiles; ++k) {
        load_tile(k + kTiledStages - 1, (k + kTiledStages - 1) % kTiledStages);
        // tile k is in shared memory (a bounded wait; on a timeout the CTA reports and stops)
        if (!__syncthreads_and(mbar_wait(&full[k % kTiledStages], (k / kTiledStages) & 1))) {
            if (tid == 0) report(p.err, SSD_DEVERR_TIMEOUT);
            break;
        }
        const uint8_t *st = tsm + (k % kTiledStages) * kStageBytes;
        const int tt = tt0 + k * step;
        const int ta = tt * kTileTok + grp * kRunT;  // this thread's first token
        const int tz = min(ta + kRunT, p.T);
        if (active && ta < p.T && !bad) {
            // shared-memory row of token t (the tile holds tokens tt*kTileTok - (W-1) ...)
            auto srow = [&](int t) {
                return reinterpret_cast<const Tin *>(st + (t - tt * kTileTok + (W - 1)) * kTileRowBytes) + v * kVec;
            };
            float win[W - 1][kVec];
            auto fill_window = [&](int t) {  // the W-1 inputs before token t, within t's sequence
#pragma unroll
                for (int jj = 0; jj < W - 1; ++jj) {
                    const int tau = t - (W - 1) + jj;
                    if (tau >= s0) {
                        Vec8<Tin>::load(srow(tau), win[jj]);
                    } else if (hslot >= 0) {
                        Vec8<Tin>::load(state + ((size_t)hslot * (W - 1) + (W - 1) - (s0 - tau)) * p.D + c0, win[jj]);
                    } else {
#pragma unroll
                        for (int i = 0; i < kVec; ++i) win[jj][i] = 0.f;
                    }
                }
            };
            // move to the sequence holding ta (empty sequences have no tokens to visit)
            auto advance = [&](int t) {
                while (t >= e0) {
                    if (r + 1 >= p.S) {  // cu_seqlens does not end at T
                        if (c0 == 0 && grp == 0) report(p.err, SSD_DEVERR_METADATA);
                        bad = true;
                        return;
                    }
                    ++r;
                    s0 = p.cu_seqlens[r];
                    e0 = p.cu_seqlens[r + 1];
                    hslot = history_slot(p, r, c0 == 0 && grp == 0);
                }
            };
            advance(ta);
            if (!bad && tz == ta + kRunT && ta - (W - 1) >= s0 && tz <= e0) {
                // the whole run and its window lie inside one sequence (the common case): inputs
                // straight from shared memory, the loop fully unrolled so the window shift is
                // register renaming, no boundary checks
                float wv[W][kVec];
#pragma unroll
                for (int jj = 0; jj < W - 1; ++jj) Vec8<Tin>::load(srow(ta - (W - 1) + jj), wv[jj]);
#pragma unroll
                for (int j = 0; j < kRunT; ++j) {
                    Vec8<Tin>::load(srow(ta + j), wv[W - 1]);
                    float o[kVec];
#pragma unroll
                    for (int i = 0; i < kVec; ++i) {
                        float acc = b[i];
#pragma unroll
                        for (int kk = 0; kk < W; ++kk) acc = fmaf(w[kk][i], wv[kk][i], acc);
                        o[i] = p.activation ? silu(acc) : acc;
                    }
                    Vec8<Tin>::store(out + (size_t)(ta + j) * ostride + ocol, o);
#pragma unroll
                    for (int kk = 0; kk + 1 < W; ++kk)
#pragma unroll
                        for (int i = 0; i < kVec; ++i) wv[kk][i] = wv[kk + 1][i];
                }
            } else {
                if (!bad) fill_window(ta);
                for (int t = ta; t < tz && !bad; ++t) {
                    if (t >= e0) {
                        advance(t);
                        if (bad) break;
                        fill_window(t);
                    }
                    float cur[kVec];
                    Vec8<Tin>::load(srow(t), cur);
                    float o[kVec];
    #pragma unroll
                    for (int i = 0; i < kVec; ++i) {
                        float acc = b[i];
    #pragma unroll
                        for (int kk = 0; kk < W - 1; ++kk) acc = fmaf(w[kk][i], win[kk][i], acc);
                        acc = fmaf(w[W - 1][i], cur[i], acc);
                        o[i] = p.activation ? silu(acc) : acc;
                    }
                    Vec8<Tin>::store(out + (size_t)t * ostride + ocol, o);
    #pragma unroll
                    for (int jj = 0; jj + 1 < W - 1; ++jj)
    #pragma unroll
                        for (int i = 0; i < kVec; ++i) win[jj][i] = win[jj + 1][i];
    #pragma unroll
                    for (int i = 0; i < kVec; ++i) win[W - 2][i] = cur[i];
                }
            }
        }
        __syncthreads();  // every thread is done with this stage before it is refilled
    }
}

// Conv states of sequence r: the W-1 inputs ending at each of its chunk ends and at its
// last token (for a request of the decode call: its own slot).  The history this needs
// is read into registers before any store, so a slot may be both read and written.
template <typename Tin, int W>
__global__ void __launch_bounds__(kConvThreads) conv_state_kernel(const Tin *__restrict__ xbc, Tin *state, ConvParams p) {
    const int vec = blockIdx.x * kConvThreads + threadIdx.x;
    const int r = blockIdx.y;
    if (vec * kVec >= p.D) return;
    const int c0 = vec * kVec;
    const int hslot = history_slot(p, r, false);
    if (hslot == -2) return;  // padding request
    const int s0 = seq_start(p, r), e0 = seq_end(p, r);
    if (s0 < 0 || e0 < s0 || e0 > p.T) {
        if (vec == 0) report(p.err, SSD_DEVERR_METADATA);
        return;
    }
    Tin hist[W - 1][kVec];
#pragma unroll
    for (int j = 0; j < W - 1; ++j)
#pragma unroll
        for (int i = 0; i < kVec; ++i)
            hist[j][i] = hslot >= 0 ? state[((size_t)hslot * (W - 1) + j) * p.D + c0 + i] : Tin(0.f);
    // window ending at token e (inclusive) into slot s
    auto store_window = [&](int e, int32_t s) {
        if (s == p.null_id) return;
        if (s < 0 || s >= p.num_slots) {
            if (vec == 0) report(p.err, SSD_DEVERR_SLOT);
            return;
        }
#pragma unroll
        for (int j = 0; j < W - 1; ++j) {
            const int tau = e - (W - 2) + j;
            Tin *dst = state + ((size_t)s * (W - 1) + j) * p.D + c0;
            if (tau >= s0) {
                Vec8<Tin>::copy(dst, xbc + (size_t)tau * p.D + c0);
            } else {
#pragma unroll
                for (int i = 0; i < kVec; ++i) dst[i] = hist[(W - 1) - (s0 - tau)][i];
            }
        }
    };
    if (p.decode) {
        store_window(e0 - 1, p.init_slot[r]);
        return;
    }
    if (p.chunk_slot && p.last_chunk) {
        const int first = r > 0 ? p.last_chunk[r - 1] + 1 : 0, last = p.last_chunk[r];
        if (first < 0 || last >= p.K) {
            if (vec == 0) report(p.err, SSD_DEVERR_METADATA);
            return;
        }
        // kBatchK chunks at a time: their windows are loaded before any is stored, so the loads
        // overlap instead of one chunk's latency after another's
        constexpr int kBatchK = 4;
        for (int k0 = first; k0 <= last; k0 += kBatchK) {
            typename Vec8<Tin>::Raw raw[kBatchK][W - 1];
            int ends[kBatchK];
#pragma unroll
            for (int kk = 0; kk < kBatchK; ++kk) {
                const int k = k0 + kk;
                ends[kk] = k <= last ? p.cu_chunk[k + 1] - 1 : -1;  // the chunk's last token
#pragma unroll
                for (int j = 0; j < W - 1; ++j) {
                    const int tau = ends[kk] - (W - 2) + j;
                    if (k <= last && tau >= s0 && ends[kk] < e0) raw[kk][j] = Vec8<Tin>::load_raw(xbc + (size_t)tau * p.D + c0);
                }
            }
#pragma unroll
            for (int kk = 0; kk < kBatchK; ++kk) {
                const int k = k0 + kk;
                if (k > last) break;
                const int e = ends[kk];
                if (e < s0 || e >= e0) {
                    if (vec == 0) report(p.err, SSD_DEVERR_METADATA);
                    continue;
                }
                const int32_t sl = p.chunk_slot[k];
                if (sl == p.null_id) continue;
                if (sl < 0 || sl >= p.num_slots) {
                    if (vec == 0) report(p.err, SSD_DEVERR_SLOT);
                    continue;
                }
#pragma unroll
                for (int j = 0; j < W - 1; ++j) {
                    const int tau = e - (W - 2) + j;
                    Tin *dst = state + ((size_t)sl * (W - 1) + j) * p.D + c0;
                    if (tau >= s0) {
                        Vec8<Tin>::store_raw(dst, raw[kk][j]);
                    } else {
#pragma unroll
                        for (int i = 0; i < kVec; ++i) dst[i] = hist[(W - 1) - (s0 - tau)][i];
                    }
                }
            }
        }
    }
    if (p.out_slot) store_window(e0 - 1, p.out_slot[r]);
}

template <typename Tin, int W>
cudaError_t launch_w(const ssd_conv1d_args &a, const ConvParams &p, cudaStream_t st) {
    const int vecs = p.D / kVec;
    const Tin *xbc = static_cast<const Tin *>(a.xbc);
    Tin *state = static_cast<Tin *>(a.conv_state);
    if (p.T > 0 && !p.decode) {
        // persistent: two CTAs per SM, each walking tiles with a grid stride
        static int sms = 0;
        if (sms == 0) {
            int dev = 0;
            cudaGetDevice(&dev);
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (sms <= 0) sms = 1;
        }
        constexpr int smem = tiled_smem_bytes<W>();
        cudaError_t e = cudaFuncSetAttribute(conv1d_tiled_kernel<Tin, W>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
        // one channel tile per CTA, as many token-tile walkers per channel tile as fill two CTAs per SM
        const int nct = (p.D + kTileRowBytes / (int)sizeof(Tin) - 1) / (kTileRowBytes / (int)sizeof(Tin));
        const int ntt = (p.T + kTileTok - 1) / kTileTok;
        const int step = std::max(1, std::min(ntt, (2 * sms) / nct));
        const long long grid = (long long)nct * step;
        if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
        CUtensorMap tmx;
        constexpr int kChT = kTileRowBytes / (int)sizeof(Tin);
        if (!make_tmap_2d(&tmx, sizeof(Tin) == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32,
                          a.xbc, (uint64_t)p.D, (uint64_t)p.T, (uint64_t)p.D * sizeof(Tin), kChT, kTileTok + W - 1))
            return cudaErrorInvalidValue;
        conv1d_tiled_kernel<Tin, W><<<(unsigned)grid, kTiledThreads, smem, st>>>(tmx, xbc, state, static_cast<Tin *>(a.x_out),
                                                                         static_cast<Tin *>(a.B_out),
                                                                         static_cast<Tin *>(a.C_out), p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    } else if (p.T > 0) {  // decode: outputs and the new window in one kernel
        const dim3 gridd((vecs + kConvThreads - 1) / kConvThreads, p.S);
        conv1d_decode_kernel<Tin, W><<<gridd, kConvThreads, 0, st>>>(xbc, state, static_cast<Tin *>(a.x_out),
                                                                     static_cast<Tin *>(a.B_out),
                                                                     static_cast<Tin *>(a.C_out), p);
        return cudaGetLastError();
    }
    const bool any_state = p.decode || p.out_slot || (p.chunk_slot && p.last_chunk);
    if (any_state && p.S > 0) {
        const dim3 grid2((vecs + kConvThreads - 1) / kConvThreads, p.S);
        conv_state_kernel<Tin, W><<<grid2, kConvThreads, 0, st>>>(xbc, state, p);
    }
    return cudaGetLastError();
}

template <typename Tin>
cudaError_t launch_t(const ssd_conv1d_args &a, const ConvParams &p, cudaStream_t st) {
    switch (a.width) {
        case 2: return launch_w<Tin, 2>(a, p, st);
        case 3: return launch_w<Tin, 3>(a, p, st);
        default: return launch_w<Tin, 4>(a, p, st);
    }
}

}  // namespace

cudaError_t conv1d_launch(const ssd_conv1d_args &a, bool decode, cudaStream_t st) {
    ConvParams p;
    p.T = a.total_tokens;
    p.S = a.num_seqs;
    p.K = decode ? 0 : a.num_chunks;
    p.tpr = decode ? a.tokens_per_req : 0;
    p.D = a.dim_x + 2 * a.dim_bc;
    p.dim_x = a.dim_x;
    p.dim_bc = a.dim_bc;
    p.num_slots = a.num_slots;
    p.null_id = a.null_block_id;
    p.activation = a.activation;
    p.decode = decode;
    p.weight = a.weight;
    p.bias = a.bias;
    p.cu_seqlens = decode ? nullptr : a.cu_seqlens;
    p.cu_chunk = decode ? nullptr : a.cu_chunk_seqlens;
    p.last_chunk = decode ? nullptr : a.last_chunk_indices;
    p.init_slot = a.init_slot;
    p.out_slot = decode ? nullptr : a.out_slot;
    p.chunk_slot = decode ? nullptr : a.chunk_slot;
    p.err = a.err_word;
    return a.dtype == SSD_BF16 ? launch_t<__nv_bfloat16>(a, p, st) : launch_t<float>(a, p, st);
}

}  // namespace ssd
