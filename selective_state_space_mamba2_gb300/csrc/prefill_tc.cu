// Fused SSD prefill on the sm_103a tensor cores (bf16 inputs, fp32 state).
//
// The chunked scan of "[vllm] vLLM Mamba2 SSD 커널 웜업" (section
// "mamba_mixer2.py 변경 사항 (핵심)"), fused into one kernel: one CTA walks one
// (sequence, head) through its chunks in blocks of 128 tokens, keeping the
// fp32 state in registers, so the state crosses HBM only where the method
// requires it -- the optional initial state is read once and the state at the
// end of every chunk is stored to its cache slot (prefix caching, "청크 기반
// 프리픽스 캐싱" on "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링").
//
// A small kernel in front (prep_kernel) converts B and C to fp16 once per call
// and writes delta and its in-block cumsum c for every head and token.  Per
// block of L <= 128 tokens [tb, tb+L), the four dense contractions run as
// tcgen05.mma tiles with fp32 accumulators and fp16 operands (x, P, w x and
// the carried state are rounded to fp16, whose 11-bit significand keeps their
// rounding error 8x below bf16's):
//   M1  S  = C B^T                  [128 x 128], K = dstate   (SS, K/K-major)
//   M2  Y1 = P X                    [128 x  64], K = tokens   (TS: P in TMEM)
//        P[t,s] = exp(c_t - c_s) delta_s S[t,s] for s <= t, plus D on the diagonal
//   M3  Y2 = C Hprev^T              [128 x  64], K = dstate   (SS, B MN-major)
//   M4  dS = B^T (w x),  w_s = exp(c_L - c_s) delta_s   [dstate x 64]   (SS, MN/MN)
// and then y_t = Y1 + exp(c_t) Y2,   state <- exp(c_L) state + dS.
//
// Decays are factored so that an element of P costs two multiplies.  For a
// 32-column group j lying entirely below row t's group, exp(c_t - c_s) is split
// at the group's last row e: exp(c_t - c_e) exp(c_e - c_s), both factors <= 1.
// The diagonal group is split at its first row b instead (exp(c_t - c_b) <= 1,
// exp(c_b - c_s) >= 1), which keeps both factors normal fp32 numbers while the
// group's decay c_b - c_e is at most 80; beyond that it takes one exponential
// per element, in an out-of-line function.
//
// Only the state itself is a serial dependency from block to block (64 FMAs
// per thread); everything else is pipelined.  One CTA per SM, 320 threads:
//   warps 0-3  "producer" warpgroup, one block ahead: the column factors from
//              delta and c, w x and x -> fp16, the P pass (S -> P in TMEM, in place)
//   warps 4-7  "consumer" warpgroup: state update, the fp16 state tile for
//              the next block's M3, the chunk-boundary stores, y (staged in the
//              spent x slot and written by one tensor copy per whole block)
//   warp 8     TMA producer: C/B tiles in two stages, x tiles in three (128-byte
//              swizzle)
//   warp 9     TMEM allocation (512 columns) and MMA issue
// Thread t of a warpgroup owns TMEM lane t: token row t of S, Y1, Y2 and
// dstate row t of dS and of the state.  Every mbarrier wait is bounded; on a
// timeout the CTA reports SSD_DEVERR_TIMEOUT, drains its own in-flight copies
// and MMAs, frees its TMEM and exits.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

#include <algorithm>

namespace ssd {

struct TcParams {
    int T, S, K, H, G;
    int dt_softplus;
    float dt_min, dt_max;
    int num_slots, null_id;
    const __nv_bfloat16 *dt;
    const float *A, *D, *dt_bias;
    const int32_t *cu_seqlens, *cu_chunk, *last_chunk;
    const int32_t *init_slot, *chunk_slot;
    float *cache;
    const __nv_bfloat16 *z;  // output gate [T, H, P] or NULL
    __nv_bfloat16 *y;
    uint32_t *err;
    const int32_t *seq_order;
    long long wait_limit;  // cycles a device-side wait may take before the CTA gives up
    const float *cum;      // [H, T] in-block inclusive cumsum of delta * A (written by prep_kernel)
    const float *delta;    // [H, T] delta (written by prep_kernel)
    int nseg;              // segments each sequence is cut into (1: none)
    float *seg_state;      // [S, nseg - 1, H, P, N]: state at the end of segments 0 .. nseg - 2
    float *seg_decay;      // [S, nseg - 1, H]: for segments 1 .. nseg - 2, the product of their decays
};

namespace {
using namespace tc;

constexpr int kL = 128;  // tokens per block
constexpr int kP = 64;   // headdim
constexpr int kN = 128;  // dstate
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
// TMEM columns
constexpr uint32_t COL_S0 = 0;     // S of even blocks (128 fp32 columns); P over its first 64
constexpr uint32_t COL_S1 = 128;   // S of odd blocks
constexpr uint32_t COL_Y1 = 256;   // P X
constexpr uint32_t COL_Y2 = 320;   // C Hprev^T, even / odd blocks at +0 / +64
constexpr uint32_t COL_DS = 448;   // B^T (w x)
// shared memory (offsets from the 1024-aligned dynamic base)
constexpr uint32_t CB_STAGE = 65536;         // C 32 KB | B 32 KB (fp16)
constexpr uint32_t X_STAGE = 16384;          // x tile; then its fp16 copy; then y staging
constexpr int kCbStages = 2, kXStages = 3;
constexpr uint32_t OFF_X = kCbStages * CB_STAGE;
constexpr uint32_t OFF_XW = OFF_X + kXStages * X_STAGE;  // w x (fp16)
constexpr uint32_t OFF_H = OFF_XW + 16384;   // fp16 state entering the block
constexpr uint32_t OFF_F = OFF_H + 16384;    // column factors (two kinds), c_t and delta_t: [2 blocks][4][128]
constexpr uint32_t OFF_E = OFF_F + 4096;     // exp(c_t) per block, ring of 4 [4][128]
constexpr uint32_t OFF_DEC = OFF_E + 2048;   // exp(c_L) per block, ring of 4
constexpr uint32_t OFF_TM = OFF_DEC + 16;    // TMEM base address
constexpr uint32_t OFF_INFO = OFF_TM + 16;   // the CTA's part of its sequence [4]
constexpr uint32_t OFF_BAR = OFF_INFO + 16;  // mbarriers
constexpr uint32_t kSmemBytes = OFF_BAR + 24 * 8;
constexpr int kRing = 4;

enum {
    FULL_CB0 = 0, FULL_CB1, EMPTY_CB0, EMPTY_CB1,      // C/B ring: freed once M3 of the block is done
    FULL_X0, FULL_X1, FULL_X2, EMPTY_X0, EMPTY_X1, EMPTY_X2,  // x ring: freed after y (EMPTY: 4 arrivals)
    S_RDY0, S_RDY1,                                    // S of the block, per S buffer
    OPS_W,     // producer wg: w x and fp16 x of the block are in smem          (4 arrivals)
    PRDY0, PRDY1,  // producer wg: P of the block is in TMEM, per S buffer          (4)
                   // (one barrier per buffer keeps each waiter within one phase of its
                   // barrier whichever order M1 of the next block and M2 of this one go out in)
    OPS_H,     // consumer wg: fp16 state entering the block is in smem         (4)
    DS_FREE,   // consumer wg: read dS of the previous block                    (4)
    Y1_FREE,   // consumer wg: read Y1 of the previous block                    (4)
    ACC_DS,    // M4 of the block done (also frees w x)
    H_FREE,    // M3 of the block done (the state tile may be rewritten)
    ACC_Y,     // M2 and M3 of the block done
    DRAIN,
    NBAR
};
constexpr uint32_t BAR_PG = 1;  // named barrier of the producer warpgroup
constexpr uint32_t BAR_CG = 2;  // named barrier of the consumer warpgroup

__device__ __forceinline__ bool named_bar_and(uint32_t id, uint32_t n, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\tsetp.ne.u32 q, %1, 0;\n\tbar.red.and.pred p, %2, %3, q;\n\tselp.u32 %0, 1, 0, "
        "p;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)v), "r"(id), "r"(n)
        : "memory");
    return r != 0;
}

// One lane per warp polls the barrier; the warp learns the outcome by shuffle.
__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, long long limit) {
    bool ok = true;
    if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, limit);
    ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
    __syncwarp();
    return ok;
}

// Walks the blocks of one sequence (or of one segment of it, from any block
// start): chunks up to last, each cut into blocks of at most kL tokens that
// never cross a chunk end.  The end of the
// following chunk is loaded one chunk ahead (from a clamped index, so the
// load is unconditional), so moving to the next chunk never waits on memory.
struct Cursor {
    const int32_t *cu_chunk;
    int k, last, tb, ce, ce_next;
    // from block start tb inside chunk k
    __device__ void start_at(const int32_t *cc, int k_, int tb_, int last_) {
        cu_chunk = cc;
        k = k_;
        last = last_;
        tb = tb_;
        ce = cc[k_ + 1];
        ce_next = cc[min(k_ + 2, last_ + 1)];
    }
    __device__ int len() const { return min(kL, ce - tb); }
    __device__ bool ends_chunk() const { return tb + len() == ce; }
    __device__ void next() {
        tb += len();
        if (tb == ce && k < last) {
            ++k;
            ce = ce_next;
            ce_next = cu_chunk[min(k + 2, last + 1)];
        }
    }
};

// What the producer warpgroup needs of row t of a block [tb, tb + L): delta, the in-block
// cumsum, and the cumsum at the end of each 32-row group (row min(32 j + 31, L - 1)).
struct RowVals {
    float c, d, g[4];
    __device__ __forceinline__ void load(const float *cum, const float *dl, int tb, int L, int t) {
        const int r = min(t, L - 1);
        c = cum[tb + r];
        d = t < L ? dl[tb + r] : 0.f;
#pragma unroll
        for (int j = 0; j < 4; ++j) g[j] = cum[tb + min(32 * j + 31, L - 1)];
    }
};

// The diagonal group of the P pass when the group's decay is beyond the factored range: one
// exponential per element.  Out of line: it is rarely taken, and the P pass's common path stays
// small in the instruction cache.  Reads S from s_col, writes P (fp16) to p_col; cc and dd are the
// group's cumsum and delta values.  Called by a whole warp.
__device__ __noinline__ void diag_group_per_element(uint32_t s_col, uint32_t p_col, const float *cc, const float *dd,
                                                     float c, float Dh, int lane) {
    uint32_t v[32], pk[16];
    tmem_ld32(s_col, v);
    const float4 *c4 = reinterpret_cast<const float4 *>(cc);
    const float4 *d4 = reinterpret_cast<const float4 *>(dd);
    tmem_ld_wait();
#pragma unroll
    for (int u4 = 0; u4 < 8; ++u4) {
        const float4 cs = c4[u4], ds = d4[u4];
        const float cv[4] = {cs.x, cs.y, cs.z, cs.w}, dv[4] = {ds.x, ds.y, ds.z, ds.w};
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int u = 4 * u4 + e;
            const float ex = __expf(fminf(c - cv[e], 0.f));
            const float val = __uint_as_float(v[u]) * ex * dv[e];
            pv[e] = (u < lane) ? val : ((u == lane) ? val + Dh : 0.f);
        }
        pk[2 * u4] = pack_f16_sat(pv[0], pv[1]);
        pk[2 * u4 + 1] = pack_f16_sat(pv[2], pv[3]);
    }
    tmem_st16(p_col, pk);
}

// fp16 copy of a state row (dstate row n: its 64 headdim values) into the M3 operand tile
__device__ __forceinline__ void store_state_row(uint8_t *sH, int n, const float (&st)[kP]) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 v;
        v.x = pack_f16_sat(st[8 * c + 0], st[8 * c + 1]);
        v.y = pack_f16_sat(st[8 * c + 2], st[8 * c + 3]);
        v.z = pack_f16_sat(st[8 * c + 4], st[8 * c + 5]);
        v.w = pack_f16_sat(st[8 * c + 6], st[8 * c + 7]);
        *reinterpret_cast<uint4 *>(sH + sw128_offset(n, c)) = v;
    }
}

// kGate: y is multiplied by silu(z) (a separate instance, so the ungated kernel keeps its
// registers for the rest of the epilogue).
// kState: the segment pass.  When a sequence is cut into nseg segments of whole blocks (too few
// sequences and heads to fill the GPU), this instance runs first, one CTA per (sequence, segment
// 0 .. nseg - 2, head): x, B, w x, M4 and the state update only, from the initial state for
// segment 0 and from zero for the others.  It writes each segment's end state and, for segments
// 1 .., the product of its blocks' decays.  The full instance then runs one CTA per (sequence,
// segment, head) and starts segment j >= 1 from the state those give at its first token.
template <bool kGate, bool kState>
__global__ void __launch_bounds__(kThreads, 1)
    ssd_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const __grid_constant__ CUtensorMap tmY,
                          const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    launch_dependents();  // the fused kernel after the segment pass may be scheduled
    const int nsg = kState ? p.nseg - 1 : p.nseg;  // segments with a CTA in this launch
    const int slot_r = blockIdx.x / (p.H * nsg);
    const int jh = blockIdx.x - slot_r * p.H * nsg;
    const int j = jh / p.H;  // segment
    const int h = jh - j * p.H;
    const int r = p.seq_order ? p.seq_order[slot_r] : slot_r;
    if (r < 0 || r >= p.S) {
        if (tid == 0 && h == 0 && j == 0) report(p.err, SSD_DEVERR_METADATA);
        return;
    }
    const int g = h / (p.H / p.G);

    // ---- the sequence's chunk range, validated, and this CTA's part of it: blocks [b0, b1) of
    //      the sequence's nb, b0 = j nb / nseg.  Warp 8 works it out, 32 chunks per step.
    const int first = r > 0 ? p.last_chunk[r - 1] + 1 : 0;
    const int last = p.last_chunk[r];
    int *sInfo = reinterpret_cast<int *>(smem + OFF_INFO);
    if (warp == kProducerWarp) {
        bool bad = last >= first && (first < 0 || last >= p.K || p.cu_chunk[first] != p.cu_seqlens[r] ||
                                     p.cu_chunk[last + 1] != p.cu_seqlens[r + 1]);
        int total = 0;
        if (last >= first && !bad) {
            for (int k0 = first; k0 <= last; k0 += 32) {
                const int k = k0 + lane;
                int nb = 0;
                if (k <= last) {
                    const int a = p.cu_chunk[k], b = p.cu_chunk[k + 1];
                    if (a < 0 || b <= a || b > p.T) bad = true;
                    else nb = (b - a + kL - 1) / kL;
                }
                total += __reduce_add_sync(0xffffffffu, nb);
            }
            bad = __any_sync(0xffffffffu, bad);
        }
        const int b0 = (int)((long long)j * total / p.nseg), b1 = (int)((long long)(j + 1) * total / p.nseg);
        int seg_k = first, seg_tb = 0;
        if (!bad && b1 > b0) {
            seg_tb = p.cu_chunk[first];
            int before = 0;  // blocks in the chunks of earlier steps
            for (int k0 = first; b0 > 0 && k0 <= last; k0 += 32) {
                const int k = k0 + lane;
                const int nb = k <= last ? (p.cu_chunk[k + 1] - p.cu_chunk[k] + kL - 1) / kL : 0;
                int incl = nb;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int v = __shfl_up_sync(0xffffffffu, incl, off);
                    if (lane >= off) incl += v;
                }
                const unsigned m = __ballot_sync(0xffffffffu, nb > 0 && before + incl - nb <= b0 && b0 < before + incl);
                if (m) {
                    const int src = __ffs(m) - 1;
                    seg_k = __shfl_sync(0xffffffffu, k, src);
                    seg_tb = p.cu_chunk[seg_k] + (b0 - before - __shfl_sync(0xffffffffu, incl - nb, src)) * kL;
                    break;
                }
                before += __shfl_sync(0xffffffffu, incl, 31);
            }
        }
        if (lane == 0) {
            sInfo[0] = seg_k;
            sInfo[1] = seg_tb;
            sInfo[2] = bad ? 0 : b1 - b0;
            sInfo[3] = bad;
            if (bad && h == 0 && j == 0) report(p.err, SSD_DEVERR_METADATA);
        }
    }
    __syncthreads();
    const int seg_k = sInfo[0], seg_tb = sInfo[1], nblocks = sInfo[2];
    if (sInfo[3]) return;
    if (!kState && nblocks == 0) return;  // no new tokens (or none in this segment)
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) report(p.err, SSD_DEVERR_INTERNAL);
        return;
    }
    uint8_t *sXW = smem + OFF_XW, *sH = smem + OFF_H;
    float *sFCD = reinterpret_cast<float *>(smem + OFF_F);
    float *sE = reinterpret_cast<float *>(smem + OFF_E);
    float *sDec = reinterpret_cast<float *>(smem + OFF_DEC);
    uint32_t *sTM = reinterpret_cast<uint32_t *>(smem + OFF_TM);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);
    auto stage_c = [&](int s) { return smem + s * CB_STAGE; };
    auto stage_b = [&](int s) { return smem + s * CB_STAGE + 32768; };
    auto stage_x = [&](int b) { return smem + OFF_X + (b % kXStages) * X_STAGE; };  // by block index

    if (tid == 0) {
        for (int b = 0; b < NBAR; ++b) {
            const bool four = b == OPS_W || b == PRDY0 || b == PRDY1 || b == OPS_H || b == DS_FREE || b == Y1_FREE ||
                              (b >= EMPTY_X0 && b <= EMPTY_X2);
            mbar_init(&bar[b], four ? 4 : 1);
        }
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sTM, kTmemCols);
        tmem_relinquish();
    }
    if (warp == kProducerWarp && lane == 0) {
        tma_prefetch_desc(&tmX);
        tma_prefetch_desc(&tmB);
        tma_prefetch_desc(&tmC);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *sTM;
    // This kernel is launched as a programmatic dependent of the one before it (the prep kernel,
    // or the segment pass): everything above reads only the call's arguments, and from here on
    // that kernel's results (the fp16 B and C, delta, the cumsum, the segment states) must be
    // complete.
    grid_dependency_wait();

    if (warp == kProducerWarp) {
        // ------------------------------------------------ TMA producer ----
        if (lane != 0) {
            // The idle lanes check, for one head of each sequence, that seq_order names this
            // sequence exactly once (with every entry in range, a permutation then follows): a
            // repeated entry would run one sequence twice and leave another's y unwritten.
            if (!kState && h == 0 && j == 0 && p.seq_order) {
                int cnt = 0;
                for (int i = lane - 1; i < p.S; i += 31) cnt += p.seq_order[i] == r;
                cnt = __reduce_add_sync(0xfffffffeu, cnt);
                if (lane == 1 && cnt != 1) report(p.err, SSD_DEVERR_METADATA);
            }
        } else {
            // Two rings, each refilled as soon as its slot frees: C/B tiles once M3 of the
            // block two back is done, x tiles once y of the block three back is out.
            Cursor ccb, cx;
            ccb.start_at(p.cu_chunk, seg_k, seg_tb, last);
            cx.start_at(p.cu_chunk, seg_k, seg_tb, last);
            int ncb = 0, nx = 0;
            long long t_prog = clock64();
            while (ncb < nblocks || nx < nblocks) {
                bool prog = false;
                if (ncb < nblocks) {
                    const int s = ncb & 1;
                    if (ncb < kCbStages || mbar_test(&bar[EMPTY_CB0 + s], ((ncb >> 1) - 1) & 1)) {
                        uint64_t *full = &bar[FULL_CB0 + s];
                        mbar_arrive_expect_tx(full, kState ? CB_STAGE / 2 : CB_STAGE);  // the segment pass needs no C
                        if (!kState) {
                            tma_load_3d(stage_c(s), &tmC, 0, g, ccb.tb, full);
                            tma_load_3d(stage_c(s) + 16384, &tmC, 64, g, ccb.tb, full);
                        }
                        tma_load_3d(stage_b(s), &tmB, 0, g, ccb.tb, full);
                        tma_load_3d(stage_b(s) + 16384, &tmB, 64, g, ccb.tb, full);
                        ccb.next();
                        ++ncb;
                        prog = true;
                    }
                }
                if (nx < nblocks) {
                    if (nx < kXStages || mbar_test(&bar[EMPTY_X0 + nx % kXStages], (nx / kXStages - 1) & 1)) {
                        uint64_t *full = &bar[FULL_X0 + nx % kXStages];
                        mbar_arrive_expect_tx(full, X_STAGE);
                        tma_load_3d(stage_x(nx), &tmX, 0, h, cx.tb, full);
                        cx.next();
                        ++nx;
                        prog = true;
                    }
                }
                if (prog) {
                    t_prog = clock64();
                } else if (clock64() - t_prog > p.wait_limit) {
                    report(p.err, SSD_DEVERR_TIMEOUT);
                    break;
                } else if (ncb < nblocks) {
                    // nothing to issue: the hardware suspends this thread until the next C/B stage
                    // frees, or a short while passes so the x ring is looked at again
                    mbar_try_wait_sleep(&bar[EMPTY_CB0 + (ncb & 1)], ((ncb >> 1) - 1) & 1, 300);
                } else {
                    mbar_try_wait_sleep(&bar[EMPTY_X0 + nx % kXStages], (nx / kXStages - 1) & 1, 300);
                }
            }
            // drain: no copy may still be landing when the CTA exits
            for (int i = max(ncb - kCbStages, 0); i < ncb; ++i) mbar_wait(&bar[FULL_CB0 + (i & 1)], (i >> 1) & 1);
            for (int i = max(nx - kXStages, 0); i < nx; ++i) mbar_wait(&bar[FULL_X0 + i % kXStages], (i / kXStages) & 1);
        }
    } else if (warp == kMmaWarp) {
        // ------------------------------------------------ MMA issue -------
        if (lane == 0) {
            int nblocks_mma = nblocks;
            constexpr uint32_t kIdS = idesc_f16(128, 128, 0, 0);
            constexpr uint32_t kIdY = idesc_f16(128, 64, 0, 1);
            constexpr uint32_t kIdD = idesc_f16(128, 64, 1, 1);
            // Tile descriptors, built once: a K slice is desc_at(tile, its byte offset), so the
            // issue of each MMA waits on nothing but the previous one.
            const uint64_t dC0 = sw128_desc(smem_u32(stage_c(0)), 16, 1024), dC1 = sw128_desc(smem_u32(stage_c(1)), 16, 1024);
            const uint64_t dBk0 = sw128_desc(smem_u32(stage_b(0)), 16, 1024), dBk1 = sw128_desc(smem_u32(stage_b(1)), 16, 1024);
            const uint64_t dBm0 = sw128_desc(smem_u32(stage_b(0)), 16384, 1024);
            const uint64_t dBm1 = sw128_desc(smem_u32(stage_b(1)), 16384, 1024);
            const uint64_t dX0 = sw128_desc(smem_u32(stage_x(0)), 1024, 1024), dX1 = sw128_desc(smem_u32(stage_x(1)), 1024, 1024),
                           dX2 = sw128_desc(smem_u32(stage_x(2)), 1024, 1024);
            const uint64_t dH = sw128_desc(smem_u32(sH), 1024, 1024), dXW = sw128_desc(smem_u32(sXW), 1024, 1024);
            auto issue_m1 = [&](int b) {
                const int sb = b & 1;
                const uint64_t da = sb ? dC1 : dC0, db = sb ? dBk1 : dBk0;
                const uint32_t dS = tm + (sb ? COL_S1 : COL_S0);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_ss(dS, desc_at(da, ko), desc_at(db, ko), kIdS, k > 0);
                }
                mma_commit(&bar[S_RDY0 + sb]);
            };
            bool ok = true;
            if (kState) {
                // the segment pass: M4 only, per block
                for (int i = 0; ok && i < nblocks; ++i) {
                    const int s = i & 1;
                    if (!(ok = mbar_wait(&bar[OPS_W], i & 1, p.wait_limit)) || !(ok = mbar_wait(&bar[DS_FREE], i & 1, p.wait_limit)) ||
                        !(ok = mbar_wait(&bar[FULL_CB0 + s], (i >> 1) & 1, p.wait_limit)))
                        break;
                    tc_fence_after();
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mma_ss(tm + COL_DS, desc_at(s ? dBm1 : dBm0, 2048 * k), desc_at(dXW, 2048 * k), kIdD, k > 0);
                    mma_commit(&bar[ACC_DS]);
                    mma_commit(&bar[EMPTY_CB0 + s]);
                }
                nblocks_mma = 0;  // the loop below is the full pass
            } else if ((ok = mbar_wait(&bar[FULL_CB0], 0, p.wait_limit))) {
                tc_fence_after();
                issue_m1(0);
            }
            // Per block, in this order: M4 (the state update waits on it), M3, M2 (y), then M1 of
            // the next block, whose S is needed only after the next block's scan and w x.
            for (int i = 0; ok && i < nblocks_mma; ++i) {
                const int s = i & 1, xs = i % kXStages;
                const uint64_t dCs = s ? dC1 : dC0, dBms = s ? dBm1 : dBm0;
                const uint64_t dXs = xs == 0 ? dX0 : (xs == 1 ? dX1 : dX2);
                // M4: dS = B^T (w x) once w x exists and dS of the previous block was read
                if (!(ok = mbar_wait(&bar[OPS_W], i & 1, p.wait_limit)) || !(ok = mbar_wait(&bar[DS_FREE], i & 1, p.wait_limit))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ss(tm + COL_DS, desc_at(dBms, 2048 * k), desc_at(dXW, 2048 * k), kIdD, k > 0);
                mma_commit(&bar[ACC_DS]);
                // M3: Y2 = C Hprev^T once the state entering the block exists
                if (!(ok = mbar_wait(&bar[OPS_H], i & 1, p.wait_limit))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_ss(tm + COL_Y2 + 64 * s, desc_at(dCs, ko), desc_at(dH, 2048 * k), kIdY, k > 0);
                }
                mma_commit(&bar[H_FREE]);
                mma_commit(&bar[EMPTY_CB0 + s]);  // M1, M4 and M3 of the block have read its C/B stage
                // M2: Y1 = P X once P is ready and Y1 of the previous block was read
                if (!(ok = mbar_wait(&bar[PRDY0 + s], (i >> 1) & 1, p.wait_limit)) || !(ok = mbar_wait(&bar[Y1_FREE], i & 1, p.wait_limit))) break;
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ts(tm + COL_Y1, tm + (s ? COL_S1 : COL_S0) + 8 * k, desc_at(dXs, 2048 * k), kIdY, k > 0);
                mma_commit(&bar[ACC_Y]);
                if (i + 1 < nblocks_mma) {
                    if (!(ok = mbar_wait(&bar[FULL_CB0 + ((i + 1) & 1)], ((i + 1) >> 1) & 1, p.wait_limit))) break;
                    tc_fence_after();
                    issue_m1(i + 1);
                }
            }
            if (!ok) report(p.err, SSD_DEVERR_TIMEOUT);
            mma_commit(&bar[DRAIN]);  // one more commit covers every MMA issued
            mbar_wait(&bar[DRAIN], 0);
        }
    } else if (warp < 4) {
        // ------------------------------------ producer warpgroup (P) -------
        const int q = warp;
        const int t = q * 32 + lane;
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const float Dh = p.D ? p.D[h] : 0.f;
        const float *cum = p.cum + (size_t)h * p.T, *dl = p.delta + (size_t)h * p.T;
        Cursor cur;
        cur.start_at(p.cu_chunk, seg_k, seg_tb, last);
        // Row t's delta and cumsum, and the cumsum at the end of each 32-row group (clamped to the
        // block's last row), loaded one block ahead.  Rows past the block's end take delta 0 and
        // the cumsum of the last row.
        RowVals nxt;
        nxt.load(cum, dl, cur.tb, cur.len(), t);
        for (int i = 0; i < nblocks; ++i, cur.next()) {
            const int s = i & 1;
            const uint32_t ph = (i >> 1) & 1;
            const int L = cur.len();
            uint8_t *sXs = stage_x(i);
            const uint32_t colS = s ? COL_S1 : COL_S0;
            const RowVals rv = nxt;
            if (i + 1 < nblocks) {
                Cursor cn = cur;
                cn.next();
                nxt.load(cum, dl, cn.tb, cn.len(), t);
            }
            const float c = rv.c, delta = rv.d, c_last = rv.g[3];
            if constexpr (!kState) {
                float *sF = sFCD + (i & 1) * 512, *sCc = sF + 128, *sDl = sF + 256, *sF2 = sF + 384;
                sF[t] = __expf(rv.g[q] - c) * delta;  // column factor of column t (relative to its group's end)
                sCc[t] = c;
                sDl[t] = delta;
                // column factor of column t relative to its group's first row (the diagonal group)
                sF2[t] = __expf(__shfl_sync(0xffffffffu, c, 0) - c) * delta;
                sE[(i % kRing) * 128 + t] = __expf(c);  // carried-state factor of row t (consumer)
            }
            if (t == 0) sDec[i % kRing] = __expf(c_last);
            // w_t as fp16x2, for w x computed as an fp16 product of the (exactly) converted x
            const uint32_t w2 = pack_f16_sat(__expf(c_last - c) * delta, __expf(c_last - c) * delta);

            // ---- w x (fp16) into the M4 operand once M4 of the previous block is done; x -> fp16
            bool ok = warp_wait(&bar[FULL_X0 + i % kXStages], (i / kXStages) & 1, p.wait_limit);
            if (ok && i > 0) ok = warp_wait(&bar[ACC_DS], (i - 1) & 1, p.wait_limit);
            if (!named_bar_and(BAR_PG, 128, ok)) {
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            // Rows t >= L hold the next sequence's tokens (the TMA box is always 128 rows): they are
            // replaced by zeros, not scaled by w = 0, so a non-finite value there cannot reach this
            // sequence's products (0 * inf is NaN).
            const bool live = t < L;
#pragma unroll
            for (int cc = 0; cc < 8; ++cc) {
                const uint4 xh = bf16x8_to_f16x8(*reinterpret_cast<const uint4 *>(sXs + sw128_offset(t, cc)));
                const uint4 xw = make_uint4(hmul2_u32(xh.x, w2), hmul2_u32(xh.y, w2), hmul2_u32(xh.z, w2),
                                            hmul2_u32(xh.w, w2));
                *reinterpret_cast<uint4 *>(sXW + sw128_offset(t, cc)) = xw;
                if (!kState) *reinterpret_cast<uint4 *>(sXs + sw128_offset(t, cc)) = xh;
            }
            if (!live) {  // only in a sequence's last, short block: these rows become zeros
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    *reinterpret_cast<uint4 *>(sXW + sw128_offset(t, cc)) = make_uint4(0u, 0u, 0u, 0u);
                    if (!kState) *reinterpret_cast<uint4 *>(sXs + sw128_offset(t, cc)) = make_uint4(0u, 0u, 0u, 0u);
                }
            }
            if constexpr (kState) {
                // the segment pass: B's rows past a short block's end are cleared for M4 (no M1 reads
                // the stage here); the x slot is free once w x is written
                if (L < kL && !live) {
                    uint8_t *sB = stage_b(s);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        *reinterpret_cast<uint4 *>(sB + sw128_offset(t, cc)) = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(sB + 16384 + sw128_offset(t, cc)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bar[OPS_W]);
                    mbar_arrive(&bar[EMPTY_X0 + i % kXStages]);
                }
                continue;
            }
            bool s_ready = false;
            if (L < kL) {
                // A short block: M4 sums B rows against w x over all 128 rows, so B's rows past the
                // block end are cleared too, once M1 (the other reader of the stage) is done with them.
                ok = warp_wait(&bar[S_RDY0 + s], ph, p.wait_limit);
                if (!named_bar_and(BAR_PG, 128, ok)) {
                    if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                    break;
                }
                s_ready = true;
                if (!live) {
                    uint8_t *sB = stage_b(s);
#pragma unroll
                    for (int cc = 0; cc < 8; ++cc) {
                        *reinterpret_cast<uint4 *>(sB + sw128_offset(t, cc)) = make_uint4(0u, 0u, 0u, 0u);
                        *reinterpret_cast<uint4 *>(sB + 16384 + sw128_offset(t, cc)) = make_uint4(0u, 0u, 0u, 0u);
                    }
                }
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[OPS_W]);

            // ---- S ready: P pass, S (fp32) -> P (fp16) over the same columns
            if (!s_ready) {
                ok = warp_wait(&bar[S_RDY0 + s], ph, p.wait_limit);
                if (!named_bar_and(BAR_PG, 128, ok)) {
                    if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                    break;
                }
            }
            tc_fence_after();
            // Group j of P goes over columns [16j, 16j+16), which hold S groups <= j that this
            // warp has already read.  The loops stay rolled: the four warp roles run different
            // code, and unrolled copies of these bodies overflow the instruction cache.
#pragma unroll 1
            for (int j = 0; j < q; ++j) {  // groups below the diagonal
                uint32_t v[32], pk[16];
                tmem_ld32(tm + lane_base + colS + 32 * j, v);
                const float R = __expf(c - (j == 0 ? rv.g[0] : (j == 1 ? rv.g[1] : rv.g[2])));
                const float4 *f4 = reinterpret_cast<const float4 *>(sFCD + (i & 1) * 512 + 32 * j);
                tmem_ld_wait();
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 f = f4[u];
                    const float2 a = mul_f2(mul_f2(make_float2(__uint_as_float(v[4 * u]), __uint_as_float(v[4 * u + 1])),
                                                   make_float2(f.x, f.y)), make_float2(R, R));
                    const float2 b = mul_f2(mul_f2(make_float2(__uint_as_float(v[4 * u + 2]), __uint_as_float(v[4 * u + 3])),
                                                   make_float2(f.z, f.w)), make_float2(R, R));
                    pk[2 * u] = pack_f16_sat(a.x, a.y);
                    pk[2 * u + 1] = pack_f16_sat(b.x, b.y);
                }
                tmem_st16(tm + lane_base + colS + 16 * j, pk);
            }
            {  // the diagonal group j = q, the mask by select
                // exp(c_t - c_s) = exp(c_t - c_b) exp(c_b - c_s), b the group's first row: both factors
                // stay normal fp32 numbers while the group's total decay c_b - c_e is at most 80;
                // beyond that, one exponential per element.  The same for the whole warp.
                const float cb = __shfl_sync(0xffffffffu, c, 0);
                if (cb - rv.g[q] <= 80.f) {
                    uint32_t v[32], pk[16];
                    tmem_ld32(tm + lane_base + colS + 32 * q, v);
                    const float R2 = __expf(c - cb);
                    const float4 *f4 = reinterpret_cast<const float4 *>(sFCD + (i & 1) * 512 + 384 + 32 * q);
                    tmem_ld_wait();
#pragma unroll
                    for (int u4 = 0; u4 < 8; ++u4) {
                        const float4 f = f4[u4];
                        // at most |S| delta for u <= lane
                        const float2 a = mul_f2(mul_f2(make_float2(__uint_as_float(v[4 * u4]), __uint_as_float(v[4 * u4 + 1])),
                                                       make_float2(R2, R2)), make_float2(f.x, f.y));
                        const float2 b = mul_f2(mul_f2(make_float2(__uint_as_float(v[4 * u4 + 2]), __uint_as_float(v[4 * u4 + 3])),
                                                       make_float2(R2, R2)), make_float2(f.z, f.w));
                        const float vals[4] = {a.x, a.y, b.x, b.y};
                        float pv[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int u = 4 * u4 + e;
                            const float val = vals[e];
                            pv[e] = (u < lane) ? val : ((u == lane) ? val + Dh : 0.f);
                        }
                        pk[2 * u4] = pack_f16_sat(pv[0], pv[1]);
                        pk[2 * u4 + 1] = pack_f16_sat(pv[2], pv[3]);
                    }
                    tmem_st16(tm + lane_base + colS + 16 * q, pk);
                } else {
                    diag_group_per_element(tm + lane_base + colS + 32 * q, tm + lane_base + colS + 16 * q,
                                           sFCD + (i & 1) * 512 + 128 + 32 * q, sFCD + (i & 1) * 512 + 256 + 32 * q,
                                           c, Dh, lane);
                }
            }
            {
                uint32_t zero[16];
#pragma unroll
                for (int u = 0; u < 16; ++u) zero[u] = 0u;
#pragma unroll 1
                for (int j = q + 1; j < 4; ++j) tmem_st16(tm + lane_base + colS + 16 * j, zero);  // above the diagonal
            }
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[PRDY0 + s]);
        }
    } else {
        // ------------------------------------ consumer warpgroup (E) -------
        const int q = warp - 4;
        const int t = q * 32 + lane;  // TMEM lane: token row t of Y, dstate row t of dS and the state
        const uint32_t lane_base = (uint32_t)(q * 32) << 16;
        const size_t HPN = (size_t)p.H * kP * kN;
        float st[kP];  // state h[p][n = t]
        // segment outputs of this sequence and head: [segment][P][N] with a stride of H P N
        const size_t seg0 = ((size_t)r * (p.nseg - 1) * p.H + h) * kP * kN + t;
        if (j == 0) {  // the sequence's initial state
            const int32_t is = p.init_slot ? p.init_slot[r] : p.null_id;
            if (slot_usable(is, p.null_id, p.num_slots, (t == 0) ? p.err : nullptr)) {
                const float *src = p.cache + (size_t)is * HPN + (size_t)h * kP * kN + t;
#pragma unroll
                for (int e = 0; e < kP; ++e) st[e] = src[(size_t)e * kN];
            } else {
#pragma unroll
                for (int e = 0; e < kP; ++e) st[e] = 0.f;
            }
        } else if (kState) {  // later segments of the segment pass start from zero
#pragma unroll
            for (int e = 0; e < kP; ++e) st[e] = 0.f;
        } else {  // the state at this segment's first token: segment 0's end, carried through 1 .. j-1
#pragma unroll
            for (int e = 0; e < kP; ++e) st[e] = p.seg_state[seg0 + (size_t)e * kN];
            for (int jj = 1; jj < j; ++jj) {
                const float d = p.seg_decay[((size_t)r * (p.nseg - 1) + jj) * p.H + h];
                const float *src = p.seg_state + seg0 + (size_t)jj * HPN;
#pragma unroll
                for (int e = 0; e < kP; ++e) st[e] = fmaf(d, st[e], src[(size_t)e * kN]);
            }
        }
        if constexpr (kState) {
            // the segment pass: the state through the segment's blocks, then its end state and
            // the product of its decays
            if (lane == 0) mbar_arrive(&bar[DS_FREE]);
            float dprod = 1.f;
            for (int i = 0; i < nblocks; ++i) {
                bool ok = warp_wait(&bar[ACC_DS], i & 1, p.wait_limit);
                if (!named_bar_and(BAR_CG, 128, ok)) {
                    if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
                const float decay = sDec[i % kRing];
                uint32_t d[64];
                tmem_ld64(tm + lane_base + COL_DS, d);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 u = fma_f2(make_float2(decay, decay), make_float2(st[e], st[e + 1]),
                                            make_float2(__uint_as_float(d[e]), __uint_as_float(d[e + 1])));
                    st[e] = u.x;
                    st[e + 1] = u.y;
                }
                dprod *= decay;
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[DS_FREE]);
            }
            float *dst = p.seg_state + seg0 + (size_t)j * HPN;
#pragma unroll
            for (int e = 0; e < kP; ++e) dst[(size_t)e * kN] = st[e];
            if (t == 0) p.seg_decay[((size_t)r * (p.nseg - 1) + j) * p.H + h] = dprod;
        } else {
        store_state_row(sH, t, st);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&bar[OPS_H]);    // the state entering block 0
            mbar_arrive(&bar[DS_FREE]);  // dS and Y1 start out free
            mbar_arrive(&bar[Y1_FREE]);
        }
        Cursor cur;
        cur.start_at(p.cu_chunk, seg_k, seg_tb, last);
        // cache slot of the current chunk's end state, loaded a chunk ahead of its use
        int32_t cs = p.chunk_slot ? p.chunk_slot[seg_k] : p.null_id;
        for (int i = 0; i < nblocks; ++i, cur.next()) {
            const int s = i & 1;
            const int tb = cur.tb, L = cur.len();
            // ---- dS: the state after this block, then the fp16 state for the next block's M3
            bool ok = warp_wait(&bar[ACC_DS], i & 1, p.wait_limit);
            if (!named_bar_and(BAR_CG, 128, ok)) {
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            const float decay = sDec[i % kRing];
            const float e_row = sE[(i % kRing) * 128 + t];
            {
                uint32_t d[64];
                tmem_ld64(tm + lane_base + COL_DS, d);
                tmem_ld_wait();
#pragma unroll
                for (int e = 0; e < 64; e += 2) {
                    const float2 u = fma_f2(make_float2(decay, decay), make_float2(st[e], st[e + 1]),
                                            make_float2(__uint_as_float(d[e]), __uint_as_float(d[e + 1])));
                    st[e] = u.x;
                    st[e + 1] = u.y;
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[DS_FREE]);  // M4 of the next block may overwrite dS
            ok = warp_wait(&bar[H_FREE], i & 1, p.wait_limit);         // M3 of this block has read the state tile
            if (!named_bar_and(BAR_CG, 128, ok)) {
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            store_state_row(sH, t, st);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[OPS_H]);  // the state entering the next block
            if (cur.ends_chunk()) {
                if (slot_usable(cs, p.null_id, p.num_slots, (t == 0) ? p.err : nullptr)) {
                    float *dst = p.cache + (size_t)cs * HPN + (size_t)h * kP * kN + t;
#pragma unroll
                    for (int e = 0; e < kP; ++e) dst[(size_t)e * kN] = st[e];
                }
                if (p.chunk_slot) cs = p.chunk_slot[min(cur.k + 1, last)];
            }
            // ---- y = Y1 + exp(c_t) Y2
            ok = warp_wait(&bar[ACC_Y], i & 1, p.wait_limit);
            if (!named_bar_and(BAR_CG, 128, ok)) {
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            uint8_t *sY = stage_x(i);  // y staging: the block's x slot, which M2 has finished with
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
                uint32_t y1[32], y2[32];
                tmem_ld32(tm + lane_base + COL_Y1 + 32 * half, y1);
                tmem_ld32(tm + lane_base + COL_Y2 + 64 * s + 32 * half, y2);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    float yv[8];
#pragma unroll
                    for (int u = 0; u < 8; u += 2) {
                        const float2 o = fma_f2(make_float2(e_row, e_row),
                                                make_float2(__uint_as_float(y2[8 * cc + u]), __uint_as_float(y2[8 * cc + u + 1])),
                                                make_float2(__uint_as_float(y1[8 * cc + u]), __uint_as_float(y1[8 * cc + u + 1])));
                        yv[u] = o.x;
                        yv[u + 1] = o.y;
                    }
                    if (kGate) {  // output gate y * silu(z); rows past the block end read a clamped
                                  // token (no lane-dependent branch between tcgen05 loads) and are
                                  // never stored
                        const size_t zrow = (size_t)min(tb + t, p.T - 1);
                        const uint4 zz =
                            *reinterpret_cast<const uint4 *>(p.z + (zrow * p.H + h) * kP + 32 * half + 8 * cc);
                        const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            yv[2 * u] = silu_gate(yv[2 * u], __uint_as_float(zw[u] << 16));
                            yv[2 * u + 1] = silu_gate(yv[2 * u + 1], __uint_as_float(zw[u] & 0xFFFF0000u));
                        }
                    }
                    const uint4 v = make_uint4(pack_bf16(yv[0], yv[1]), pack_bf16(yv[2], yv[3]),
                                               pack_bf16(yv[4], yv[5]), pack_bf16(yv[6], yv[7]));
                    *reinterpret_cast<uint4 *>(sY + sw128_offset(t, 4 * half + cc)) = v;
                }
            }
            tc_fence_before();
            fence_proxy_async_smem();  // the staged rows are visible to the tensor-copy engine
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[Y1_FREE]);  // M2 of the next block may overwrite Y1
            named_bar_sync(BAR_CG, 128);  // y tile staged
            if (L == kL) {
                // a whole block: one tensor copy of the tile; its issuer waits until the copy has
                // read the slot before the slot is given back to the x ring
                if (t == 0) {
                    tma_store_3d(&tmY, sY, 0, h, tb);
                    bulk_commit();
                    bulk_wait_read();
                }
                __syncwarp();
            } else {
                // a short block: rows past its end belong to the next sequence and are not written
#pragma unroll
                for (int rr = 0; rr < 8; ++rr) {
                    const int row = rr * 16 + (t >> 3), cc = t & 7;
                    if (row < L) {
                        const uint4 v = *reinterpret_cast<const uint4 *>(sY + sw128_offset(row, cc));
                        *reinterpret_cast<uint4 *>(p.y + ((size_t)(tb + row) * p.H + h) * kP + 8 * cc) = v;
                    }
                }
                fence_proxy_async_smem();  // this warp's reads of the slot come before the next TMA write
                __syncwarp();
            }
            if (lane == 0) mbar_arrive(&bar[EMPTY_X0 + i % kXStages]);
        }
        }
    }
    if (warp == 4 && lane == 0) bulk_wait();  // the y tile copies this thread issued are complete
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

// Per call, before the fused kernel:
//  - B and C (bf16) -> fp16: every head of a group reads the same tiles, so converting them once
//    here instead of in each head's CTA saves that work (and its shared-memory traffic) H/G times.
//  - delta = clamp(softplus(dt + dt_bias)) and the cumsum of delta * A within each block of the
//    fused kernel (the 128-token pieces of every chunk, starting at the chunk's first token), for
//    every head, into [H, T] arrays.
// The scan CTAs come first, one per (chunk, piece, 32 heads): piece m of chunk k is the block
// starting at token cu_chunk[k] + 128 m (pieces m + mpc, m + 2 mpc, ... too, for a chunk longer
// than mpc pieces).  Its four warps take 32 tokens each, lane = head (so the dt loads of a warp
// are 64-byte row segments); each scans its 32 tokens on its own, and a warp adds the totals of
// the warps before it.  The conversion CTAs follow, grid-stride.
struct PrepParams {
    int T, H, K;
    int mpc;       // pieces per chunk with a CTA of their own (chunk_size / 128, at least 1)
    int nscan;     // scan CTAs, K * mpc * ceil(H / 32); the rest convert B and C
    size_t row16;  // 16-byte units per token row of B (and C)
    const uint4 *B, *C;
    uint4 *Bh, *Ch;
    const __nv_bfloat16 *dt;
    const float *A, *dt_bias;
    int dt_softplus;
    float dt_min, dt_max;
    const int32_t *cu_chunk;
    float *cum, *delta;
};

constexpr int kPrepThreads = 128;  // 4 warps

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const PrepParams p) {
    __shared__ float sC[32][129], sD[32][129];  // one block's outputs: 32 heads x 128 tokens (padded)
    __shared__ float sTail[4][32];              // per warp and head: the sum over its 32 tokens
    launch_dependents();  // the call's next kernel may set itself up meanwhile
    // The scan CTAs (the first nscan) compute their piece first.  When there are enough of them
    // (large calls), every CTA then converts its grid-stride share of B and C, so the conversion's
    // bandwidth-bound work runs beside the scan's latency-bound CTAs throughout the grid; small
    // calls get conversion CTAs of their own after the scan CTAs.
    if ((int)blockIdx.x < p.nscan) {
        const int nhb = (p.H + 31) / 32;
        const int hb = blockIdx.x % nhb;
        const int km = blockIdx.x / nhb;
        const int k = km / p.mpc, m0 = km - k * p.mpc;
        const int cs = p.cu_chunk[k], ce = p.cu_chunk[k + 1];
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int h = hb * 32 + lane;
        const bool hv = h < p.H;
        const float Ah = hv ? p.A[h] : 0.f;
        const float bias = (hv && p.dt_bias) ? p.dt_bias[h] : 0.f;
        const __nv_bfloat16 *dth = p.dt + (hv ? h : 0);
        for (int tb = cs + 128 * m0; tb < ce; tb += 128 * p.mpc) {
            const int L = min(128, ce - tb);
            const int ta = tb + 32 * warp;
            const int mw = max(0, min(32, tb + L - ta));  // this warp's tokens
            float dv[32];
    #pragma unroll
            for (int j = 0; j < 32; ++j) dv[j] = j < mw ? __bfloat162float(dth[(size_t)(ta + j) * p.H]) : 0.f;
            float run = 0.f;  // the cumsum within this warp's 32 tokens
    #pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (j < mw) {
                    const float d = fast_delta(dv[j] + bias, p.dt_softplus, p.dt_min, p.dt_max);
                    run = fmaf(d, Ah, run);
                    sC[lane][32 * warp + j] = run;
                    sD[lane][32 * warp + j] = d;
                }
            }
            sTail[warp][lane] = run;
            __syncthreads();
            // coalesced stores: warp w writes heads w, w + 4, ...; a token adds the totals of the
            // 32-token quarters before its own
            for (int hh = warp; hh < 32; hh += 4) {
                const int h2 = hb * 32 + hh;
                if (h2 >= p.H) break;
                float carry = 0.f;
                for (int u0 = 0; u0 < L; u0 += 32) {
                    const int u = u0 + lane;
                    if (u < L) {
                        const size_t o = (size_t)h2 * p.T + tb + u;
                        p.cum[o] = sC[hh][u] + carry;
                        p.delta[o] = sD[hh][u];
                    }
                    carry += sTail[u0 >> 5][hh];
                }
            }
            __syncthreads();  // the staging arrays are reused by the next piece
        }
    }
    // B and C -> fp16, grid-stride over 16-byte units, four of each in flight per thread
    const int c0 = (int)gridDim.x > p.nscan ? p.nscan : 0;  // the first converting CTA
    if ((int)blockIdx.x >= c0) {
        const size_t cnt = (size_t)p.T * p.row16;
        const size_t stride = (size_t)(gridDim.x - c0) * kPrepThreads;
        size_t i = (size_t)(blockIdx.x - c0) * kPrepThreads + threadIdx.x;
        for (; i + 3 * stride < cnt; i += 4 * stride) {
            uint4 b[4], c[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                b[u] = p.B[i + u * stride];
                c[u] = p.C[i + u * stride];
            }
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                p.Bh[i + u * stride] = bf16x8_to_f16x8(b[u]);
                p.Ch[i + u * stride] = bf16x8_to_f16x8(c[u]);
            }
        }
        for (; i < cnt; i += stride) {
            p.Bh[i] = bf16x8_to_f16x8(p.B[i]);
            p.Ch[i] = bf16x8_to_f16x8(p.C[i]);
        }
    }
}

}  // namespace

static size_t up256(size_t n) { return (n + 255) & ~(size_t)255; }

// Segments per sequence.  One CTA per (sequence, head) fills the GPU when there are at least
// half as many of them as SMs; below that each sequence is cut into k segments of whole blocks
// (k CTAs per (sequence, head), at most 8, and on average at least two blocks each), at the
// price of the segment pass.  0 SMs (no device) means no split.
static int sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

int tc_prefill_segments(const ssd_prefill_args &a) {
    const long long sh = (long long)a.num_seqs * a.nheads;
    const int sms = sm_count();
    if (sh <= 0 || 2 * sh > sms) return 1;
    long long k = sms / sh;
    const long long avg_blocks = (long long)a.total_tokens / a.num_seqs / kL;
    k = std::min(k, std::max(1ll, avg_blocks / 2));
    return (int)std::min(k, 8ll);
}

size_t tc_prefill_workspace(const ssd_prefill_args &a) {
    const size_t bc = (size_t)a.total_tokens * a.ngroups * kN * 2;
    const size_t ht = (size_t)a.total_tokens * a.nheads * 4;
    const int k = tc_prefill_segments(a);
    const size_t sg = (size_t)a.num_seqs * (k - 1) * a.nheads;
    return 2 * up256(bc) + 2 * up256(ht) + (k > 1 ? up256(sg * kP * kN * 4) + up256(sg * 4) : 0);
}

bool tc_prefill_supported(const ssd_prefill_args &a) {
    return a.dtype == SSD_BF16 && a.headdim == kP && a.dstate == kN && a.total_tokens > 0;
}

// A launch of the fused kernel (or the segment pass) that may begin while the kernel before it on
// the stream is finishing: its CTAs set up shared memory and TMEM as SMs free up, then wait in
// grid_dependency_wait() for that kernel's results.
using TcKernel = void (*)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap, const TcParams);
cudaError_t launch_tc(TcKernel k, unsigned grid, bool programmatic, cudaStream_t s, const CUtensorMap &mX,
                      const CUtensorMap &mB, const CUtensorMap &mC, const CUtensorMap &mY, const TcParams &p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = programmatic ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, k, mX, mB, mC, mY, p);
}

cudaError_t tc_prefill_launch(const ssd_prefill_args &a, void *workspace, cudaStream_t s, cudaEvent_t after_prep,
                              cudaEvent_t before_fused) {
    CUtensorMap mX, mB, mC, mY;
    const uint64_t T = (uint64_t)a.total_tokens;
    const size_t bc = (size_t)a.total_tokens * a.ngroups * kN * 2;
    const size_t ht = (size_t)a.total_tokens * a.nheads * 4;
    uint8_t *Bh = static_cast<uint8_t *>(workspace);
    uint8_t *Ch = Bh + up256(bc);
    float *cum = reinterpret_cast<float *>(Ch + up256(bc));
    float *delta = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(cum) + up256(ht));
    {
        PrepParams q;
        q.T = a.total_tokens;
        q.H = a.nheads;
        q.K = a.num_chunks;
        q.row16 = (size_t)a.ngroups * kN * 2 / 16;  // kN * 2 bytes per group row: a multiple of 16
        q.B = static_cast<const uint4 *>(a.B);
        q.C = static_cast<const uint4 *>(a.C);
        q.Bh = reinterpret_cast<uint4 *>(Bh);
        q.Ch = reinterpret_cast<uint4 *>(Ch);
        q.dt = static_cast<const __nv_bfloat16 *>(a.dt);
        q.A = a.A;
        q.dt_bias = a.dt_bias;
        q.dt_softplus = a.dt_softplus;
        q.dt_min = a.dt_min;
        q.dt_max = a.dt_max;
        q.cu_chunk = a.cu_chunk_seqlens;
        q.cum = cum;
        q.delta = delta;
        q.mpc = std::max(1, std::min((a.chunk_size + kL - 1) / kL, 64));
        q.nscan = a.num_chunks * q.mpc * ((a.nheads + 31) / 32);
        const int sms = std::max(sm_count(), 1);
        const size_t conv = std::min<size_t>(((size_t)a.total_tokens * q.row16 + 4 * kPrepThreads - 1) / (4 * kPrepThreads),
                                             (size_t)sms * 8);
        // large calls: the scan CTAs also do the conversion; small ones: conversion CTAs of their own
        const size_t grid = (size_t)q.nscan >= conv ? (size_t)q.nscan : q.nscan + std::max<size_t>(conv, 1);
        prep_kernel<<<(unsigned)std::max<size_t>(grid, 1), kPrepThreads, 0, s>>>(q);
        cudaError_t e = cudaGetLastError();
        if (e == cudaSuccess && after_prep) e = cudaEventRecord(after_prep, s);
        if (e != cudaSuccess) return e;
    }
    if (!make_tmap_bf16_3d(&mX, a.x, kP, a.nheads, T, (uint64_t)kP * 2, (uint64_t)a.nheads * kP * 2, 64, 1, kL) ||
        !make_tmap_f16_3d(&mB, Bh, kN, a.ngroups, T, (uint64_t)kN * 2, (uint64_t)a.ngroups * kN * 2, 64, 1, kL) ||
        !make_tmap_f16_3d(&mC, Ch, kN, a.ngroups, T, (uint64_t)kN * 2, (uint64_t)a.ngroups * kN * 2, 64, 1, kL) ||
        !make_tmap_bf16_3d(&mY, a.y, kP, a.nheads, T, (uint64_t)kP * 2, (uint64_t)a.nheads * kP * 2, 64, 1, kL))
        return cudaErrorInvalidValue;
    TcParams p;
    p.T = a.total_tokens;
    p.S = a.num_seqs;
    p.K = a.num_chunks;
    p.H = a.nheads;
    p.G = a.ngroups;
    p.dt_softplus = a.dt_softplus;
    p.dt_min = a.dt_min;
    p.dt_max = a.dt_max;
    p.num_slots = a.num_slots;
    p.null_id = a.null_block_id;
    p.dt = static_cast<const __nv_bfloat16 *>(a.dt);
    p.A = a.A;
    p.D = a.D;
    p.dt_bias = a.dt_bias;
    p.cu_seqlens = a.cu_seqlens;
    p.cu_chunk = a.cu_chunk_seqlens;
    p.last_chunk = a.last_chunk_indices;
    p.init_slot = a.init_slot;
    p.chunk_slot = a.chunk_slot;
    p.cache = a.state_cache;
    p.z = static_cast<const __nv_bfloat16 *>(a.z);
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    p.err = a.err_word;
    p.seq_order = a.seq_order;
    p.wait_limit = a.wait_limit_cycles > 0 ? (long long)a.wait_limit_cycles : 2000000000ll;
    p.cum = cum;
    p.delta = delta;
    p.nseg = tc_prefill_segments(a);
    p.seg_state = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(delta) + up256(ht));
    p.seg_decay = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(p.seg_state) +
                                            up256((size_t)a.num_seqs * (p.nseg - 1) * a.nheads * kP * kN * 4));
    const long long grid = (long long)a.num_seqs * a.nheads;
    if (grid <= 0) return cudaSuccess;
    cudaError_t e;
    if (p.nseg > 1) {
        auto seg_kernel = ssd_prefill_tc_kernel<false, true>;
        e = cudaFuncSetAttribute(seg_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
        if (e != cudaSuccess) return e;
        // programmatic unless an event was recorded after the prep kernel (the mixed step's)
        e = launch_tc(seg_kernel, (unsigned)(grid * (p.nseg - 1)), !after_prep, s, mX, mB, mC, mY, p);
        if (e != cudaSuccess) return e;
    }
    auto kernel = p.z ? ssd_prefill_tc_kernel<true, false> : ssd_prefill_tc_kernel<false, false>;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    if (before_fused) {
        e = cudaEventRecord(before_fused, s);
        if (e != cudaSuccess) return e;
    }
    // programmatic unless an event sits between it and the kernel before it (the caller's mark,
    // or the mixed step's event after the prep kernel when there is no segment pass)
    return launch_tc(kernel, (unsigned)(grid * p.nseg), !before_fused && !(p.nseg == 1 && after_prep), s, mX, mB,
                     mC, mY, p);
}

}  // namespace ssd
