// Fused SSD prefill on the sm_103a tensor cores (bf16 operands, fp32 state).
//
// The chunked scan of "[vllm] vLLM Mamba2 SSD 커널 웜업" (section
// "mamba_mixer2.py 변경 사항 (핵심)"), fused into one kernel: one CTA walks one
// (sequence, head) through its chunks in blocks of 128 tokens, keeping the
// fp32 state in registers, so the state crosses HBM only where the method
// requires it -- the optional initial state is read once and the state at the
// end of every chunk is stored to its cache slot (prefix caching, "청크 기반
// 프리픽스 캐싱" on "[vLLM] Mamba (SSM): 선형 시간 복잡도 시퀀스 모델링").
//
// Per block of L <= 128 tokens [tb, tb+L) with in-block cumsum c_t of
// delta*A, the four dense contractions run as tcgen05.mma tiles (fp32
// accumulators).  M1 takes the bf16 inputs as they are; the operands the
// kernel forms itself (P, w x, the carried state) are rounded to fp16, whose
// 11-bit significand keeps their rounding error 8x below bf16's, and the x, B
// and C tiles they meet are converted to fp16 in shared memory (exactly, for
// values in fp16's range) because both operands of an MMA share one type:
//   M1  S  = C B^T                  [128 x 128], K = dstate   (SS, K/K-major)
//   M2  Y1 = P X                    [128 x  64], K = tokens   (TS: P in TMEM)
//        P[t,s] = exp(c_t - c_s) delta_s S[t,s] for s <= t, plus D on the diagonal
//   M3  Y2 = C Hprev^T              [128 x  64], K = dstate   (SS, B MN-major)
//   M4  dS = B^T (w x),  w_s = exp(c_L - c_s) delta_s   [dstate x 64]   (SS, MN/MN)
// and then y_t = Y1 + exp(c_t) Y2,   state <- exp(c_L) state + dS.
//
// Decays are always exponentials of non-positive differences.  For a
// 32-column group j lying entirely at or below row t, exp(c_t - c_s) is split
// at the group's last row e: exp(c_t - c_e) exp(c_e - c_s), both factors <= 1,
// so only the diagonal group needs one exponential per element.
//
// Warp roles (192 threads, two CTAs per SM):
//   warps 0-3  compute: scan of delta, w x, the P pass (TMEM -> TMEM),
//              epilogue (TMEM -> y), state update; thread t owns TMEM lane t
//              (token row t for S/Y, dstate row t for dS and the state)
//   warp 4     TMA producer (C, B, x tiles; 128-byte swizzle)
//   warp 5     TMEM allocation and MMA issue
// Every mbarrier wait is bounded; on a timeout the CTA reports
// SSD_DEVERR_TIMEOUT, drains its own in-flight copies and MMAs, frees its
// TMEM and exits.
#include "common.cuh"
#include "tc_ptx.cuh"
#include "tmap.h"

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
    __nv_bfloat16 *y;
    uint32_t *err;
    const int32_t *seq_order;
};

namespace {
using namespace tc;

constexpr int kL = 128;  // tokens per block
constexpr int kP = 64;   // headdim
constexpr int kN = 128;  // dstate
constexpr int kThreads = 192;
constexpr int kProducerWarp = 4, kMmaWarp = 5;
constexpr uint32_t kTmemCols = 256;
// TMEM columns
constexpr uint32_t COL_S = 0;    // S (128 fp32 columns); P (64 packed bf16x2 columns) overwrites its first half
constexpr uint32_t COL_P = 0;
constexpr uint32_t COL_DS = 64;  // dS, after the P pass has read S
constexpr uint32_t COL_Y1 = 128;
constexpr uint32_t COL_Y2 = 192;
// shared memory (offsets from the 1024-aligned dynamic base)
constexpr uint32_t OFF_C = 0;        // C tile: two [128 x 64] bf16 atoms
constexpr uint32_t OFF_B = 32768;    // B tile
constexpr uint32_t OFF_X = 65536;    // x tile [128 tokens x 64]
constexpr uint32_t OFF_XW = 81920;   // w-scaled x; reused to stage y
constexpr uint32_t OFF_H = 98304;    // bf16 state entering the block, row n = 64 headdim values
constexpr uint32_t OFF_F = 114688;   // column factors [128] fp32
constexpr uint32_t OFF_WT = OFF_F + 512;   // per-warp sums of delta*A [4]
constexpr uint32_t OFF_TM = OFF_WT + 16;   // TMEM base address
constexpr uint32_t OFF_BAR = OFF_WT + 32;  // mbarriers
constexpr uint32_t kSmemBytes = OFF_BAR + 8 * 8;
constexpr uint32_t kTxBytes = 32768 + 32768 + 16384;

enum { BAR_FULL = 0, BAR_EMPTY, BAR_S, BAR_P, BAR_ACC, BAR_DSFREE };

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

// Walks the blocks of one sequence: chunks [first, last], each cut into
// blocks of at most kL tokens that never cross a chunk end.
struct Cursor {
    const int32_t *cu_chunk;
    int k, last, tb, ce;
    __device__ void start(const int32_t *cc, int first, int last_) {
        cu_chunk = cc;
        k = first;
        last = last_;
        tb = cc[first];
        ce = cc[first + 1];
    }
    __device__ int len() const { return min(kL, ce - tb); }
    __device__ bool ends_chunk() const { return tb + len() == ce; }
    __device__ void next() {
        tb += len();
        if (tb == ce && k < last) {
            ++k;
            ce = cu_chunk[k + 1];
        }
    }
};

// fp16 copy of the state row (dstate row n = thread) into the M3 operand tile
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

// row r of a [128 x 128] bf16 tile held as two 64-wide swizzled atoms -> fp16, in place
__device__ __forceinline__ void tile_row_to_f16(uint8_t *tile, int r) {
#pragma unroll
    for (int a = 0; a < 2; ++a) {
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            uint4 *q = reinterpret_cast<uint4 *>(tile + a * 16384 + sw128_offset(r, c));
            *q = bf16x8_to_f16x8(*q);
        }
    }
}

__global__ void __launch_bounds__(kThreads, 2)
    ssd_prefill_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmB,
                          const __grid_constant__ CUtensorMap tmC, const TcParams p) {
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int slot_r = blockIdx.x / p.H;
    const int h = blockIdx.x - slot_r * p.H;
    const int r = p.seq_order ? p.seq_order[slot_r] : slot_r;
    if (r < 0 || r >= p.S) {
        if (threadIdx.x == 0 && h == 0) report(p.err, SSD_DEVERR_METADATA);
        return;
    }
    const int g = h / (p.H / p.G);

    // ---- the sequence's chunk range, validated before anything is set up
    const int first = r > 0 ? p.last_chunk[r - 1] + 1 : 0;
    const int last = p.last_chunk[r];
    if (last < first) return;  // no new tokens
    int nblocks = 0;
    {
        bool bad = first < 0 || last >= p.K || p.cu_chunk[first] != p.cu_seqlens[r] ||
                   p.cu_chunk[last + 1] != p.cu_seqlens[r + 1];
        for (int k = first; !bad && k <= last; ++k) {
            const int a = p.cu_chunk[k], b = p.cu_chunk[k + 1];
            if (a < 0 || b <= a || b > p.T) bad = true;
            else nblocks += (b - a + kL - 1) / kL;
        }
        if (bad) {
            if (tid == 0 && h == 0) report(p.err, SSD_DEVERR_METADATA);
            return;
        }
    }
    if ((smem_u32(smem) & 1023u) != 0) {  // the swizzled tiles need a 1024-byte aligned base
        if (tid == 0) report(p.err, SSD_DEVERR_INTERNAL);
        return;
    }
    uint8_t *sC = smem + OFF_C, *sB = smem + OFF_B, *sX = smem + OFF_X, *sXW = smem + OFF_XW, *sH = smem + OFF_H;
    float *sF = reinterpret_cast<float *>(smem + OFF_F);
    float *sWT = reinterpret_cast<float *>(smem + OFF_WT);
    uint32_t *sTM = reinterpret_cast<uint32_t *>(smem + OFF_TM);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + OFF_BAR);

    if (tid == 0) {
        mbar_init(&bar[BAR_FULL], 1);
        mbar_init(&bar[BAR_EMPTY], 1);
        mbar_init(&bar[BAR_S], 1);
        mbar_init(&bar[BAR_P], 4);
        mbar_init(&bar[BAR_ACC], 1);
        mbar_init(&bar[BAR_DSFREE], 4);
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

    if (warp == kProducerWarp) {
        if (lane == 0) {
            Cursor cur;
            cur.start(p.cu_chunk, first, last);
            int issued = 0;
            for (int i = 0; i < nblocks; ++i, cur.next()) {
                if (i > 0 && !mbar_wait(&bar[BAR_EMPTY], (i - 1) & 1)) {
                    report(p.err, SSD_DEVERR_TIMEOUT);
                    break;
                }
                mbar_arrive_expect_tx(&bar[BAR_FULL], kTxBytes);
                tma_load_3d(sC, &tmC, 0, g, cur.tb, &bar[BAR_FULL]);
                tma_load_3d(sC + 16384, &tmC, 64, g, cur.tb, &bar[BAR_FULL]);
                tma_load_3d(sB, &tmB, 0, g, cur.tb, &bar[BAR_FULL]);
                tma_load_3d(sB + 16384, &tmB, 64, g, cur.tb, &bar[BAR_FULL]);
                tma_load_3d(sX, &tmX, 0, h, cur.tb, &bar[BAR_FULL]);
                issued = i + 1;
            }
            // drain: the last issued copy must land before the CTA may exit
            if (issued > 0) mbar_wait(&bar[BAR_FULL], (issued - 1) & 1);
        }
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            const uint32_t aC = smem_u32(sC), aB = smem_u32(sB), aX = smem_u32(sX), aXW = smem_u32(sXW),
                           aH = smem_u32(sH);
            constexpr uint32_t kIdS = idesc_bf16(128, 128, 0, 0);  // raw bf16 C and B
            constexpr uint32_t kIdY = idesc_f16(128, 64, 0, 1);    // fp16 operands from here on
            constexpr uint32_t kIdD = idesc_f16(128, 64, 1, 1);
            int committed = 0;  // blocks whose final commit was issued
            for (int i = 0; i < nblocks; ++i) {
                const uint32_t ph = i & 1;
                if (!mbar_wait(&bar[BAR_FULL], ph) || (i > 0 && !mbar_wait(&bar[BAR_DSFREE], (i - 1) & 1))) {
                    report(p.err, SSD_DEVERR_TIMEOUT);
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_ss(tm + COL_S, sw128_desc(aC + ko, 16, 1024), sw128_desc(aB + ko, 16, 1024), kIdS, k > 0);
                }
                mma_commit(&bar[BAR_S]);
                if (!mbar_wait(&bar[BAR_P], ph)) {
                    report(p.err, SSD_DEVERR_TIMEOUT);
                    mbar_wait(&bar[BAR_S], ph);  // drain M1
                    break;
                }
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ts(tm + COL_Y1, tm + COL_P + 8 * k, sw128_desc(aX + 2048 * k, 1024, 1024), kIdY, k > 0);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const uint32_t ko = (k >> 2) * 16384 + (k & 3) * 32;
                    mma_ss(tm + COL_Y2, sw128_desc(aC + ko, 16, 1024), sw128_desc(aH + 2048 * k, 1024, 1024), kIdY,
                           k > 0);
                }
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mma_ss(tm + COL_DS, sw128_desc(aB + 2048 * k, 16384, 1024),
                           sw128_desc(aXW + 2048 * k, 1024, 1024), kIdD, k > 0);
                mma_commit(&bar[BAR_ACC]);
                mma_commit(&bar[BAR_EMPTY]);
                committed = i + 1;
            }
            if (committed > 0) mbar_wait(&bar[BAR_EMPTY], (committed - 1) & 1);  // drain
        }
    } else {
        // ------------------------------------------------ compute warps ----
        const int t = tid;  // TMEM lane / token row / dstate row
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
        const float Ah = p.A[h];
        const float Dh = p.D ? p.D[h] : 0.f;
        const float bias = p.dt_bias ? p.dt_bias[h] : 0.f;
        const size_t HPN = (size_t)p.H * kP * kN;
        float st[kP];
        {
            const int32_t is = p.init_slot ? p.init_slot[r] : p.null_id;
            if (slot_usable(is, p.null_id, p.num_slots, t == 0 ? p.err : nullptr)) {
                const float *src = p.cache + (size_t)is * HPN + (size_t)h * kP * kN + t;
#pragma unroll
                for (int q = 0; q < kP; ++q) st[q] = src[(size_t)q * kN];
            } else {
#pragma unroll
                for (int q = 0; q < kP; ++q) st[q] = 0.f;
            }
        }
        store_state_row(sH, t, st);

        Cursor cur;
        cur.start(p.cu_chunk, first, last);
        for (int i = 0; i < nblocks; ++i, cur.next()) {
            const uint32_t ph = i & 1;
            const int tb = cur.tb, L = cur.len();
            // ---- delta, in-block cumsum c_t, factors
            float delta = 0.f, a = 0.f;
            if (t < L) {
                const float v = __bfloat162float(p.dt[(size_t)(tb + t) * p.H + h]) + bias;
                delta = step_delta(v, p.dt_softplus, p.dt_min, p.dt_max);
                a = delta * Ah;
            }
            float c = a;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float v = __shfl_up_sync(0xffffffffu, c, off);
                if (lane >= off) c += v;
            }
            if (lane == 31) sWT[warp] = c;
            named_bar_sync(1, 128);
            float wt[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) wt[j] = sWT[j];
            float prefix = 0.f, own = 0.f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                if (j < warp) prefix += wt[j];
                if (j == warp) own = wt[j];
            }
            c += prefix;                                     // c_t
            const float c_last = wt[0] + wt[1] + wt[2] + wt[3];
            const float c_gend = prefix + own;              // c at the end of my group
            sF[t] = __expf(c_gend - c) * delta;              // column factor of column t
            const float w_x = __expf(c_last - c) * delta;    // state-update weight of token t
            const float e_row = __expf(c);                   // carried-state factor of row t
            const float decay = __expf(c_last);

            // ---- x tile landed: w x into the M4 operand tile
            bool ok = mbar_wait(&bar[BAR_FULL], ph);
            if (!named_bar_and(1, 128, ok)) {
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            {
                // x row t: w x into the M4 operand (fp16) and x itself -> fp16 in place (M2 operand)
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    uint4 v = *reinterpret_cast<const uint4 *>(sX + sw128_offset(t, cc));
                    uint4 xw;
                    xw.x = pack_f16_sat(w_x * __uint_as_float(v.x << 16), w_x * __uint_as_float(v.x & 0xFFFF0000u));
                    xw.y = pack_f16_sat(w_x * __uint_as_float(v.y << 16), w_x * __uint_as_float(v.y & 0xFFFF0000u));
                    xw.z = pack_f16_sat(w_x * __uint_as_float(v.z << 16), w_x * __uint_as_float(v.z & 0xFFFF0000u));
                    xw.w = pack_f16_sat(w_x * __uint_as_float(v.w << 16), w_x * __uint_as_float(v.w & 0xFFFF0000u));
                    *reinterpret_cast<uint4 *>(sXW + sw128_offset(t, cc)) = xw;
                    *reinterpret_cast<uint4 *>(sX + sw128_offset(t, cc)) = bf16x8_to_f16x8(v);
                }
            }
            // ---- S ready: P pass, S (fp32) -> P (bf16) in TMEM
            ok = mbar_wait(&bar[BAR_S], ph);
            if (!named_bar_and(1, 128, ok)) {  // also publishes sF to the compute warps
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t pk[16];
                if (j < warp) {
                    uint32_t v[32];
                    tmem_ld32(tm + lane_base + COL_S + 32 * j, v);
                    tmem_ld_wait();
                    float gend = 0.f;
#pragma unroll
                    for (int q = 0; q <= j; ++q) gend += wt[q];
                    const float R = __expf(c - gend);
                    const float4 *f4 = reinterpret_cast<const float4 *>(sF + 32 * j);
#pragma unroll
                    for (int q = 0; q < 8; ++q) {
                        const float4 f = f4[q];
                        pk[2 * q] = pack_f16_sat(__uint_as_float(v[4 * q]) * f.x * R, __uint_as_float(v[4 * q + 1]) * f.y * R);
                        pk[2 * q + 1] = pack_f16_sat(__uint_as_float(v[4 * q + 2]) * f.z * R,
                                                     __uint_as_float(v[4 * q + 3]) * f.w * R);
                    }
                } else if (j == warp) {
                    uint32_t v[32];
                    tmem_ld32(tm + lane_base + COL_S + 32 * j, v);
                    tmem_ld_wait();
                    float pv[32];
#pragma unroll
                    for (int q = 0; q < 32; ++q) {
                        const float cs_s = __shfl_sync(0xffffffffu, c, q);
                        const float d_s = __shfl_sync(0xffffffffu, delta, q);
                        float val = q <= lane ? __uint_as_float(v[q]) * __expf(c - cs_s) * d_s : 0.f;
                        if (q == lane) val += Dh;
                        pv[q] = val;
                    }
#pragma unroll
                    for (int q = 0; q < 16; ++q) pk[q] = pack_f16_sat(pv[2 * q], pv[2 * q + 1]);
                } else {
#pragma unroll
                    for (int q = 0; q < 16; ++q) pk[q] = 0u;
                }
                tmem_st16(tm + lane_base + COL_P + 16 * j, pk);
            }
            // M1 is done with the raw tiles: C and B rows -> fp16 for M3 and M4
            tile_row_to_f16(sC, t);
            tile_row_to_f16(sB, t);
            tmem_st_wait();
            fence_proxy_async_smem();  // w x, x, B, C and the state tile -> async proxy
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar[BAR_P]);

            // ---- accumulators ready
            ok = mbar_wait(&bar[BAR_ACC], ph);
            if (!named_bar_and(1, 128, ok)) {
                if (t == 0) report(p.err, SSD_DEVERR_TIMEOUT);
                break;
            }
            tc_fence_after();
            {
                uint32_t d0[32], d1[32];
                tmem_ld32(tm + lane_base + COL_DS, d0);
                tmem_ld32(tm + lane_base + COL_DS + 32, d1);
                tmem_ld_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&bar[BAR_DSFREE]);
#pragma unroll
                for (int q = 0; q < 32; ++q) {
                    st[q] = fmaf(decay, st[q], __uint_as_float(d0[q]));
                    st[32 + q] = fmaf(decay, st[32 + q], __uint_as_float(d1[q]));
                }
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t y1[32], y2[32];
                tmem_ld32(tm + lane_base + COL_Y1 + 32 * half, y1);
                tmem_ld32(tm + lane_base + COL_Y2 + 32 * half, y2);
                tmem_ld_wait();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint4 v;
                    uint32_t *vv = reinterpret_cast<uint32_t *>(&v);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const int e = 8 * cc + 2 * q;
                        vv[q] = pack_bf16(fmaf(e_row, __uint_as_float(y2[e]), __uint_as_float(y1[e])),
                                          fmaf(e_row, __uint_as_float(y2[e + 1]), __uint_as_float(y1[e + 1])));
                    }
                    *reinterpret_cast<uint4 *>(sXW + sw128_offset(t, 4 * half + cc)) = v;
                }
            }
            store_state_row(sH, t, st);
            if (cur.ends_chunk()) {
                const int32_t cs = p.chunk_slot ? p.chunk_slot[cur.k] : p.null_id;
                if (slot_usable(cs, p.null_id, p.num_slots, t == 0 ? p.err : nullptr)) {
                    float *dst = p.cache + (size_t)cs * HPN + (size_t)h * kP * kN + t;
#pragma unroll
                    for (int q = 0; q < kP; ++q) dst[(size_t)q * kN] = st[q];
                }
            }
            named_bar_sync(1, 128);  // y tile staged
#pragma unroll
            for (int rr = 0; rr < 8; ++rr) {
                const int row = rr * 16 + (t >> 3), cc = t & 7;
                if (row < L) {
                    const uint4 v = *reinterpret_cast<const uint4 *>(sXW + sw128_offset(row, cc));
                    *reinterpret_cast<uint4 *>(p.y + ((size_t)(tb + row) * p.H + h) * kP + 8 * cc) = v;
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tm, kTmemCols);
    }
}

}  // namespace

bool tc_prefill_supported(const ssd_prefill_args &a) {
    return a.dtype == SSD_BF16 && a.headdim == kP && a.dstate == kN && a.total_tokens > 0;
}

cudaError_t tc_prefill_launch(const ssd_prefill_args &a, cudaStream_t s) {
    CUtensorMap mX, mB, mC;
    const uint64_t T = (uint64_t)a.total_tokens;
    if (!make_tmap_bf16_3d(&mX, a.x, kP, a.nheads, T, (uint64_t)kP * 2, (uint64_t)a.nheads * kP * 2, 64, 1, kL) ||
        !make_tmap_bf16_3d(&mB, a.B, kN, a.ngroups, T, (uint64_t)kN * 2, (uint64_t)a.ngroups * kN * 2, 64, 1, kL) ||
        !make_tmap_bf16_3d(&mC, a.C, kN, a.ngroups, T, (uint64_t)kN * 2, (uint64_t)a.ngroups * kN * 2, 64, 1, kL))
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
    p.y = static_cast<__nv_bfloat16 *>(a.y);
    p.err = a.err_word;
    p.seq_order = a.seq_order;
    cudaError_t e = cudaFuncSetAttribute(ssd_prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes);
    if (e != cudaSuccess) return e;
    const long long grid = (long long)a.num_seqs * a.nheads;
    if (grid <= 0) return cudaSuccess;
    ssd_prefill_tc_kernel<<<(unsigned)grid, kThreads, kSmemBytes, s>>>(mX, mB, mC, p);
    return cudaGetLastError();
}

}  // namespace ssd
