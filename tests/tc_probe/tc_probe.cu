// Test-only probe: checks, on one CTA, each tensor-core operand form the
// fused prefill kernel uses, against plain matrix products computed by the
// test.  Inputs (bf16, row-major):
//   Cg [128 x 128], Bg [128 x 128], Xg [128 x 64]   -> TMA, 128B swizzle
//   Hg [128 x 64], Wg [128 x 64]                     -> written by threads
//   Pg [128 x 128]                                   -> tcgen05.st into TMEM
// Outputs (fp32):
//   O1 = Cg Bg^T  (SS, K-major A and B, N=128)
//   O2 = Pg Xg    (TS, A in TMEM, B MN-major, N=64)
//   O3 = Cg Hg    (SS, K-major A, MN-major B)
//   O4 = Bg^T Wg  (SS, MN-major A over two 64-wide atoms, MN-major B)
//   O5 = Bg^T Wg  with the two descriptor offsets of A swapped (diagnostic)
//   O6 = Cg [Hg | Wg]  (SS, K-major A, MN-major B over two 64-wide atoms, N=128;
//                       a second phase, after O1..O5 were read)
#include <cuda_bf16.h>
#include <stdint.h>

#include "tc_ptx.cuh"
#include "tmap.h"

using namespace ssd::tc;

namespace {

constexpr uint32_t kSmem = 200 * 1024;

__global__ void __launch_bounds__(128, 1) probe_kernel(const __grid_constant__ CUtensorMap tmC,
                                                        const __grid_constant__ CUtensorMap tmB,
                                                        const __grid_constant__ CUtensorMap tmX,
                                                        const __nv_bfloat16 *Hg, const __nv_bfloat16 *Wg,
                                                        const __nv_bfloat16 *Pg, float *O1, float *O2, float *O3,
                                                        float *O4, float *O5, float *O6, int *status) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sC = smem;              // 32 KB: two [128 x 64] atoms
    uint8_t *sB = smem + 32768;      // 32 KB
    uint8_t *sX = smem + 65536;      // 16 KB
    uint8_t *sH = smem + 81920;      // 16 KB
    uint8_t *sW = smem + 98304;      // 16 KB
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + 131072);
    uint32_t *tbase = reinterpret_cast<uint32_t *>(smem + 131072 + 64);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        mbar_init(&bars[0], 1);
        mbar_init(&bars[1], 1);
        mbar_init(&bars[2], 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(tbase, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tm = *tbase;
    if (tid == 0) {
        mbar_arrive_expect_tx(&bars[0], 32768 + 32768 + 16384);
        tma_load_3d(sC, &tmC, 0, 0, 0, &bars[0]);
        tma_load_3d(sC + 16384, &tmC, 64, 0, 0, &bars[0]);
        tma_load_3d(sB, &tmB, 0, 0, 0, &bars[0]);
        tma_load_3d(sB + 16384, &tmB, 64, 0, 0, &bars[0]);
        tma_load_3d(sX, &tmX, 0, 0, 0, &bars[0]);
    }
    // thread r writes row r of H and W (64 bf16 = 8 chunks of 16 bytes)
    {
        const uint4 *h = reinterpret_cast<const uint4 *>(Hg + tid * 64);
        const uint4 *w = reinterpret_cast<const uint4 *>(Wg + tid * 64);
        for (int c = 0; c < 8; ++c) {
            *reinterpret_cast<uint4 *>(sH + sw128_offset(tid, c)) = h[c];
            *reinterpret_cast<uint4 *>(sW + sw128_offset(tid, c)) = w[c];
        }
    }
    // P row `tid` into TMEM columns [128, 192): 64 columns of packed bf16 pairs
    {
        const uint32_t *p = reinterpret_cast<const uint32_t *>(Pg + tid * 128);
        for (int j = 0; j < 4; ++j) {
            uint32_t r[16];
            for (int i = 0; i < 16; ++i) r[i] = p[16 * j + i];
            tmem_st16(tmem_addr(tm, warp * 32, 128 + 16 * j), r);
        }
        tmem_st_wait();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    if (tid == 0) {
        tc_fence_after();
        bool ok = mbar_wait(&bars[0], 0);
        if (!ok) {
            atomicOr(status, 1);
        } else {
            const uint32_t aC = smem_u32(sC), aB = smem_u32(sB), aX = smem_u32(sX), aH = smem_u32(sH),
                           aW = smem_u32(sW);
            for (int k = 0; k < 8; ++k) {
                const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
                mma_ss(tm + 0, sw128_desc(aC + koff, 16, 1024), sw128_desc(aB + koff, 16, 1024),
                       idesc_bf16(128, 128, 0, 0), k > 0);
            }
            for (int k = 0; k < 8; ++k)
                mma_ts(tm + 192, tm + 128 + 8 * k, sw128_desc(aX + 2048 * k, 1024, 1024), idesc_bf16(128, 64, 0, 1),
                       k > 0);
            for (int k = 0; k < 8; ++k) {
                const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
                mma_ss(tm + 256, sw128_desc(aC + koff, 16, 1024), sw128_desc(aH + 2048 * k, 1024, 1024),
                       idesc_bf16(128, 64, 0, 1), k > 0);
            }
            for (int k = 0; k < 8; ++k)
                mma_ss(tm + 320, sw128_desc(aB + 2048 * k, 16384, 1024), sw128_desc(aW + 2048 * k, 1024, 1024),
                       idesc_bf16(128, 64, 1, 1), k > 0);
            for (int k = 0; k < 8; ++k)
                mma_ss(tm + 384, sw128_desc(aB + 2048 * k, 1024, 16384), sw128_desc(aW + 2048 * k, 1024, 1024),
                       idesc_bf16(128, 64, 1, 1), k > 0);
            mma_commit(&bars[1]);
        }
    }
    __syncthreads();
    const bool ok = mbar_wait(&bars[1], 0);  // also gates phase 2
    if (!ok) atomicOr(status, 2);
    tc_fence_after();
    if (ok) {
        const int row = warp * 32 + lane;
        uint32_t r[32];
        for (int j = 0; j < 4; ++j) {
            tmem_ld32(tmem_addr(tm, warp * 32, 32 * j), r);
            tmem_ld_wait();
            for (int i = 0; i < 32; ++i) O1[row * 128 + 32 * j + i] = __uint_as_float(r[i]);
        }
        float *outs[4] = {O2, O3, O4, O5};
        for (int o = 0; o < 4; ++o)
            for (int j = 0; j < 2; ++j) {
                tmem_ld32(tmem_addr(tm, warp * 32, 192 + 64 * o + 32 * j), r);
                tmem_ld_wait();
                for (int i = 0; i < 32; ++i) outs[o][row * 64 + 32 * j + i] = __uint_as_float(r[i]);
            }
    }
    // phase 2: the H and W tiles are adjacent 16 KB atoms, one MN-major B operand with N = 128
    tc_fence_before();
    __syncthreads();
    if (tid == 0 && ok) {
        tc_fence_after();
        const uint32_t aC = smem_u32(sC), aH = smem_u32(sH);
        for (int k = 0; k < 8; ++k) {
            const uint32_t koff = (k >> 2) * 16384 + (k & 3) * 32;
            mma_ss(tm + 0, sw128_desc(aC + koff, 16, 1024), sw128_desc(aH + 2048 * k, 16384, 1024),
                   idesc_bf16(128, 128, 0, 1), k > 0);
        }
        mma_commit(&bars[2]);
    }
    __syncthreads();
    if (ok) {
        const bool ok2 = mbar_wait(&bars[2], 0);
        if (!ok2) atomicOr(status, 4);
        tc_fence_after();
        if (ok2) {
            const int row = warp * 32 + lane;
            uint32_t r[32];
            for (int j = 0; j < 4; ++j) {
                tmem_ld32(tmem_addr(tm, warp * 32, 32 * j), r);
                tmem_ld_wait();
                for (int i = 0; i < 32; ++i) O6[row * 128 + 32 * j + i] = __uint_as_float(r[i]);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tm, 512);
    }
}

}  // namespace

extern "C" int tc_probe_run(const void *Cg, const void *Bg, const void *Xg, const void *Hg, const void *Wg,
                            const void *Pg, float *O1, float *O2, float *O3, float *O4, float *O5, float *O6,
                            int *status, void *stream) {
    CUtensorMap mC, mB, mX;
    if (!ssd::make_tmap_bf16_3d(&mC, Cg, 128, 1, 128, 256, 256, 64, 1, 128)) return 1;
    if (!ssd::make_tmap_bf16_3d(&mB, Bg, 128, 1, 128, 256, 256, 64, 1, 128)) return 2;
    if (!ssd::make_tmap_bf16_3d(&mX, Xg, 64, 1, 128, 128, 128, 64, 1, 128)) return 3;
    if (cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem + 1024) != cudaSuccess)
        return 4;
    probe_kernel<<<1, 128, kSmem + 1024, static_cast<cudaStream_t>(stream)>>>(
        mC, mB, mX, static_cast<const __nv_bfloat16 *>(Hg), static_cast<const __nv_bfloat16 *>(Wg),
        static_cast<const __nv_bfloat16 *>(Pg), O1, O2, O3, O4, O5, O6, status);
    return cudaGetLastError() == cudaSuccess ? 0 : 5;
}
