// Host helper: encode a 3-D bf16 TMA tensor map with 128-byte swizzle
// (internal).  The driver entry point is fetched through the runtime, so the
// library does not link libcuda directly.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

namespace ssd {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

// Tensor of dims (d0 innermost, d1, d2) 16-bit elements with byte strides
// s1 (between d1 entries) and s2 (between d2 entries); box (b0, b1, b2).
// Returns false if the driver rejects it.
inline bool make_tmap_16bit_3d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t d0, uint64_t d1,
                               uint64_t d2, uint64_t s1, uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {d0, d1, d2};
    cuuint64_t strides[2] = {s1, s2};
    cuuint32_t box[3] = {b0, b1, b2};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, type, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major 2-D tensor [rows, cols] of 2- or 4-byte elements (cols innermost, row stride in
// bytes), box (box_cols, box_rows), no swizzle: the box lands in shared memory as box_rows
// rows of box_cols elements.  Elements outside the tensor read as zeros.
inline bool make_tmap_2d(CUtensorMap *m, CUtensorMapDataType type, const void *base, uint64_t cols, uint64_t rows,
                         uint64_t row_stride, uint32_t box_cols, uint32_t box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {row_stride};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, type, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

inline bool make_tmap_bf16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                              uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    return make_tmap_16bit_3d(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, d0, d1, d2, s1, s2, b0, b1, b2);
}

inline bool make_tmap_f16_3d(CUtensorMap *m, const void *base, uint64_t d0, uint64_t d1, uint64_t d2, uint64_t s1,
                             uint64_t s2, uint32_t b0, uint32_t b1, uint32_t b2) {
    return make_tmap_16bit_3d(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, base, d0, d1, d2, s1, s2, b0, b1, b2);
}

}  // namespace ssd
