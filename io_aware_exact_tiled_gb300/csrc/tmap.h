// Host-side construction of TMA tensor maps (CUtensorMap) without linking the
// driver library: the encoder is fetched through the runtime's driver entry
// point query.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace fa {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encode_tiled_fn() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    }
    return fn;
}

// Row-major [rows, cols] matrix of `elem_bytes`-byte elements, read in boxes
// of [box_rows, box_cols] with the 128-byte swizzle (box_cols * elem_bytes
// must be 128). Returns false on failure.
inline bool make_tmap_2d_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, int elem_bytes,
                               uint32_t box_rows, uint32_t box_cols) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMapDataType dt = elem_bytes == 1   ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                             : elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                               : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t gdim[2] = {cols, rows};
    cuuint64_t gstride[1] = {cols * static_cast<uint64_t>(elem_bytes)};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estride[2] = {1, 1};
    CUresult r = fn(map, dt, 2, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Packed token-major tensor [tokens][heads][cols] (variable-length batches),
// read in boxes of box_rows consecutive tokens of one head and box_cols
// columns, with the 128-byte swizzle. A box of one head is laid out in shared
// memory exactly like the [box_rows, box_cols] box of make_tmap_2d_sw128.
// Rows past `tokens` read as zero.
inline bool make_tmap_packed_sw128(CUtensorMap* map, const void* base, uint64_t tokens, uint64_t heads,
                                   uint64_t cols, int elem_bytes, uint32_t box_rows, uint32_t box_cols) {
    EncodeTiledFn fn = encode_tiled_fn();
    if (!fn) return false;
    CUtensorMapDataType dt =
        elem_bytes == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    cuuint64_t gdim[3] = {cols, heads, tokens};
    cuuint64_t gstride[2] = {cols * static_cast<uint64_t>(elem_bytes), heads * cols * static_cast<uint64_t>(elem_bytes)};
    cuuint32_t box[3] = {box_cols, 1, box_rows};
    cuuint32_t estride[3] = {1, 1, 1};
    CUresult r = fn(map, dt, 3, const_cast<void*>(base), gdim, gstride, box, estride, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace fa
