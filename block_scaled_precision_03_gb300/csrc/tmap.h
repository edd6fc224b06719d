// Host-side TMA tensor-map builders (driver entry point resolved at run time).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace bsq {
namespace tmap {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

inline EncodeTiledFn encoder() {
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(f);
    }
    return fn;
}

// K-major code matrix [rows, row_bytes] (uint8), box = 128 bytes x box_rows,
// 128-byte swizzle; out-of-range rows / columns read as zero.
inline bool codes_2d(CUtensorMap* m, const void* ptr, int64_t rows, int64_t row_bytes, uint32_t box_rows) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
    cuuint32_t box[2] = {128u, box_rows};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tiled scale buffer viewed as [bands][atoms][128 x u32]: one 512-byte
// 128x4 tile per (128-row band, group of 4 scale columns).  Box =
// 128 words x box_atoms x box_bands; atoms or bands past the end read as 0.
inline bool scales_3d(CUtensorMap* m, const void* ptr, int64_t bands, int64_t atoms, uint32_t box_atoms,
                      uint32_t box_bands) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[3] = {128, (cuuint64_t)atoms, (cuuint64_t)bands};
    cuuint64_t strides[2] = {512, (cuuint64_t)(atoms * 512)};
    cuuint32_t box[3] = {128u, box_atoms, box_bands};
    cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 3, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The same tiled scale buffer read for a 128x256b scale copy: per atom
// (4 scale columns of a 128-row band; one 16-element block each for NVFP4)
// the box holds box_bands bands x 4 copies of the band's 512-byte tile, i.e.
// for lane r = 32 q + l of the copy the 16-byte row l of each band's tile
// (the scales of rows l, 32 + l, 64 + l, 96 + l of the band).  The copy
// index q has stride 0: the four lane quarters each get the whole tile.
// Box = 128 words x 4 copies x box_bands x box_atoms, atoms outermost.
inline bool scales_4d_quarters(CUtensorMap* m, const void* ptr, int64_t bands, int64_t atoms, uint32_t box_atoms,
                               uint32_t box_bands) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    cuuint64_t dims[4] = {128, 4, (cuuint64_t)bands, (cuuint64_t)atoms};
    cuuint64_t strides[3] = {0, (cuuint64_t)(atoms * 512), 512};
    cuuint32_t box[4] = {128u, 4u, box_bands, box_atoms};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, 4, const_cast<void*>(ptr), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major output matrix [rows, cols] of BF16 or FP32 for TMA stores: box =
// 64 bytes x 32 rows, 64-byte swizzle; elements outside the matrix are not
// written.  Needs a 16-byte aligned base and a row pitch that is a multiple
// of 16 bytes.
inline bool out_2d(CUtensorMap* m, void* ptr, int64_t rows, int64_t cols, int64_t ld, bool bf16) {
    EncodeTiledFn enc = encoder();
    if (!enc) return false;
    const uint32_t esz = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    cuuint64_t strides[1] = {(cuuint64_t)(ld * esz)};
    cuuint32_t box[2] = {64u / esz, 32u};
    cuuint32_t estr[2] = {1, 1};
    return enc(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, ptr, dims, strides, box,
               estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace tmap
}  // namespace bsq
