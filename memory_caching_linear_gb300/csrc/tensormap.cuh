// tensormap.cuh -- host helpers: 2-D and 3-D bf16 TMA descriptors with 128-byte swizzle,
// encoded through the driver entry point (no link-time dependency on libcuda).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

namespace mc {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (fn == nullptr) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
        else
            cudaGetLastError();
    }
    return fn;
}

// A row-major [rows][cols] bf16 matrix moved in boxes of box_rows x box_cols
// elements with the given swizzle.  base must be 16-byte aligned, cols * 2 a
// multiple of 16 and box_cols * 2 no wider than the swizzle span.  Returns false
// if the driver rejects it.
inline bool make_tmap_bf16(CUtensorMap *map, const void *base, unsigned long long rows, unsigned long long cols,
                           unsigned box_cols, unsigned box_rows, CUtensorMapSwizzle swizzle)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// Boxes of box_rows x 64 elements (one 128-byte swizzle panel per box).
inline bool make_tmap_bf16_sw128(CUtensorMap *map, const void *base, unsigned long long rows,
                                 unsigned long long cols, unsigned box_rows)
{
    return make_tmap_bf16(map, base, rows, cols, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

// A [heads][rows][cols] bf16 tensor (row-major, contiguous) moved in boxes of
// box_rows x 64 elements of one head, 128-byte swizzled.  Coordinates are (column,
// row, head); rows at or past `rows` read as zeros (the TMA's out-of-bounds fill), so
// a box that runs past a head's last row never touches the next head.
inline bool make_tmap_bf16_3d_sw128(CUtensorMap *map, const void *base, unsigned long long heads,
                                    unsigned long long rows, unsigned long long cols, unsigned box_rows)
{
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return false;
    cuuint64_t dims[3] = {cols, rows, heads};
    cuuint64_t strides[2] = {cols * 2, rows * cols * 2};
    cuuint32_t box[3] = {64, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                     CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace mc
