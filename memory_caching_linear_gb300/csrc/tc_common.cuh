// tc_common.cuh -- constants and small helpers shared by the tensor-core kernels
// (k_tc.cu: the constant-segment state-form path; k_gen.cu: the general path and
// the factorised readout).
//
// Operand tiles are bf16, 128-byte swizzled (see sm100.cuh): a 128-row tile of
// 128 elements is two 16 KB panels of 64 elements.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "sm100.cuh"

namespace mc {

constexpr int kD = 128;            // the widest head dimension (tiles of the router and the backward are 128 wide)
constexpr int kTcMaxTopk = 16;     // SSC selections per token handled by the tensor-core paths
constexpr int kCT = 128;           // tokens per chunk / tile
constexpr uint32_t kTile = 32768;  // one 128 x 128 bf16 operand tile
constexpr uint32_t kPanel = 16384; // one 128 x 64 bf16 operand panel

// Key-mean image of a head: blocks of 64 segments (row = segment % 64), each three
// 64-row panels holding kbar as hi, mid and lo bf16 terms.  hi = RN(kbar),
// mid = RN(kbar - hi), lo = kbar - hi - mid; both differences are exact in fp32 and lo
// is exactly representable, so hi + mid + lo = kbar and u . kbar (u exact in bf16) is
// a sum of exact products.
constexpr uint32_t kKbPanel = 16384;
constexpr uint32_t kKbImg = 3 * kKbPanel;  // one block of 64 segments

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Element (segment, column) of a head's key-mean image (NB blocks of 64 segments).
__device__ __forceinline__ void store_kbar_terms(uint8_t *head_img, int seg, int col, float kb)
{
    uint8_t *img = head_img + (size_t)(seg >> 6) * kKbImg;
    const __nv_bfloat16 hi = __float2bfloat16_rn(kb);
    const float r1 = kb - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r1 - __bfloat162float(mid));
    const uint32_t off = sm100::sw128_offset(seg & 63, col, 64);
    *reinterpret_cast<__nv_bfloat16 *>(img + off) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(img + kKbPanel + off) = mid;
    *reinterpret_cast<__nv_bfloat16 *>(img + 2 * kKbPanel + off) = lo;
}

// K-major SW128 descriptor start for the 16-wide K step kk of a tile with `rows` rows.
__device__ __forceinline__ uint32_t kmaj_off(int kk, uint32_t rows) { return (kk >> 2) * rows * 128u + (kk & 3) * 32u; }

inline size_t pad256(size_t x) { return (x + 255) & ~(size_t)255; }

// Streaming multiprocessors of the current device (cached per device ordinal).
inline int sm_count()
{
    static int cached[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return 148;
    }
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] <= 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
            cudaGetLastError();
            n = 148;
        }
        cached[dev] = n;
    }
    return cached[dev];
}

}  // namespace mc
