// mc_selftest.cu -- diagnostic kernels (include/mc_selftest.h): one tcgen05 MMA
// chain per operand form the forward kernels use, and a bounded-wait check.
#include <cstdint>

#include "mc_internal.cuh"
#include "mc_selftest.h"
#include "sm100.cuh"
#include "tensormap.cuh"

namespace mc {
namespace {

using namespace sm100;

struct UmmaArgs {
    const __nv_bfloat16 *X;
    float *D;
    int form;
    int *err;
};

__global__ void __launch_bounds__(128) umma_selftest_kernel(const __grid_constant__ CUtensorMap mX,
                                                            const __grid_constant__ CUtensorMap mW,
                                                            const __grid_constant__ CUtensorMap mW64, UmmaArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t *sX = sm;
    uint8_t *sW = sm + 32768;
    __shared__ uint64_t bar_tma, bar_mma;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int tid = threadIdx.x, warp = tid / 32;
    const int form = a.form;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (tid == 0) {
        abort_flag = 0;
        mbar_init(&bar_tma, 1);
        mbar_init(&bar_mma, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t a_tmem = tb + 128;

    if (tid == 0) {
        mbar_arrive_expect_tx(&bar_tma, form == 4 ? 32768u + 16384u : 65536u);
        tma_load_2d(sX, &mX, 0, 0, &bar_tma);
        tma_load_2d(sX + 16384, &mX, 64, 0, &bar_tma);
        if (form == 4) {
            tma_load_2d(sW, &mW64, 0, 0, &bar_tma);
            tma_load_2d(sW + 8192, &mW64, 64, 0, &bar_tma);
        } else {
            tma_load_2d(sW, &mW, 0, 0, &bar_tma);
            tma_load_2d(sW + 16384, &mW, 64, 0, &bar_tma);
        }
    }
    bool ok = mbar_wait(&bar_tma, 0, &abort_flag);

    const bool a_in_tmem = form == 1 || form == 2 || form == 4;
    if (a_in_tmem) {
        const __nv_bfloat16 *row = a.X + (size_t)tid * 128;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            uint32_t r[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
                r[i] = pack_bf16x2(__bfloat162float(row[32 * j + 2 * i]), __bfloat162float(row[32 * j + 2 * i + 1]));
            tmem_st16(tmem_addr(a_tmem, warp * 32, 16 * j), r);
        }
        tmem_wait_st();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0 && ok) {
        const uint32_t x0 = smem_u32(sX), w0 = smem_u32(sW);
        for (int kk = 0; kk < 8; ++kk) {
            const uint32_t acc = kk > 0;
            const uint32_t kmaj = (kk >> 2) * 16384u + (kk & 3) * 32u;  // K step in a 128-row K-major tile
            const uint32_t mnmaj = kk * 2048u;                           // K step in an MN-major tile
            switch (form) {
            case 0:
                mma_ss(tb, make_desc_sw128(x0 + kmaj, 0, 1024), make_desc_sw128(w0 + kmaj, 0, 1024),
                       idesc_bf16(128, 128, false, false), acc);
                break;
            case 1:
                mma_ts(tb, a_tmem + kk * 8, make_desc_sw128(w0 + kmaj, 0, 1024), idesc_bf16(128, 128, false, false),
                       acc);
                break;
            case 2:
                mma_ts(tb, a_tmem + kk * 8, make_desc_sw128(w0 + mnmaj, 16384, 1024),
                       idesc_bf16(128, 128, false, true), acc);
                break;
            case 3:
                mma_ss(tb, make_desc_sw128(x0 + mnmaj, 16384, 1024), make_desc_sw128(w0 + mnmaj, 16384, 1024),
                       idesc_bf16(128, 128, true, true), acc);
                break;
            case 4:
                mma_ts(tb, a_tmem + kk * 8, make_desc_sw128(w0 + (kk >> 2) * 8192u + (kk & 3) * 32u, 0, 1024),
                       idesc_bf16(128, 64, false, false), acc);
                break;
            default:
                mma_ss(tb, make_desc_sw128(x0 + kmaj, 0, 1024), make_desc_sw128(w0 + mnmaj, 16384, 1024),
                       idesc_bf16(128, 128, false, true), acc);
                break;
            }
        }
        mma_commit(&bar_mma);
    }
    if (ok) ok = mbar_wait(&bar_mma, 0, &abort_flag);
    tc_fence_after();
    const int ncols = form == 4 ? 64 : 128;
    for (int j = 0; j < ncols / 16; ++j) {
        uint32_t r[16];
        tmem_ld16(tmem_addr(tb, warp * 32, 16 * j), r);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) a.D[(size_t)tid * 128 + 16 * j + i] = ok ? __uint_as_float(r[i]) : __int_as_float(0x7fc00000);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tb, 256);
    if (!ok && tid == 0) atomicExch(a.err, 1);
}

__global__ void wait_timeout_kernel(int *status, unsigned long long limit_ns)
{
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        abort_flag = 0;
        mbar_init(&bar, 1);  // nobody ever arrives
        fence_mbar_init();
    }
    __syncthreads();
    const bool ok = mbar_wait_limit(&bar, 0, &abort_flag, limit_ns);
    __syncthreads();
    if (threadIdx.x == 0) *status = ok ? 0 : 1;
}

}  // namespace
}  // namespace mc

extern "C" int mc_selftest_umma(const void *X, const void *W, float *D, int form, mc_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (!X || !W || !D) return MC_ERR_NULL;
    if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(W) | reinterpret_cast<uintptr_t>(D)) & 15u)
        return MC_ERR_ALIGN;
    if (form < 0 || form > 5) return MC_ERR_MODE;
    CUtensorMap mX, mW, mW64;
    if (!mc::make_tmap_bf16_sw128(&mX, X, 128, 128, 128) || !mc::make_tmap_bf16_sw128(&mW, W, 128, 128, 128) ||
        !mc::make_tmap_bf16_sw128(&mW64, W, 128, 128, 64))
        return MC_ERR_CUDA;
    int *err = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&err), sizeof(int), stream) != cudaSuccess) return MC_ERR_ALLOC;
    cudaMemsetAsync(err, 0, sizeof(int), stream);
    const size_t smem = 65536 + 1024;
    cudaFuncSetAttribute(mc::umma_selftest_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    mc::UmmaArgs a{static_cast<const __nv_bfloat16 *>(X), D, form, err};
    mc::umma_selftest_kernel<<<1, 128, smem, stream>>>(mX, mW, mW64, a);
    cudaError_t e = cudaGetLastError();
    int h_err = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h_err, err, sizeof(int), cudaMemcpyDeviceToHost, stream);
    cudaFreeAsync(err, stream);
    cudaError_t es = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || es != cudaSuccess) return MC_ERR_CUDA;
    return h_err ? MC_ERR_DEVICE_TIMEOUT : MC_OK;
}

extern "C" int mc_selftest_wait_timeout(int limit_ms, mc_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (limit_ms < 1 || limit_ms > 5000) return MC_ERR_SHAPE;
    int *st = nullptr;
    if (cudaMallocAsync(reinterpret_cast<void **>(&st), sizeof(int), stream) != cudaSuccess) return MC_ERR_ALLOC;
    mc::wait_timeout_kernel<<<1, 32, 0, stream>>>(st, (unsigned long long)limit_ms * 1000000ull);
    cudaError_t e = cudaGetLastError();
    int h = -1;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&h, st, sizeof(int), cudaMemcpyDeviceToHost, stream);
    cudaFreeAsync(st, stream);
    cudaError_t es = cudaStreamSynchronize(stream);
    if (e != cudaSuccess || es != cudaSuccess) return MC_ERR_CUDA;
    return h == 1 ? MC_ERR_DEVICE_TIMEOUT : MC_OK;
}
