// k_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) path of the Memory Caching forward for
// bf16 inputs, seg_len a multiple of 128, L a multiple of seg_len, Residual / GRM / Soup /
// SSC (topk <= 16) / Mean: the host launchers of the state-form kernels of
// tc_state_form.cuh at head dimension 128 (k_tc64.cu launches the 64-wide ones), the
// shape predicates, the state pass the backward reads, and the SSC router's kernels.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
//
// gate_tiles_tc -- the scores <u_t, kbar_i> per 128-token chunk (kbar as hi + mid + lo
//   bf16 rows), for the SSC router alone (the selected segments of every token) and for
//   the gates of the backward pass.
// kbar_images_tc -- the key means alone, as the router's operand image.
#include <cstdint>

#include "mc_internal.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"
#include "tensormap.cuh"
#include "tc_state_form.cuh"

namespace mc {
namespace {


// Key means alone, as hi/lo bf16 image rows (for the stand-alone SSC router):
// the same sequential fp32 sum over the segment's tokens as seg_state_tc, so the
// router sees bit-identical scores.
__global__ void __launch_bounds__(kD) kbar_images_tc(const __nv_bfloat16 *__restrict__ k, TcArgs a)
{
    const int seg = blockIdx.x % a.N, bh = blockIdx.x / a.N;
    const int col = threadIdx.x;
    if (col >= a.d) return;  // the image's padded columns stay zero
    const __nv_bfloat16 *src = k + ((size_t)bh * a.L + (size_t)seg * a.C) * a.d + col;
    float s = 0.f;
    for (int c0 = 0; c0 < a.C; c0 += kCT) {  // the state kernel's order: 16-row groups, then chunks
        float cs = 0.f;
        for (int rg = 0; rg < 8; ++rg) {
            float p = 0.f;
            for (int i = 0; i < 16; ++i) p += __bfloat162float(src[(size_t)(c0 + 16 * rg + i) * a.d]);
            cs += p;
        }
        s += cs;
    }
    store_kbar_terms(a.kbar_img + (size_t)bh * a.NB * kKbImg, seg, col, s / (float)a.C);
}

// ============================================================================
// gate_tiles_tc -- the SSC router ([MC-sum §3.4]): for every token the topk
// cached segments with the largest scores r_{t,i} = <u_t, kbar_i> (i < n), in rank
// order, equal scores to the lower index, -1 padded; or the backward's gates.  Per 128-token chunk;
// the scores come from three MMA sets (kbar as hi + mid + lo bf16 rows, which sum to the
// fp32 kbar exactly; u is exact in bf16), so each score is an fp32 sum of exact products.
// ============================================================================
constexpr int kRouterThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 selection
constexpr size_t kRouterSmem = 2 * kTile + kKbImg + 1024;  // two U tiles, one key-mean image (one CTA per SM)

// Persistent: CTA b handles the contiguous tile range [b*per, (b+1)*per) of the
// (bh, chunk) tiles, so consecutive tiles share a head and its kbar image.
// MODE 0: the SSC router (sel_out).  MODE 1 / 2: the gates of the backward pass --
// GRM / Soup softmax, or SSC -- with the online score r_on, written as g_{t,i}
// ([N][L] per head, 0 where not taken) and the online gate.
template <int MODE>
__global__ void __launch_bounds__(kRouterThreads, 1) gate_tiles_tc(const __grid_constant__ CUtensorMap mU, TcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sU = sm, *sKb = sm + 2 * kTile;
    __shared__ uint64_t u_full[2], u_empty[2], kb_full, kb_empty, s_full[2], s_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int chunks = a.L / kCT;
    const int total = a.BH * chunks;
    const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int first = (int)blockIdx.x * per;
    const int last = min(total, first + per);  // tiles [first, last)
    if (warp == 0) {
        tmem_alloc(&tmem_base, 128);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&u_full[i], 1);
            mbar_init(&u_empty[i], 1);
            mbar_init(&s_full[i], 1);
            mbar_init(&s_empty[i], 128);
        }
        mbar_init(&kb_full, 1);
        mbar_init(&kb_empty, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mU);
            int kb_round = 0, prev_bh = -1;
            for (int it = first; it < last; ++it) {
                const int i = it - first;
                const int bh = it / chunks, t0 = (it % chunks) * kCT;
                if (bh != prev_bh) {
                    if (!mbar_wait(&kb_empty, (kb_round & 1) ^ 1, &abort_flag)) break;
                    mbar_arrive_expect_tx(&kb_full, kKbImg);
                    bulk_load(sKb, a.kbar_img + (size_t)bh * kKbImg, kKbImg, &kb_full);
                    ++kb_round;
                    prev_bh = bh;
                }
                const int b = i & 1;
                if (!mbar_wait(&u_empty[b], ((i >> 1) & 1) ^ 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&u_full[b], kTile);
                tma_load_2d(sU + b * kTile, &mU, 0, bh * a.L + t0, &u_full[b]);
                tma_load_2d(sU + b * kTile + 16384, &mU, 64, bh * a.L + t0, &u_full[b]);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
            const uint64_t dKb = make_desc_sw128(smem_u32(sKb), 0, 1024);
            int kb_round = 0, prev_bh = -1;
            for (int it = first; it < last; ++it) {
                const int i = it - first, b = i & 1;
                const int bh = it / chunks;
                if (bh != prev_bh) {
                    if (!mbar_wait(&kb_full, kb_round & 1, &abort_flag)) break;
                    ++kb_round;
                    prev_bh = bh;
                }
                if (!mbar_wait(&u_full[b], (i >> 1) & 1, &abort_flag)) break;
                if (!mbar_wait(&s_empty[b], ((i >> 1) & 1) ^ 1, &abort_flag)) break;
                tc_fence_after();
                const uint64_t dU = make_desc_sw128(smem_u32(sU + b * kTile), 0, 1024);
                const uint32_t td = tb + b * 64;
#pragma unroll
                for (int term = 0; term < 3; ++term)  // hi, mid, lo
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(td, dU + (kmaj_off(kk, 128) >> 4), dKb + ((term * kKbPanel + kmaj_off(kk, 64)) >> 4), idS,
                               (term | kk) != 0);
                mma_commit(&s_full[b]);
                mma_commit(&u_empty[b]);
                if (it + 1 == last || (it + 1) / chunks != bh) mma_commit(&kb_empty);  // last tile of this head
            }
        }
    } else {
        // Two epilogue groups (warps 2-5 and 6-9) take alternate tiles, matching the
        // two score buffers.
        const int grp = (warp - 2) >> 2;
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        for (int it = first + grp; it < last; it += 2) {
            const int i = it - first, b = i & 1;
            const int bh = it / chunks, t0 = (it % chunks) * kCT;
            const int n = t0 / a.C;
            if (!mbar_wait(&s_full[b], (i >> 1) & 1, &abort_flag)) break;
            tc_fence_after();
            // Only the first n scores take part (n is the same for the whole tile).
            float sc[64];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                if (16 * m < n) {
                    tmem_ld16f(tb + b * 64 + lane_base + 16 * m, sc + 16 * m);
                } else {
#pragma unroll
                    for (int k = 0; k < 16; ++k) sc[16 * m + k] = 0.f;
                }
            }
            tmem_wait_ld();
            tc_fence_before();
            mbar_arrive(&s_empty[b]);
            const size_t tok = (size_t)bh * a.L + t0 + row;
            if (MODE == 0) {
                token_gates<true>(sc, n, 0.f, a.topk, a.sel_out + tok * a.topk);
            } else {
                const float inv = token_gates<MODE == 2>(sc, n, a.r_on[tok], a.topk, nullptr);
                float *g = a.gam_out + (size_t)bh * a.N * a.L + t0 + row;
                for (int k = 0; k < n; ++k) g[(size_t)k * a.L] = sc[k] * inv;
                a.tok_out[tok * kBwdTokWords + 2] = sc[63] * inv;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 128);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_tc_abort, 1);
}

int g_num_sms = 0;

}  // namespace

cudaError_t take_device_abort(int *was_set) { return take_tc_abort(was_set); }

constexpr int kTcMaxN = 512;  // cached segments the gate kernel handles (gates through HBM beyond 64)

bool tc_supported(const Problem &p)
{
    return p.bf16 && (p.d == kD || p.d == 64) && p.C % kCT == 0 && p.L % p.C == 0 &&
           (!mode_uses_u(p.mode) || p.N <= kTcMaxN) &&
           (p.mode == MC_GRM || p.mode == MC_SOUP || p.mode == MC_RESIDUAL ||
            p.mode == MC_MEAN || (p.mode == MC_SSC && p.topk >= 0 && p.topk <= kTcMaxTopk));
}

bool tc_fused_gates(const Problem &p) { return tc_supported(p) && p.N <= 64; }

size_t tc_scratch_bytes(const Problem &p) { return forward_scratch_bytes(p); }

// SSC router alone (mc_ssc_select) on the tensor-core path's shapes: key-mean
// images, then the router kernel.
size_t tc_select_scratch_bytes(const Problem &p) { return pad256((size_t)p.BH * kKbImg); }

cudaError_t launch_ssc_select_tc(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    TcArgs a{};
    a.kbar_img = static_cast<uint8_t *>(scratch);
    a.sel_out = fa.sel_out;
    a.topk = p.topk;
    a.BH = p.BH;
    a.L = p.L;
    a.C = p.C;
    a.N = p.N;
    a.CPS = p.C / kCT;
    a.d = p.d; a.NB = (p.N + 63) / 64;
    CUtensorMap mU;
    if (!make_tmap_bf16_sw128(&mU, fa.u, (unsigned long long)p.BH * p.L, p.d, 128)) return cudaErrorInvalidValue;
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    cudaError_t e = cudaMemsetAsync(a.kbar_img, 0, (size_t)p.BH * kKbImg, s);
    if (e != cudaSuccess) return e;
    kbar_images_tc<<<(unsigned)(p.BH * p.N), kD, 0, s>>>(static_cast<const __nv_bfloat16 *>(fa.k), a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gate_tiles_tc<0>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRouterSmem);
    if (e != cudaSuccess) return e;
    const int gtiles = p.BH * (p.L / kCT);
    const int ggrid = gtiles < g_num_sms ? gtiles : g_num_sms;
    gate_tiles_tc<0><<<ggrid, kRouterThreads, kRouterSmem, s>>>(mU, a);
    return cudaGetLastError();
}

size_t tc_state_scratch_bytes(const Problem &p)
{
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT;
    return pad256(BH * N * kTile) + pad256(BH * N * CPS * kTile) + pad256(BH * kKbImg) + pad256(sizeof(float) * BH * p.L);
}

// The forward's segment-state kernel alone (plain update): the fp32 states, their and
// the chunks' prefix-state bf16 images and, for the routed aggregations, the online
// scores r_on and the key-mean images -- the operands the tensor-core backward reads.
cudaError_t launch_state_tc(const Problem &p, const FwdArgs &fa, void *scratch, TcImages *out, cudaStream_t s)
{
    const bool gated = mode_uses_u(p.mode);
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    TcArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(fa.q);
    a.u = static_cast<const __nv_bfloat16 *>(fa.u);
    a.states = fa.states;
    a.states_img = base;
    base += pad256(BH * N * kTile);
    a.spre_img = base;
    base += pad256(BH * N * CPS * kTile);
    a.kbar_img = base;
    base += pad256(BH * kKbImg);
    a.r_on = reinterpret_cast<float *>(base);
    a.kbar_out = gated ? fa.kbar : nullptr;
    a.kpre_out = gated ? fa.kpre_tiles : nullptr;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.CPS = (int)CPS; a.d = p.d; a.NB = (p.N + 63) / 64;
    a.num_tiles = (int)(BH * N * CPS);
    CUtensorMap mK, mV, mU;
    const unsigned long long rows = (unsigned long long)BH * p.L;
    if (!make_tmap_bf16_sw128(&mK, fa.k, rows, p.d, 128) || !make_tmap_bf16_sw128(&mV, fa.v, rows, p.d, 128))
        return cudaErrorInvalidValue;
    if (gated) {
        if (!make_tmap_bf16_sw128(&mU, fa.u, rows, p.d, 128)) return cudaErrorInvalidValue;
    } else {
        mU = mK;
    }
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    cudaError_t e;
    if (gated && (e = cudaMemsetAsync(a.kbar_img, 0, BH * kKbImg, s)) != cudaSuccess) return e;
    auto k1 = gated ? seg_state_tc<true, false> : seg_state_tc<false, false>;
    const size_t smem1 = t1_smem_bytes<false>();
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)) != cudaSuccess) return e;
    const int nseg = (int)(BH * N);
    k1<<<nseg < g_num_sms ? nseg : g_num_sms, kT1Threads, smem1, s>>>(mK, mV, mU, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    out->states_img = a.states_img;
    out->spre_img = a.spre_img;
    out->kbar_img = a.kbar_img;
    out->r_on = a.r_on;
    return cudaSuccess;
}

// The backward's gates from the state kernel's key-mean images and r_on (routed modes).
cudaError_t launch_bwd_gates_tc(const Problem &p, const void *u, const TcImages &img, float *gam, float *tok, cudaStream_t s)
{
    TcArgs a{};
    a.kbar_img = const_cast<uint8_t *>(img.kbar_img);
    a.r_on = const_cast<float *>(img.r_on);
    a.gam_out = gam;
    a.tok_out = tok;
    a.topk = p.topk;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.CPS = p.C / kCT; a.d = p.d; a.NB = (p.N + 63) / 64;
    CUtensorMap mU;
    if (!make_tmap_bf16_sw128(&mU, u, (unsigned long long)p.BH * p.L, p.d, 128)) return cudaErrorInvalidValue;
    auto k = p.mode == MC_SSC ? gate_tiles_tc<2> : gate_tiles_tc<1>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kRouterSmem);
    if (e != cudaSuccess) return e;
    const int gtiles = p.BH * (p.L / kCT);
    const int ggrid = gtiles < g_num_sms ? gtiles : g_num_sms;
    k<<<ggrid, kRouterThreads, kRouterSmem, s>>>(mU, a);
    return cudaGetLastError();
}

cudaError_t launch_state_tc_segments(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch,
                                     cudaStream_t s)
{
    return p.d == 64 ? launch_state_tc_segments64(p, fa, tb, scratch, s) : state_segments_impl<128>(p, fa, tb, scratch, s);
}

cudaError_t launch_readout_tc_segments(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch,
                                       cudaStream_t s)
{
    return p.d == 64 ? launch_readout_tc_segments64(p, fa, tb, scratch, s)
                     : readout_segments_impl<128>(p, fa, tb, scratch, s);
}

size_t tc_segments_scratch_bytes(const Problem &p, int NC, int nslots) { return segments_scratch_bytes(p, NC, nslots); }

// d = 64 runs the 64-wide instantiations, compiled in their own translation unit.
cudaError_t launch_forward_tc(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    return p.d == 64 ? launch_forward_tc64(p, fa, scratch, s) : forward_impl<128>(p, fa, scratch, s);
}

}  // namespace mc
