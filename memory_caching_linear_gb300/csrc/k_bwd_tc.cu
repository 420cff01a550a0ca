// k_bwd_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) kernels of the Memory Caching
// backward pass over a linear memory, for bf16 inputs on the shapes the forward's
// tensor-core path takes (d = 64 or 128, seg_len a multiple of 128, L a multiple of
// seg_len, N <= 64).
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//
// bwd_G_tc -- the gradient of every cached state ([MC-ja §3 after eq. 4b]: the cached
//   M^(i) is read by every token of the later segments with its gate g_{t,i}):
//     G_i = sum_{t in segments > i} g_{t,i} dy_t q_t^T        (d_v x d_k, fp32 accumulation,
//                                                              written as a bf16 operand image)
//   One CTA per (b,h, pair of cached segments), the pair with the most later tokens
//   first.  Per 128-token tile: the TMA brings dy and q (two 64-column
//   128-byte-swizzled panels each), the four worker warps scale their token's dy row
//   by the two gates in shared memory, and one thread issues D_i += (g_i o dy)^T q
//   for both states, alternating eight 128x128x16 MMAs each, with both operands read
//   MN-major from shared memory.
#include <cstdint>

#include "mc_internal.cuh"
#include "sm100.cuh"
#include "tensormap.cuh"

namespace mc {

// Set by a backward tensor-core kernel that abandoned its work after a bounded wait
// ran out; read and cleared by mc_check_device().
__device__ int g_bwd_abort;

namespace {

using namespace sm100;

constexpr int kGT = 128;             // tokens per tile
constexpr uint32_t kGTile = 32768;   // one 128 x 128 bf16 operand tile (two 16 KB panels)
// The G kernel streams 64-token tiles (two 8 KB panels per operand) so that four
// tile stages fit in shared memory: dy (scaled in place for the first segment), q,
// g o dy for the second segment, and both segments' gates.
constexpr int kG2 = 64;                    // tokens per G tile
constexpr uint32_t kG2Tile = 16384;        // one 64 x 128 bf16 operand tile (two 8 KB panels)
constexpr int kGStages = 2;   // per CTA; two CTAs share an SM
constexpr int kGThreads = 192;             // warp 0 TMA, warp 1 MMA issuer, warps 2-5 scale and drain
constexpr uint32_t kGStage = 3 * kG2Tile + 1024;
constexpr size_t kGSmem = kGStages * kGStage + 1024;

struct GArgs {
    const float *gam;  // [BH][N][L]: g_{t,i} of the cached segments (routed aggregations)
    uint8_t *G;        // [BH][N] x 32 KB: G_i as a bf16 operand image (rows = value dim, as a state image)
    int BH, L, C, N, d, mode, pairs;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

// One CTA per (b,h, pair of cached segments i0 = 2p, i1 = 2p + 1): every tile after
// segment i0 is loaded once and feeds both accumulators (the tiles of segment i1
// only the first).  Every CTA walks its tiles from the sequence's end backwards, so
// the pairs of a head that run at the same time read the same tiles (from L2).
__global__ void __launch_bounds__(kGThreads, 2)
    bwd_G_tc(const __grid_constant__ CUtensorMap mY, const __grid_constant__ CUtensorMap mQ, GArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t full[kGStages], scaled[kGStages], empty[kGStages], done;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int pr = (int)blockIdx.x / a.BH, bh = (int)blockIdx.x % a.BH;
    const int i0 = 2 * pr, i1 = 2 * pr + 1;
    const bool two = i1 < a.N - 1;  // segment N-1 has no later tokens
    const int t_begin = (i0 + 1) * a.C;
    const int ntiles = (a.L - t_begin) / kG2;
    const int split = a.C / kG2;  // tiles of segment i1: the second state starts after them
    const bool routed = a.mode == MC_GRM || a.mode == MC_SOUP || a.mode == MC_SSC;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int s = 0; s < kGStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&scaled[s], 128);
            mbar_init(&empty[s], 1);
        }
        mbar_init(&done, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tD = tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tensormap(&mY);
            prefetch_tensormap(&mQ);
            int issued = 0;
            for (int j = 0; j < ntiles; ++j) {
                const int s = j % kGStages;
                if (!mbar_wait(&empty[s], ((j / kGStages) & 1) ^ 1, &abort_flag)) break;
                uint8_t *st = sm + s * kGStage;
                const int jt = ntiles - 1 - j;  // the tile, from the end
                const int row = bh * a.L + t_begin + jt * kG2;
                const bool g0 = routed, g1 = routed && two && jt >= split;  // gates to bring along
                mbar_arrive_expect_tx(&full[s], 2 * kG2Tile + (g0 ? 256 : 0) + (g1 ? 256 : 0));
                tma_load_2d(st, &mY, 0, row, &full[s]);
                tma_load_2d(st + kG2Tile / 2, &mY, 64, row, &full[s]);
                tma_load_2d(st + kG2Tile, &mQ, 0, row, &full[s]);
                tma_load_2d(st + kG2Tile + kG2Tile / 2, &mQ, 64, row, &full[s]);
                const size_t goff = (size_t)t_begin + (size_t)jt * kG2;
                if (g0) bulk_load(st + 3 * kG2Tile, a.gam + ((size_t)bh * a.N + i0) * a.L + goff, 256, &full[s]);
                if (g1) bulk_load(st + 3 * kG2Tile + 512, a.gam + ((size_t)bh * a.N + i1) * a.L + goff, 256, &full[s]);
                issued = j + 1;
            }
            // leave no copy in flight
            int give_up = 0;
            for (int j = issued > kGStages ? issued - kGStages : 0; j < issued; ++j)
                mbar_wait_limit(&full[j % kGStages], (j / kGStages) & 1, &give_up, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idG = idesc_bf16(128, 128, true, true);  // A = (g o dy)^T, B = q: both MN-major
            bool ok = true;
            for (int j = 0; j < ntiles && ok; ++j) {
                const int s = j % kGStages;
                if (!(ok = mbar_wait(&scaled[s], (j / kGStages) & 1, &abort_flag))) break;
                tc_fence_after();
                const uint32_t y0 = smem_u32(sm + s * kGStage), q0 = y0 + kG2Tile, y1 = y0 + 2 * kG2Tile;
                const bool second = two && ntiles - 1 - j >= split;  // segment i1's tiles come last
#pragma unroll
                for (int kk = 0; kk < 4; ++kk) {  // 16 tokens per step: 16 rows of 128 bytes; the 64-column halves 8 KB apart
                    const uint64_t bq = make_desc_sw128(q0 + kk * 2048u, kG2Tile / 2, 1024);
                    mma_ss(tD, make_desc_sw128(y0 + kk * 2048u, kG2Tile / 2, 1024), bq, idG, (j | kk) != 0);
                    if (second)
                        mma_ss(tD + 128, make_desc_sw128(y1 + kk * 2048u, kG2Tile / 2, 1024), bq, idG, (j | kk) != 0);
                }
                mma_commit(&empty[s]);
            }
            // leave no MMA in flight; the drain waits for this
            mma_commit(&done);
        }
    } else {
        // ---------------------------------------------------------- workers: a thread scales one panel row
        const int q4 = warp & 3;
        const int r = 32 * q4 + lane;
        const int trow = r & 63, h = r >> 6;  // token row of the tile, 64-column panel
        for (int j = 0; j < ntiles; ++j) {
            const int s = j % kGStages;
            const int jt = ntiles - 1 - j;  // the tile, from the end
            const bool second = two && jt >= split;
            if (!mbar_wait(&full[s], (j / kGStages) & 1, &abort_flag)) break;
            // the gates came with the tile (routed); Residual 1, Mean 1 / (n(t) + 1)
            const float *gsm = reinterpret_cast<const float *>(sm + s * kGStage + 3 * kG2Tile);
            const float gc = a.mode == MC_MEAN ? 1.f / (float)((t_begin + jt * kG2) / a.C + 1) : 1.f;
            const float g0 = routed ? gsm[trow] : gc;
            const float g1 = routed ? (second ? gsm[128 + trow] : 0.f) : gc;
            const __nv_bfloat162 g02 = __float2bfloat162_rn(g0), g12 = __float2bfloat162_rn(g1);
            uint8_t *rowp = sm + s * kGStage + h * (kG2Tile / 2) + trow * 128;  // the row's 128 bytes of one panel
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                // every chunk of the row takes the same gate: start each row at its own chunk so
                // that the eight rows of a shared-memory phase hit eight different banks
                const int pc = (c + trow) & 7;
                uint4 *p = reinterpret_cast<uint4 *>(rowp + pc * 16);
                const uint4 x = *p;
                uint4 x0 = x, x1 = x;
                __nv_bfloat162 *e0 = reinterpret_cast<__nv_bfloat162 *>(&x0);
                __nv_bfloat162 *e1 = reinterpret_cast<__nv_bfloat162 *>(&x1);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    e0[k] = __hmul2(e0[k], g02);
                    e1[k] = __hmul2(e1[k], g12);
                }
                *p = x0;
                if (second) *reinterpret_cast<uint4 *>(rowp + 2 * kG2Tile + pc * 16) = x1;
            }
            fence_async_smem();  // the tensor core reads what these threads wrote
            mbar_arrive(&scaled[s]);
        }
        // drain: TMEM lane = value dim (row of G), thread = lane; G_i0 then G_i1 as bf16
        // images (128-byte swizzle: 16-byte chunk c of row r at chunk c ^ (r % 8); zero beyond d)
        const bool got = mbar_wait(&done, 0, &abort_flag);
        tc_fence_after();
        for (int which = 0; which < (two ? 2 : 1); ++which) {
            uint8_t *img = a.G + ((size_t)bh * a.N + (which ? i1 : i0)) * kGTile + r * 128;
            for (int c0 = 0; c0 < 128; c0 += 32) {
                uint32_t x[32];
                tmem_ld32(tD + 128 * which + ((uint32_t)(32 * q4) << 16) + c0, x);
                tmem_wait_ld();
                if (got) {
#pragma unroll
                    for (int q = 0; q < 4; ++q) {  // 8 columns = one 16-byte chunk
                        const int c8 = c0 / 8 + q, hh = c8 >> 3, cc = c8 & 7;
                        const uint4 v = make_uint4(
                            pack_bf16x2(__uint_as_float(x[8 * q]), __uint_as_float(x[8 * q + 1])),
                            pack_bf16x2(__uint_as_float(x[8 * q + 2]), __uint_as_float(x[8 * q + 3])),
                            pack_bf16x2(__uint_as_float(x[8 * q + 4]), __uint_as_float(x[8 * q + 5])),
                            pack_bf16x2(__uint_as_float(x[8 * q + 6]), __uint_as_float(x[8 * q + 7])));
                        *reinterpret_cast<uint4 *>(img + hh * 16384 + ((cc ^ (r & 7)) << 4)) = v;
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tD, 256);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_bwd_abort, 1);
}

// ============================================================================
// bwd_cached_tc -- per 128-token tile (b,h, segment n, chunk c) the reads of every
// memory the tile's tokens use, as the gradient needs them:
//   the online memory M_t = S_pre(c) + sum_{j in chunk, j <= t} v_j k_j^T (gate g_on):
//     dg_on_t  = dy_t . M_t q_t = q_t . (S_pre^T dy_t) + sum_{j<=t} (dy_t . v_j)(k_j . q_t)
//     dq_t    += g_on (S_pre^T dy_t + sum_{j<=t} k_j (v_j . dy_t))
//   every cached M^(i), i < n (gate g_{t,i}):
//     dg_{t,i} = q_t . (M^(i)^T dy_t),   dq_t += g_{t,i} M^(i)^T dy_t
// On the tensor cores: G1 = Q K^T and G2 = dY V^T (SS); P2 = g_on mask(G2) -> P2 K
// (TS), which starts the workers' dq; then for the prefix state and each cached state
// X: W = dY X (SS, the image read MN-major), whose row t is M^T dy_t: the workers take
// dg = q . W and, since the gate is a per-row scalar, dq += g W in fp32 registers
// (one product per state).  Every product lands in one of kCW rotating TMEM buffers.
// Persistent, one CTA per SM, tiles with the most cached segments first.  Warp 0
// loads Q and dY of the tile (TMA, resident while the tile runs) and streams K, V
// and one 32 KB image per state through a five-slot ring (K and V are read by the
// tile's first three products only); warp 1 issues; eight worker warps, two per TMEM
// lane quadrant: warp half h owns the token rows of its quadrant, the columns
// [64h, 64h+64) of q, W and dq, and the TMEM A columns [32h, 32h+32) of P2; the two
// halves' partial dots go to two dg buffers, which the route kernel adds.
// TMEM: W0 [0,128) | W1 [128,256) | W2 [256,384) | A0 [384,448) | A1 [448,512).
// ============================================================================
constexpr int kCRing = 5;
constexpr int kCW = 3;  // TMEM product buffers
constexpr int kCWorkers = 256;
constexpr int kCThreads = 64 + kCWorkers;
constexpr size_t kCSmem = 2 * kGTile + kCRing * kGTile + 1024;

struct CArgs {
    const uint8_t *images;  // [BH][N] x 32 KB state images
    const uint8_t *spre;    // [BH][N][CPS] x 32 KB prefix-state images (chunk c > 0)
    const float *gam;       // [BH][N][L] gates of the cached segments (routed aggregations)
    const float *tok;       // [BH][L][kBwdTokWords]: word 2 is the online gate (routed aggregations)
    float *dg;              // 2 x [BH][N][L] out: dy_t . M^(i) q_t, summed over each column half
    float *dgon;            // 2 x [BH][L] out: dy_t . M_t q_t, the same
    __nv_bfloat16 *dq;      // [BH][L][d] out: dq
    int BH, L, C, N, CPS, d, mode, num_tiles;
};

__global__ void __launch_bounds__(kCThreads, 1)
    bwd_cached_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                  const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mY, CArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sQ = sm, *sY = sm + kGTile, *ring = sm + 2 * kGTile;
    __shared__ uint64_t tile_full, tile_empty, ring_full[kCRing], ring_empty[kCRing];
    __shared__ uint64_t w_full[kCW], w_empty[kCW], a_full[2], a_empty[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int my_tiles = blockIdx.x < (unsigned)a.num_tiles ? (a.num_tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile = [&](int j, int &bh, int &n, int &c) {  // heaviest first: n = N-1 down to 0
        const int id = (int)blockIdx.x + j * (int)gridDim.x;
        const int per = a.BH * a.CPS;
        n = a.N - 1 - id / per;
        c = (id % per) / a.BH;
        bh = (id % per) % a.BH;
    };

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        mbar_init(&tile_full, 1);
        mbar_init(&tile_empty, 1 + kCWorkers);  // the tile's last MMA reading Q, dY + every worker has its rows
        for (int s = 0; s < kCRing; ++s) {
            mbar_init(&ring_full[s], 1);
            mbar_init(&ring_empty[s], 1);
        }
        for (int s = 0; s < kCW; ++s) {
            mbar_init(&w_full[s], 1);
            mbar_init(&w_empty[s], kCWorkers);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&a_full[s], kCWorkers);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(&fin, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tW0 = tb, tA0 = tb + 128 * kCW;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0 && my_tiles > 0) {
            prefetch_tensormap(&mQ);
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            prefetch_tensormap(&mY);
            uint32_t gr = 0;  // ring items
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                int bh, n, c;
                tile(j, bh, n, c);
                if (!(ok = mbar_wait(&tile_empty, (j & 1) ^ 1, &abort_flag))) break;
                const int row = bh * a.L + n * a.C + c * kGT;
                mbar_arrive_expect_tx(&tile_full, 2 * kGTile);
                tma_load_2d(sQ, &mQ, 0, row, &tile_full);
                tma_load_2d(sQ + 16384, &mQ, 64, row, &tile_full);
                tma_load_2d(sY, &mY, 0, row, &tile_full);
                tma_load_2d(sY + 16384, &mY, 64, row, &tile_full);
                // ring items: K, V, then the prefix state (chunk c > 0) and the cached states
                const int nimg = (c > 0 ? 1 : 0) + n;
                for (int m = -2; m < nimg && ok; ++m, ++gr) {
                    const int s = gr % kCRing;
                    if (!(ok = mbar_wait(&ring_empty[s], ((gr / kCRing) & 1) ^ 1, &abort_flag))) break;
                    mbar_arrive_expect_tx(&ring_full[s], kGTile);
                    uint8_t *dst = ring + s * kGTile;
                    if (m < 0) {
                        const CUtensorMap *map = m == -2 ? &mK : &mV;
                        tma_load_2d(dst, map, 0, row, &ring_full[s]);
                        tma_load_2d(dst + 16384, map, 64, row, &ring_full[s]);
                        continue;
                    }
                    const uint8_t *src = (c > 0 && m == 0)
                                             ? a.spre + (((size_t)bh * a.N + n) * a.CPS + c) * kGTile
                                             : a.images + ((size_t)bh * a.N + (m - (c > 0 ? 1 : 0))) * kGTile;
                    bulk_load(dst, src, kGTile, &ring_full[s]);
                }
            }
            // leave no copy in flight: the last use of every slot has landed
            int give_up = 0;
            for (uint32_t k = 0; k < (uint32_t)kCRing && k < gr; ++k) {
                const uint32_t u = gr - 1 - k;
                mbar_wait_limit(&ring_full[u % kCRing], (u / kCRing) & 1, &give_up, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && my_tiles > 0) {
            constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);  // both K-major
            constexpr uint32_t idKM = idesc_bf16(128, 128, false, true);   // B MN-major
            uint32_t gw = 0, ga = 0, gr = 0;
            bool ok = true;
            const uint32_t q0 = smem_u32(sQ), y0 = smem_u32(sY);
            const uint32_t r0 = smem_u32(ring);
            auto kmaj = [](int kk) { return (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32); };
            for (int j = 0; j < my_tiles && ok; ++j) {
                int bh, n, c;
                tile(j, bh, n, c);
                const int nimg = (c > 0 ? 1 : 0) + n;
                // K and V: the tile's first two ring items
                const uint32_t sk = gr % kCRing, sv = (gr + 1) % kCRing;
                const uint32_t k0 = r0 + sk * kGTile, v0 = r0 + sv * kGTile;
                if (!(ok = mbar_wait(&tile_full, j & 1, &abort_flag) &&
                           mbar_wait(&ring_full[sk], (gr / kCRing) & 1, &abort_flag) &&
                           mbar_wait(&ring_full[sv], ((gr + 1) / kCRing) & 1, &abort_flag)))
                    break;
                gr += 2;
                // G1 = Q K^T, G2 = dY V^T into the two W buffers
                const uint32_t w1 = gw % kCW, w2 = (gw + 1) % kCW;
                if (!(ok = mbar_wait(&w_empty[w1], ((gw / kCW) & 1) ^ 1, &abort_flag) &&
                           mbar_wait(&w_empty[w2], (((gw + 1) / kCW) & 1) ^ 1, &abort_flag)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tW0 + w1 * 128, make_desc_sw128(q0 + kmaj(kk), 0, 1024), make_desc_sw128(k0 + kmaj(kk), 0, 1024),
                           idKK, kk > 0);
                mma_commit(&w_full[w1]);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tW0 + w2 * 128, make_desc_sw128(y0 + kmaj(kk), 0, 1024), make_desc_sw128(v0 + kmaj(kk), 0, 1024),
                           idKK, kk > 0);
                mma_commit(&w_full[w2]);
                mma_commit(&ring_empty[sv]);  // V is spent
                gw += 2;
                // P2 K once the workers have written P2: the start of their dq
                const uint32_t w3 = gw % kCW;
                if (!(ok = mbar_wait(&a_full[ga % 2], (ga / 2) & 1, &abort_flag) &&
                           mbar_wait(&w_empty[w3], ((gw / kCW) & 1) ^ 1, &abort_flag)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tW0 + w3 * 128, tA0 + (ga % 2) * 64 + kk * 8, make_desc_sw128(k0 + kk * 2048u, 16384, 1024), idKM,
                           kk > 0);
                mma_commit(&w_full[w3]);
                mma_commit(&a_empty[ga % 2]);
                mma_commit(&ring_empty[sk]);  // K is spent
                ++gw;
                ++ga;
                if (nimg == 0) mma_commit(&tile_empty);
                for (int m = 0; m < nimg && ok; ++m, ++gw, ++gr) {
                    const uint32_t s = gr % kCRing, w = gw % kCW;
                    if (!(ok = mbar_wait(&ring_full[s], (gr / kCRing) & 1, &abort_flag) &&
                               mbar_wait(&w_empty[w], ((gw / kCW) & 1) ^ 1, &abort_flag)))
                        break;
                    tc_fence_after();
                    const uint32_t img = r0 + s * kGTile;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tW0 + w * 128, make_desc_sw128(y0 + kmaj(kk), 0, 1024),
                               make_desc_sw128(img + kk * 2048u, 16384, 1024), idKM, kk > 0);
                    mma_commit(&w_full[w]);
                    mma_commit(&ring_empty[s]);  // the image is spent
                    if (m == nimg - 1) mma_commit(&tile_empty);  // Q, K, V, dY are no longer read
                }
                if (!ok) break;
            }
            // leave no MMA in flight
            mma_commit(&fin);
            int give_up = 0;
            mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------- workers (thread = token row, column half)
        const int q4 = warp & 3, half = (warp - 2) >> 2;
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const bool routed = a.mode == MC_GRM || a.mode == MC_SOUP || a.mode == MC_SSC;
        const size_t hoff = (size_t)half * a.BH * a.L;  // this half's dg / dg_on buffer (dg: times N)
        uint32_t gw = 0, ga = 0;
        bool ok = true;
        for (int j = 0; j < my_tiles && ok; ++j) {
            int bh, n, c;
            tile(j, bh, n, c);
            const int nimg = (c > 0 ? 1 : 0) + n;
            const int t = n * a.C + c * kGT + row;  // token within the head
            if (!(ok = mbar_wait(&tile_full, j & 1, &abort_flag))) break;
            const float gon = routed ? __ldg(a.tok + ((size_t)bh * a.L + t) * kBwdTokWords + 2)
                                     : (a.mode == MC_MEAN ? 1.f / (float)(n + 1) : 1.f);
            // in-chunk online part over the half's key columns: dg_on += sum_{j<=t} G1 G2, P2 = g_on mask(G2)
            float dgon = 0.f;
            {
                const uint32_t w1 = gw % kCW, w2 = (gw + 1) % kCW;
                if (!(ok = mbar_wait(&w_full[w1], (gw / kCW) & 1, &abort_flag) &&
                           mbar_wait(&w_full[w2], ((gw + 1) / kCW) & 1, &abort_flag) &&
                           mbar_wait(&a_empty[ga % 2], ((ga / 2) & 1) ^ 1, &abort_flag)))
                    break;
                tc_fence_after();
#pragma unroll
                for (int mm = 0; mm < 4; ++mm) {  // 16 key columns at a time
                    const int m = 4 * half + mm;
                    uint32_t x1[16], x2[16], o[8];
                    tmem_ld16(tW0 + w1 * 128 + lane_base + 16 * m, x1);
                    tmem_ld16(tW0 + w2 * 128 + lane_base + 16 * m, x2);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; k += 2) {
                        const uint32_t col = 16 * m + k;
                        const float a0 = col <= row ? __uint_as_float(x2[k]) : 0.f;
                        const float a1 = col + 1 <= row ? __uint_as_float(x2[k + 1]) : 0.f;
                        dgon = fmaf(__uint_as_float(x1[k]), a0, dgon);
                        dgon = fmaf(__uint_as_float(x1[k + 1]), a1, dgon);
                        o[k / 2] = pack_bf16x2(gon * a0, gon * a1);
                    }
                    tmem_st8(tA0 + (ga % 2) * 64 + lane_base + 8 * m, o);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&w_empty[w1]);
                mbar_arrive(&w_empty[w2]);
                mbar_arrive(&a_full[ga % 2]);
                gw += 2;
                ++ga;
            }
            // the half's q columns come from the resident tile for every state (128-byte swizzle: chunk
            // c of row r at chunk c ^ (r % 8); 64 columns per 16 KB panel, the half's is panel `half`);
            // the tile is released after the last dot
            const uint8_t *qrow = sQ + half * 16384 + row * 128;
            if (nimg == 0) mbar_arrive(&tile_empty);
            // the prefix state (gate g_on) and the cached states (gate g_{t,i}): dg = q . W and
            // dq += g W over the half's 64 columns; the gates are fetched two states ahead
            const float *grow = routed ? a.gam + (size_t)bh * a.N * a.L + t : nullptr;
            float *dgrow = a.dg + hoff * a.N + (size_t)bh * a.N * a.L + t;
            const float gconst = a.mode == MC_MEAN ? 1.f / (float)(n + 1) : 1.f;
            const int i0 = c > 0 ? -1 : 0;  // state index of item m is i0 + m (-1: the prefix state)
            auto gate = [&](int m) {
                const int i = i0 + m;
                return i < 0 ? gon : (routed ? __ldg(grow + (size_t)i * a.L) : gconst);
            };
            float g_cur = nimg > 0 ? gate(0) : 0.f, g_nxt = nimg > 1 ? gate(1) : 0.f;
            // dq starts from the in-chunk product P2 K (the half's 64 columns)
            float dqa[64];
            {
                const uint32_t w = gw % kCW;
                if (!(ok = mbar_wait(&w_full[w], (gw / kCW) & 1, &abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t x[32];
                    tmem_ld32(tW0 + w * 128 + lane_base + 64 * half + 32 * h, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 32; ++k) dqa[32 * h + k] = __uint_as_float(x[k]);
                }
                tc_fence_before();
                mbar_arrive(&w_empty[w]);
                ++gw;
            }
            for (int m = 0; m < nimg && ok; ++m) {
                const float g = g_cur;
                g_cur = g_nxt;
                g_nxt = m + 2 < nimg ? gate(m + 2) : 0.f;
                const uint32_t w = gw % kCW;
                if (!(ok = mbar_wait(&w_full[w], (gw / kCW) & 1, &abort_flag))) break;
                tc_fence_after();
                float d0 = 0.f, d1 = 0.f;
#pragma unroll
                for (int h = 0; h < 2; ++h) {  // the half's 64 columns, 32 per wait
                    uint32_t x[32], qp[16];
                    tmem_ld32(tW0 + w * 128 + lane_base + 64 * half + 32 * h, x);
#pragma unroll
                    for (int c4 = 0; c4 < 4; ++c4) {
                        const int cc = 4 * h + c4;
                        const uint4 xq = *reinterpret_cast<const uint4 *>(qrow + ((cc ^ (row & 7)) << 4));
                        qp[4 * c4] = xq.x; qp[4 * c4 + 1] = xq.y; qp[4 * c4 + 2] = xq.z; qp[4 * c4 + 3] = xq.w;
                    }
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; ++k) {
                        const uint32_t qq = qp[k];
                        d0 = fmaf(__uint_as_float(qq << 16), __uint_as_float(x[2 * k]), d0);
                        d1 = fmaf(__uint_as_float(qq & 0xffff0000u), __uint_as_float(x[2 * k + 1]), d1);
                    }
#pragma unroll
                    for (int k = 0; k < 32; ++k) dqa[32 * h + k] = fmaf(g, __uint_as_float(x[k]), dqa[32 * h + k]);
                }
                tc_fence_before();
                mbar_arrive(&w_empty[w]);
                if (m == nimg - 1) mbar_arrive(&tile_empty);  // q is read for the last time
                ++gw;
                if (i0 + m < 0) dgon += d0 + d1;
                else dgrow[(size_t)(i0 + m) * a.L] = d0 + d1;
            }
            if (!ok) break;
            a.dgon[hoff + (size_t)bh * a.L + t] = dgon;
            // the half's 64 columns of dq
            __nv_bfloat16 *dqrow = a.dq + ((size_t)bh * a.L + t) * a.d;
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                const int m = 2 * half + mm;
                if (32 * m < a.d) {
#pragma unroll
                    for (int k = 0; k < 32; k += 8)
                        *reinterpret_cast<uint4 *>(dqrow + 32 * m + k) = make_uint4(
                            pack_bf16x2(dqa[32 * mm + k], dqa[32 * mm + k + 1]), pack_bf16x2(dqa[32 * mm + k + 2], dqa[32 * mm + k + 3]),
                            pack_bf16x2(dqa[32 * mm + k + 4], dqa[32 * mm + k + 5]), pack_bf16x2(dqa[32 * mm + k + 6], dqa[32 * mm + k + 7]));
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_bwd_abort, 1);
}

// ============================================================================
// bwd_kv_tc -- dk and dv of one 128-token chunk c of segment n (tokens j), from the
// cached state's gradient G_n and the online memory's reads in the segment (tokens
// t >= j, gate g_on(t)):
//   dv_j = G_n k_j + sum_{t >= j in n} g_on(t) (k_j . q_t) dy_t
//   dk_j = G_n^T v_j + sum_{t >= j in n} g_on(t) (v_j . dy_t) q_t
//          + sum_{t >= j in n} w_t u_t + dkbar_n / |n|      (w_t = dr_on(t) / cnt_t)
// On the tensor cores: D_v = K G^T, D_k = V G (the G image); then for every 64-token
// sub-chunk s from chunk c to the segment's end X = K Q'^T, Y = V dY'^T (SS, N = 64);
// the workers turn them into P3 = g_on mask(X), P4 = g_on mask(Y), P5 = w mask
// (mask: t >= j) and D_v += P3 dY', D_k += P4 Q' + P5 U' (TS, the sub-chunk tiles
// read MN-major).  X and Y are double-buffered, so the tensor cores compute the
// next sub-chunk's products while the workers mask the current one; the sub-chunk
// tiles come through a three-slot ring with the tokens' online gates and weights w, after
// the G image of the segment (the first item of a chunk, in a slot of its own).
// Eight worker warps, two per TMEM lane quadrant: warp half h takes the tokens
// [32h, 32h+32) of a sub-chunk, i.e. the 32 columns [32h, 32h+32) of X and of Y, and
// writes its P blocks into them (P3 / P4 into the first 16, P5 into the next 16 of Y).
// Persistent, one CTA per SM.  A unit of work is a pair of chunks (c, CPS-1-c) of one
// segment, so every unit streams the same number of sub-chunks, and the units of a
// segment run side by side (its q, dy, u come from HBM about once).
// TMEM: D_v [0,128) | D_k [128,256) | X0 Y0 [256,384) | X1 Y1 [384,512) (64 columns each).
// ============================================================================
constexpr int kVWorkers = 256;
constexpr int kVThreads = 64 + kVWorkers;                     // warp 0 TMA, warp 1 MMA issuer, 8 workers
constexpr uint32_t kVStage = 3 * kG2Tile + 1024;              // Q', dY', U' of a 64-token sub-chunk; gates, w
constexpr int kVRing = 3;
constexpr size_t kVSmem = 2 * kGTile + kVRing * kVStage + 1024;  // K, V; the ring

struct VArgs {
    const uint8_t *G;      // [BH][N] x 32 KB G images (segments < N-1)
    const float *gw;       // [2][BH][L]: the online gate, then the pooled-key weight w, per token
    const float *dkbar;    // [BH][N][d]
    void *dk, *dv;         // bf16 [BH][L][d] out
    int BH, L, C, N, CPS, d, routed;
    int UP;                // units per segment: ceil(CPS / 2)
    int num_units;         // BH * N * UP
};

// The CTA's k-th tile: unit blockIdx + (k / 2) * grid, its first (heavier) or second chunk.
// Returns false past the last unit; skips the repeated middle chunk of an odd CPS.
struct VTiles {
    int k = 0, h = 0;
    __device__ bool next(const VArgs &a, int &bh, int &n, int &c)
    {
        for (;;) {
            const int u = (int)blockIdx.x + k * (int)gridDim.x;
            if (u >= a.num_units) return false;
            const int p = u % a.UP, seg = u / a.UP;
            bh = seg % a.BH;
            n = seg / a.BH;
            c = h ? a.CPS - 1 - p : p;
            const bool valid = !(h && c == p);
            if (h) {
                ++k;
                h = 0;
            } else {
                h = 1;
            }
            if (valid) return true;
        }
    }
};

__global__ void __launch_bounds__(kVThreads, 1)
    bwd_kv_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
              const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mY,
              const __grid_constant__ CUtensorMap mU, VArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    // K, V of the chunk; a ring of kVRing slots, each the G image of a chunk's segment
    // (the first item of a chunk that has one) or a sub-chunk's Q', dY', U', gates and w
    uint8_t *sK = sm, *sV = sm + kGTile, *sR = sm + 2 * kGTile;
    __shared__ uint64_t kv_full, kv_empty, r_full[kVRing], r_empty[kVRing], xy_full[2], p_full[2], d_full, d_empty, fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        mbar_init(&kv_full, 1);
        mbar_init(&kv_empty, 1);
        for (int r = 0; r < kVRing; ++r) {
            mbar_init(&r_full[r], 1);
            mbar_init(&r_empty[r], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&xy_full[b], 1);
            mbar_init(&p_full[b], kVWorkers);
        }
        mbar_init(&d_full, 1);
        mbar_init(&d_empty, kVWorkers);
        mbar_init(&fin, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tDv = tb, tDk = tb + 128, tXY = tb + 256;  // X_b = tXY + 128 b, Y_b = X_b + 64

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        if (lane == 0) {
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            prefetch_tensormap(&mQ);
            prefetch_tensormap(&mY);
            if (a.routed) prefetch_tensormap(&mU);
            uint32_t rc = 0, jt = 0;  // ring items, chunks
            bool ok = true;
            VTiles it;
            int bh, n, c;
            while (ok && it.next(a, bh, n, c)) {
                const bool hasG = n < a.N - 1;
                if (!(ok = mbar_wait(&kv_empty, (jt & 1) ^ 1, &abort_flag))) break;
                const int row = bh * a.L + n * a.C + c * kGT;
                mbar_arrive_expect_tx(&kv_full, 2 * kGTile);
                tma_load_2d(sK, &mK, 0, row, &kv_full);
                tma_load_2d(sK + 16384, &mK, 64, row, &kv_full);
                tma_load_2d(sV, &mV, 0, row, &kv_full);
                tma_load_2d(sV + 16384, &mV, 64, row, &kv_full);
                const int S = 2 * (a.CPS - c);
                for (int s = hasG ? -1 : 0; s < S; ++s, ++rc) {
                    const uint32_t r = rc % kVRing;
                    if (!(ok = mbar_wait(&r_empty[r], ((rc / kVRing) & 1) ^ 1, &abort_flag))) break;
                    uint8_t *st = sR + r * kVStage;
                    if (s < 0) {
                        mbar_arrive_expect_tx(&r_full[r], kGTile);
                        bulk_load(st, a.G + ((size_t)bh * a.N + n) * kGTile, kGTile, &r_full[r]);
                        continue;
                    }
                    const int r2 = row + kG2 * s;
                    mbar_arrive_expect_tx(&r_full[r], (a.routed ? 3 : 2) * kG2Tile + (a.routed ? 512 : 256));
                    const float *gw = a.gw + (size_t)r2;  // the sub-chunk's online gates; w BH * L further
                    bulk_load(st + 3 * kG2Tile, gw, 256, &r_full[r]);
                    if (a.routed) bulk_load(st + 3 * kG2Tile + 256, gw + (size_t)a.BH * a.L, 256, &r_full[r]);
                    tma_load_2d(st, &mQ, 0, r2, &r_full[r]);
                    tma_load_2d(st + kG2Tile / 2, &mQ, 64, r2, &r_full[r]);
                    tma_load_2d(st + kG2Tile, &mY, 0, r2, &r_full[r]);
                    tma_load_2d(st + kG2Tile + kG2Tile / 2, &mY, 64, r2, &r_full[r]);
                    if (a.routed) {
                        tma_load_2d(st + 2 * kG2Tile, &mU, 0, r2, &r_full[r]);
                        tma_load_2d(st + 2 * kG2Tile + kG2Tile / 2, &mU, 64, r2, &r_full[r]);
                    }
                }
                ++jt;
            }
            // leave no copy in flight
            int give_up = 0;
            for (uint32_t q = rc > kVRing ? rc - kVRing : 0; q < rc; ++q)
                mbar_wait_limit(&r_full[q % kVRing], (q / kVRing) & 1, &give_up, kWaitLimitNs);
            if (jt > 0) mbar_wait_limit(&kv_full, (jt - 1) & 1, &give_up, kWaitLimitNs);
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idKK = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idKM = idesc_bf16(128, 128, false, true);
            constexpr uint32_t idXY = idesc_bf16(128, kG2, false, false);
            auto kmaj = [](int kk) { return (uint32_t)((kk >> 2) * 16384 + (kk & 3) * 32); };      // 128-row tile
            auto kmaj64 = [](int kk) { return (uint32_t)((kk >> 2) * 8192 + (kk & 3) * 32); };     // 64-row tile
            const uint32_t k0 = smem_u32(sK), v0 = smem_u32(sV), r0 = smem_u32(sR);
            auto slot = [&](uint32_t q) { return r0 + (q % kVRing) * kVStage; };
            // X_x = K Q'^T, Y_x = V dY'^T of the sub-chunk in ring item q, into TMEM buffer x % 2
            auto issue_xy = [&](uint32_t q, uint32_t x) {
                const uint32_t b = x & 1, st = slot(q);
                const uint32_t tX = tXY + 128 * b, tY = tX + 64;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tX, make_desc_sw128(k0 + kmaj(kk), 0, 1024), make_desc_sw128(st + kmaj64(kk), 0, 1024),
                           idXY, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tY, make_desc_sw128(v0 + kmaj(kk), 0, 1024),
                           make_desc_sw128(st + kG2Tile + kmaj64(kk), 0, 1024), idXY, kk > 0);
                mma_commit(&xy_full[b]);
            };
            uint32_t rc = 0, pc = 0, jt = 0;  // ring items, sub-chunks, chunks
            bool ok = true;
            VTiles it;
            int bh, n, c;
            while (ok && it.next(a, bh, n, c)) {
                const bool hasG = n < a.N - 1;
                const int S = 2 * (a.CPS - c);
                const uint32_t q0 = rc + (hasG ? 1 : 0);  // ring item of the first sub-chunk
                if (!(ok = mbar_wait(&kv_full, jt & 1, &abort_flag) &&
                           mbar_wait(&r_full[q0 % kVRing], (q0 / kVRing) & 1, &abort_flag)))
                    break;
                tc_fence_after();
                issue_xy(q0, pc);
                // the previous chunk's drain has read D
                if (!(ok = mbar_wait(&d_empty, (jt & 1) ^ 1, &abort_flag))) break;
                tc_fence_after();
                if (hasG) {
                    if (!(ok = mbar_wait(&r_full[rc % kVRing], (rc / kVRing) & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t g0 = slot(rc);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // D_v = K G^T: B = G image K-major (rows = value dim)
                        mma_ss(tDv, make_desc_sw128(k0 + kmaj(kk), 0, 1024), make_desc_sw128(g0 + kmaj(kk), 0, 1024),
                               idKK, kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)  // D_k = V G: B = G image MN-major
                        mma_ss(tDk, make_desc_sw128(v0 + kmaj(kk), 0, 1024), make_desc_sw128(g0 + kk * 2048u, 16384, 1024),
                               idKM, kk > 0);
                    mma_commit(&r_empty[rc % kVRing]);
                }
                for (int s = 0; s < S && ok; ++s) {
                    const uint32_t q = q0 + s, x = pc + s, b = x & 1;
                    if (s + 1 < S) {  // the next sub-chunk's products while the workers mask this one
                        if (!(ok = mbar_wait(&r_full[(q + 1) % kVRing], ((q + 1) / kVRing) & 1, &abort_flag))) break;
                        tc_fence_after();
                        issue_xy(q + 1, x + 1);
                        if (s + 2 == S) mma_commit(&kv_empty);  // K and V are read for the last time
                    }
                    if (!(ok = mbar_wait(&p_full[b], (x >> 1) & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t st = slot(q);
                    const uint32_t tX = tXY + 128 * b, tY = tX + 64;
                    const bool first = !hasG && s == 0;
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // D_v += P3 dY' (tokens 16 kk.. of P at 32 (kk/2) + 8 (kk%2))
                        mma_ts(tDv, tX + 32 * (kk >> 1) + 8 * (kk & 1),
                               make_desc_sw128(st + kG2Tile + kk * 2048u, kG2Tile / 2, 1024), idKM, !first || kk > 0);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)  // D_k += P4 Q'
                        mma_ts(tDk, tY + 32 * (kk >> 1) + 8 * (kk & 1), make_desc_sw128(st + kk * 2048u, kG2Tile / 2, 1024),
                               idKM, !first || kk > 0);
                    if (a.routed) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk)  // D_k += P5 U' (P5 16 columns after P4)
                            mma_ts(tDk, tY + 32 * (kk >> 1) + 16 + 8 * (kk & 1),
                                   make_desc_sw128(st + 2 * kG2Tile + kk * 2048u, kG2Tile / 2, 1024), idKM, 1);
                    }
                    mma_commit(&r_empty[q % kVRing]);
                }
                if (!ok) break;
                mma_commit(&d_full);
                rc = q0 + S;
                pc += S;
                ++jt;
            }
            // leave no MMA in flight
            mma_commit(&fin);
            int give_up = 0;
            mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------- workers (thread = row j of chunk c)
        const int q4 = warp & 3, half = (warp - 2) >> 2;  // lane quadrant; tokens [32 half, 32 half + 32)
        const int row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t rc = 0, pc = 0, jt = 0;  // ring items, sub-chunks, chunks
        bool ok = true;
        VTiles it;
        int bh, n, c;
        while (ok && it.next(a, bh, n, c)) {
            const int S = 2 * (a.CPS - c);
            const uint32_t q0 = rc + (n < a.N - 1 ? 1 : 0);
            const size_t tok_c = (size_t)bh * a.L + n * a.C + c * kGT;  // the chunk's first token
            for (int s = 0; s < S && ok; ++s) {
                const uint32_t q = q0 + s, x = pc + s, b = x & 1;
                // the item's gates came by TMA (this thread waits for them itself), X and Y from the MMA
                if (!(ok = mbar_wait(&r_full[q % kVRing], (q / kVRing) & 1, &abort_flag) &&
                           mbar_wait(&xy_full[b], (x >> 1) & 1, &abort_flag)))
                    break;
                tc_fence_after();
                const float *gsm = reinterpret_cast<const float *>(sR + (q % kVRing) * kVStage + 3 * kG2Tile) + 32 * half;
                const float *wsm = gsm + 64;
                const uint32_t tX = tXY + 128 * b + lane_base + 32 * half, tY = tX + 64;
                const int t_off = kG2 * s + 32 * half - row;  // token t of the half is kept when t + t_off >= 0
                const bool diag = t_off < 0;                  // some token of the half lies before row j
#pragma unroll
                for (int m = 0; m < 2; ++m) {  // 16 token columns at a time
                    uint32_t x[16], y[16], o3[8], o4[8];
                    tmem_ld16(tX + 16 * m, x);
                    tmem_ld16(tY + 16 * m, y);
                    float g[16];
#pragma unroll
                    for (int k4 = 0; k4 < 4; ++k4) {
                        const float4 v = *reinterpret_cast<const float4 *>(gsm + 16 * m + 4 * k4);
                        g[4 * k4] = v.x; g[4 * k4 + 1] = v.y; g[4 * k4 + 2] = v.z; g[4 * k4 + 3] = v.w;
                    }
                    if (diag)
#pragma unroll
                        for (int k = 0; k < 16; ++k)
                            if (16 * m + k + t_off < 0) g[k] = 0.f;
                    tmem_wait_ld();
#pragma unroll
                    for (int k = 0; k < 16; k += 2) {
                        o3[k / 2] = pack_bf16x2(g[k] * __uint_as_float(x[k]), g[k + 1] * __uint_as_float(x[k + 1]));
                        o4[k / 2] = pack_bf16x2(g[k] * __uint_as_float(y[k]), g[k + 1] * __uint_as_float(y[k + 1]));
                    }
                    tmem_st8(tX + 8 * m, o3);
                    tmem_st8(tY + 8 * m, o4);
                }
                if (a.routed) {  // P5 = w mask, written after every read of the half's Y columns
#pragma unroll
                    for (int m = 0; m < 2; ++m) {
                        float w[16];
#pragma unroll
                        for (int k4 = 0; k4 < 4; ++k4) {
                            const float4 v = *reinterpret_cast<const float4 *>(wsm + 16 * m + 4 * k4);
                            w[4 * k4] = v.x; w[4 * k4 + 1] = v.y; w[4 * k4 + 2] = v.z; w[4 * k4 + 3] = v.w;
                        }
                        uint32_t o5[8];
#pragma unroll
                        for (int k = 0; k < 16; k += 2) {
                            const float w0 = 16 * m + k + t_off >= 0 ? w[k] : 0.f;
                            const float w1 = 16 * m + k + 1 + t_off >= 0 ? w[k + 1] : 0.f;
                            o5[k / 2] = pack_bf16x2(w0, w1);
                        }
                        tmem_st8(tY + 16 + 8 * m, o5);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full[b]);
            }
            if (!ok) break;
            // drain: dv = D_v, dk = D_k + dkbar_n / |n|; the half's 64 columns
            if (!(ok = mbar_wait(&d_full, jt & 1, &abort_flag))) break;
            tc_fence_after();
            const size_t tok = tok_c + row;
            __nv_bfloat16 *dvo = static_cast<__nv_bfloat16 *>(a.dv) + tok * a.d;
            __nv_bfloat16 *dko = static_cast<__nv_bfloat16 *>(a.dk) + tok * a.d;
            const float *rho = a.dkbar + ((size_t)bh * a.N + n) * a.d;
            const float inv_len = 1.f / (float)a.C;
#pragma unroll
            for (int mm = 0; mm < 2; ++mm) {
                const int m = 2 * half + mm;
                uint32_t xv[32], xk[32];
                tmem_ld32(tDv + lane_base + 32 * m, xv);
                tmem_ld32(tDk + lane_base + 32 * m, xk);
                tmem_wait_ld();
                if (32 * m < a.d) {
#pragma unroll
                    for (int k = 0; k < 32; k += 8) {
                        uint4 ov, ok4;
                        uint32_t *pv = reinterpret_cast<uint32_t *>(&ov), *pk = reinterpret_cast<uint32_t *>(&ok4);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int col = 32 * m + k + 2 * e;
                            pv[e] = pack_bf16x2(__uint_as_float(xv[k + 2 * e]), __uint_as_float(xv[k + 2 * e + 1]));
                            const float r0 = a.routed ? __ldg(rho + col) * inv_len : 0.f;
                            const float r1 = a.routed ? __ldg(rho + col + 1) * inv_len : 0.f;
                            pk[e] = pack_bf16x2(__uint_as_float(xk[k + 2 * e]) + r0, __uint_as_float(xk[k + 2 * e + 1]) + r1);
                        }
                        *reinterpret_cast<uint4 *>(dvo + 32 * m + k) = ov;
                        *reinterpret_cast<uint4 *>(dko + 32 * m + k) = ok4;
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&d_empty);
            rc = q0 + S;
            pc += S;
            ++jt;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_bwd_abort, 1);
}

}  // namespace

bool bwd_tc_supported(const Problem &p)
{
    return p.bf16 && (p.d == 128 || p.d == 64) && p.C % kGT == 0 && p.L % p.C == 0 && p.N <= 64;
}

cudaError_t launch_bwd_G_tc(const Problem &p, const void *dy, const void *q, const float *gam, uint8_t *G, cudaStream_t s)
{
    if (p.N < 2) return cudaSuccess;
    CUtensorMap mY, mQ;
    const unsigned long long rows = (unsigned long long)p.BH * p.L;
    // a 64-wide tensor reads its second panel out of bounds: the TMA fills zeros
    if (!make_tmap_bf16_sw128(&mY, dy, rows, p.d, kG2) || !make_tmap_bf16_sw128(&mQ, q, rows, p.d, kG2))
        return cudaErrorInvalidValue;
    GArgs a{};
    a.gam = gam;
    a.G = G;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.d = p.d; a.mode = p.mode;
    a.pairs = p.N / 2;  // pairs of the cached segments 0 .. N-2
    cudaError_t e = cudaFuncSetAttribute(bwd_G_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (e != cudaSuccess) return e;
    bwd_G_tc<<<(unsigned)(p.BH * a.pairs), kGThreads, kGSmem, s>>>(mY, mQ, a);
    return cudaGetLastError();
}

// ============================================================================
// bwd_dkbar_tc -- the key-mean gradients ([MC-ja §3.1 eq. 10]: kbar_i enters the score
//   <u_t, kbar_i> of every later token):  dkbar_i = sum_t dr_{t,i} u_t, as
//     D[c][i] += sum_{t in tile} u_t[c] dr_{t,i}        (fp32 in tensor memory)
//   with A = the tile's u (MN-major: M = the head dimension, K = 128 tokens) and B = the
//   tile's dr rows (K-major: N = the tile's cached segments rounded up to 16, K = tokens),
//   dr as two bf16 terms hi + lo (16 bits; u is exact in bf16).  Persistent, one CTA per SM
//   over contiguous ranges of 128-token tiles (those of a head's first segment have no
//   cached segment and are skipped); the accumulator starts from zero for each head and is
//   added to dkbar with fp32 atomics when the CTA leaves the head.
// ============================================================================
constexpr int kDThreads = 192;                       // warp 0 TMA, warp 1 MMA issuer, warps 2-5 drain
constexpr int kDStages = 3;
constexpr uint32_t kDPlane = 16384;                  // 64 segment rows x 128 tokens of dr: two 8 KB panels
constexpr uint32_t kDStage = kGTile + 2 * kDPlane;   // u tile, dr hi, dr lo
constexpr size_t kDSmem = kDStages * kDStage + 1024;

struct DkArgs {
    float *dkbar;  // [BH][N][d], accumulated
    int BH, L, C, N, Np, d;
};

__global__ void __launch_bounds__(kDThreads, 1)
    bwd_dkbar_tc(const __grid_constant__ CUtensorMap mU, const __grid_constant__ CUtensorMap mHi,
                 const __grid_constant__ CUtensorMap mLo, DkArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t full[kDStages], empty[kDStages], acc_full, acc_ready, fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int TPH = a.L / kGT;  // tiles per head
    const int total = a.BH * TPH;
    const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int first = (int)blockIdx.x * per, last = min(total, first + per);
    auto seg_of = [&](int it) { return (it % TPH) * kGT / a.C; };  // cached segments of the tile's tokens
    // a head's first tiles (segment 0) do nothing: the working tiles of a head are contiguous,
    // so a run of one head ends at the range's end or where the head changes
    auto run_ends = [&](int it) { return it + 1 >= last || (it + 1) / TPH != it / TPH; };
    if (warp == 0) {
        tmem_alloc(&tmem_base, 64);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int i = 0; i < kDStages; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], 1);
        }
        mbar_init(&acc_full, 1);
        mbar_init(&acc_ready, 128);
        mbar_init(&fin, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tD = tmem_base;
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mU);
            prefetch_tensormap(&mHi);
            prefetch_tensormap(&mLo);
            uint32_t q = 0;
            for (int it = first; it < last; ++it) {
                if (seg_of(it) == 0) continue;
                const int bh = it / TPH, t0 = (it % TPH) * kGT;
                const int s = q % kDStages;
                if (!mbar_wait(&empty[s], ((q / kDStages) & 1) ^ 1, &abort_flag)) break;
                uint8_t *st = sm + s * kDStage;
                mbar_arrive_expect_tx(&full[s], kDStage);
                tma_load_2d(st, &mU, 0, bh * a.L + t0, &full[s]);
                tma_load_2d(st + 16384, &mU, 64, bh * a.L + t0, &full[s]);
                for (int h = 0; h < 2; ++h) {
                    tma_load_2d(st + kGTile + 8192 * h, &mHi, t0 + 64 * h, bh * a.Np, &full[s]);
                    tma_load_2d(st + kGTile + kDPlane + 8192 * h, &mLo, t0 + 64 * h, bh * a.Np, &full[s]);
                }
                ++q;
            }
            int give_up = 0;  // leave no copy in flight
            for (uint32_t i = 0; i < (uint32_t)kDStages && i < q; ++i) {
                const uint32_t u = q - 1 - i;
                mbar_wait_limit(&full[u % kDStages], (u / kDStages) & 1, &give_up, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            uint32_t q = 0, runs = 0;
            bool ok = true, fresh = true, issued = false;
            for (int it = first; it < last && ok; ++it) {
                const int n = seg_of(it);
                if (n == 0) continue;
                if (fresh) {  // the workers have zeroed the accumulator for this head
                    if (!(ok = mbar_wait(&acc_ready, runs & 1, &abort_flag))) break;
                    fresh = false;
                }
                const int s = q % kDStages;
                if (!(ok = mbar_wait(&full[s], (q / kDStages) & 1, &abort_flag))) break;
                tc_fence_after();
                const uint32_t sb = smem_u32(sm + s * kDStage);
                const int nt = (n + 15) & ~15;  // the MMA's N: the tile's cached segments, whole 16s
                const uint32_t id = idesc_bf16(128, nt, true, false);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint64_t du = make_desc_sw128(sb + kk * 2048u, 16384, 1024);  // MN-major u
#pragma unroll
                    for (int pl = 0; pl < 2; ++pl) {
                        const uint64_t dr = make_desc_sw128(sb + kGTile + pl * kDPlane + (kk >> 2) * 8192u + (kk & 3) * 32u, 0, 1024);  // K-major, 64 rows
                        mma_ss(tD, du, dr, id, 1);
                    }
                }
                issued = true;
                mma_commit(&empty[s]);
                ++q;
                if (run_ends(it)) {
                    mma_commit(&acc_full);
                    ++runs;
                    fresh = true;
                }
            }
            if (issued) {
                mma_commit(&fin);
                int give_up = 0;
                mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
            }
        }
    } else {
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;  // TMEM lane = the head dimension c
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t runs = 0;
        bool ok = true, fresh = true;
        for (int it = first; it < last && ok; ++it) {
            const int n = seg_of(it);
            if (n == 0) continue;
            if (fresh) {  // a new head: the accumulator starts from zero
                uint32_t z[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) z[i] = 0u;
#pragma unroll
                for (int c16 = 0; c16 < 4; ++c16) tmem_st16(tD + lane_base + 16 * c16, z);
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&acc_ready);
                fresh = false;
            }
            if (!run_ends(it)) continue;
            if (!(ok = mbar_wait(&acc_full, runs & 1, &abort_flag))) break;
            tc_fence_after();
            float v[64];
#pragma unroll
            for (int c16 = 0; c16 < 4; ++c16) tmem_ld16f(tD + lane_base + 16 * c16, v + 16 * c16);
            tmem_wait_ld();
            tc_fence_before();
            const int bh = it / TPH;
            if ((int)row < a.d) {
                float *dk = a.dkbar + (size_t)bh * a.N * a.d + row;
                for (int i = 0; i < a.N && i < 64; ++i)
                    if (v[i] != 0.f) atomicAdd(dk + (size_t)i * a.d, v[i]);
            }
            ++runs;
            fresh = true;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tD, 64);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_bwd_abort, 1);
}

cudaError_t launch_bwd_dkbar_tc(const Problem &p, const void *u, const __nv_bfloat16 *dr_hi,
                                const __nv_bfloat16 *dr_lo, int Np, float *dkbar, cudaStream_t s)
{
    if (p.N < 2 || Np > 64 || p.L % kGT != 0) return p.N < 2 ? cudaSuccess : cudaErrorInvalidValue;
    CUtensorMap mU, mHi, mLo;
    const unsigned long long rows = (unsigned long long)p.BH * p.L;
    if (!make_tmap_bf16_sw128(&mU, u, rows, p.d, 128) ||
        !make_tmap_bf16(&mHi, dr_hi, (unsigned long long)p.BH * Np, p.L, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_bf16(&mLo, dr_lo, (unsigned long long)p.BH * Np, p.L, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    DkArgs a{};
    a.dkbar = dkbar;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.Np = Np; a.d = p.d;
    cudaError_t e = cudaFuncSetAttribute(bwd_dkbar_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kDSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0) sms = 148;
    const int total = p.BH * (p.L / kGT);
    bwd_dkbar_tc<<<total < sms ? total : sms, kDThreads, kDSmem, s>>>(mU, mHi, mLo, a);
    return cudaGetLastError();
}

cudaError_t take_bwd_abort(int *was_set)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_bwd_abort, sizeof(int));
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        v = 0;
        e = cudaMemcpyToSymbol(g_bwd_abort, &v, sizeof(int));
    }
    return e;
}

}  // namespace mc

namespace mc {

size_t bwd_cached_scratch_bytes(const Problem &p)
{
    const size_t BH = p.BH, N = p.N, L = p.L;
    auto pad = [](size_t x) { return (x + 255) & ~(size_t)255; };
    return pad(8 * BH * N * L) + pad(8 * BH * L);  // dg and dg_on, one buffer per column half
}

cudaError_t launch_bwd_cached_tc(const Problem &p, const void *q, const void *k, const void *v, const void *dy,
                                 const TcImages &img, const float *gam, const float *tok, void *dq, void *scratch,
                                 float **dg_out, float **dgon_out, cudaStream_t s)
{
    const size_t BH = p.BH, N = p.N, L = p.L;
    auto pad = [](size_t x) { return (x + 255) & ~(size_t)255; };
    float *dg = static_cast<float *>(scratch);
    float *dgon = reinterpret_cast<float *>(reinterpret_cast<uint8_t *>(dg) + pad(8 * BH * N * L));
    *dg_out = dg;
    *dgon_out = dgon;
    CUtensorMap mQ, mK, mV, mY;
    const unsigned long long rows = (unsigned long long)BH * L;
    if (!make_tmap_bf16_sw128(&mQ, q, rows, p.d, kGT) || !make_tmap_bf16_sw128(&mK, k, rows, p.d, kGT) ||
        !make_tmap_bf16_sw128(&mV, v, rows, p.d, kGT) || !make_tmap_bf16_sw128(&mY, dy, rows, p.d, kGT))
        return cudaErrorInvalidValue;
    CArgs a{};
    a.images = img.states_img;
    a.spre = img.spre_img;
    a.gam = gam;
    a.tok = tok;
    a.dg = dg;
    a.dgon = dgon;
    a.dq = static_cast<__nv_bfloat16 *>(dq);
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.CPS = p.C / kGT; a.d = p.d; a.mode = p.mode;
    a.num_tiles = p.BH * p.N * a.CPS;
    cudaError_t e = cudaFuncSetAttribute(bwd_cached_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kCSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int grid = a.num_tiles < sms ? a.num_tiles : sms;
    bwd_cached_tc<<<grid, kCThreads, kCSmem, s>>>(mQ, mK, mV, mY, a);
    return cudaGetLastError();
}

}  // namespace mc

namespace mc {

cudaError_t launch_bwd_kv_tc(const Problem &p, const void *q, const void *k, const void *v, const void *u, const void *dy,
                             const uint8_t *G, const float *gw, const float *dkbar, void *dk, void *dv, cudaStream_t s)
{
    const bool routed = p.mode == MC_GRM || p.mode == MC_SOUP || p.mode == MC_SSC;
    CUtensorMap mK, mV, mQ, mY, mU;
    const unsigned long long rows = (unsigned long long)p.BH * p.L;
    // K, V: 128-token chunks; q, dy, u: 64-token sub-chunks
    if (!make_tmap_bf16_sw128(&mK, k, rows, p.d, kGT) || !make_tmap_bf16_sw128(&mV, v, rows, p.d, kGT) ||
        !make_tmap_bf16_sw128(&mQ, q, rows, p.d, kG2) || !make_tmap_bf16_sw128(&mY, dy, rows, p.d, kG2))
        return cudaErrorInvalidValue;
    if (routed) {
        if (!make_tmap_bf16_sw128(&mU, u, rows, p.d, kG2)) return cudaErrorInvalidValue;
    } else {
        mU = mQ;
    }
    VArgs a{};
    a.G = G;
    a.gw = gw;
    a.dkbar = dkbar;
    a.dk = dk;
    a.dv = dv;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.CPS = p.C / kGT; a.d = p.d; a.routed = routed ? 1 : 0;
    a.UP = (a.CPS + 1) / 2;
    a.num_units = p.BH * p.N * a.UP;
    cudaError_t e = cudaFuncSetAttribute(bwd_kv_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kVSmem);
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 148;
    const int grid = a.num_units < sms ? a.num_units : sms;
    bwd_kv_tc<<<grid, kVThreads, kVSmem, s>>>(mK, mV, mQ, mY, mU, a);
    return cudaGetLastError();
}

}  // namespace mc
