// k_tc.cu -- tensor-core (tcgen05 / TMEM / TMA) path of the Memory Caching
// forward for bf16 inputs, d = 128, seg_len a multiple of 128, L a multiple of
// seg_len, N <= 64, aggregations Residual / GRM / Soup.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
//
// Two kernels.
//
// seg_state_tc -- one CTA per (bh, segment n).  Walks the segment in chunks of
//   128 tokens with the running state S = sum v_j k_j^T in tensor memory (fp32):
//     S += V_c^T K_c                        (update rule, [MC-ja §3 eq. 4b])
//   Before each chunk's update it writes S (the state before the chunk) as a bf16
//   operand image (the "prefix state" of the chunk); at the end S is the
//   segment's cached state M^(n) ([MC-ja §3, after eq. 4b]), written as fp32
//   (the states output) and as a bf16 image.  It also forms the key mean
//   kbar_n ([MC-ja §3.1 eq. 10], pooled keys) as fp32 hi + lo bf16 rows of a
//   per-head operand image, and the online gate score
//     r_on[t] = <u_t, sum_{j=t0..t} k_j> / (t - t0 + 1)
//   from R = U_c K_c^T (tensor core) masked to j <= t plus <u_t, keys before the chunk>.
//
// readout_tc -- persistent; a tile is (bh, segment n, chunk c) of 128 tokens,
//   heaviest tiles first.  For the tile's tokens it computes
//     y_t = g_{t,n} [ P_t (S_pre(c) q_t) + sum_{j in chunk, j<=t} v_j (k_j . q_t) ]
//         + sum_{i<n} g_{t,i} M^(i) q_t                      ([MC-ja §3.1 eq. 9])
//   with g = softmax over {<u_t, kbar_i>}_{i<n} and r_on[t] (GRM; Soup is the
//   same sum for a linear memory, [MC-sum §3.3]) or g = 1 (Residual, [MC-ja
//   §3.1 eq. 7], where the cached sum collapses to one prefix state).  Every
//   term is an MMA into one fp32 accumulator D_Y[t][v]:
//     online:  G = Q K_c^T;  D_Y  = (g_n * mask(G)) V_c
//     cached:  D_Y += (g_i o Q) X_i^T  for X_i in {S_pre(c) (weight g_n), M^(0..n-1)}
//   The A operands (g_i o Q, the masked P) are written into tensor memory by
//   four "A" warps (thread = token row); four "aux" warps compute the next
//   tile's scores and softmax while the current tile streams its cached states,
//   and drain the double-buffered accumulator.  One warp issues TMA / bulk
//   copies, one issues the MMAs.
#include <cstdint>

#include "mc_internal.cuh"
#include "sm100.cuh"
#include "tensormap.cuh"

namespace mc {

// Set by any tensor-core kernel that abandoned its work after a bounded wait
// ran out; read and cleared by mc_check_device().
__device__ int g_device_abort;

namespace {

using namespace sm100;

constexpr int kD = 128;            // head dimension of this path
constexpr int kCT = 128;           // tokens per chunk / tile
constexpr uint32_t kTile = 32768;  // one 128 x 128 bf16 operand tile

struct TcArgs {
    const __nv_bfloat16 *q, *u;
    __nv_bfloat16 *y;
    float *states;        // [BH][N][128][128] fp32 (output)
    uint8_t *states_img;  // [BH][N] x 32 KB  bf16 operand images of M^(n)
    uint8_t *spre_img;    // [BH][N][CPS] x 32 KB  prefix state before chunk c (c >= 1)
    uint8_t *kbar_img;    // [BH] x 32 KB: hi rows (16 KB) then lo rows (16 KB), row = segment
    uint8_t *prefix_img;  // [BH][N] x 32 KB  sum_{i<n} M^(i) (Residual)
    float *r_on;          // [BH][L]
    int BH, L, C, N, CPS;
    int num_tiles;
};

__device__ __forceinline__ uint8_t *align1024(uint8_t *p)
{
    return reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(p) + 1023) & ~uintptr_t(1023));
}

__device__ __forceinline__ void named_bar_sync(int id, int count)
{
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ float bf16_at(const uint8_t *tile, uint32_t r, uint32_t k, uint32_t rows)
{
    return __bfloat162float(*reinterpret_cast<const __nv_bfloat16 *>(tile + sw128_offset(r, k, rows)));
}

// K-major SW128 descriptor start for the 16-wide K step kk of a tile with `rows` rows.
__device__ __forceinline__ uint32_t kmaj_off(int kk, uint32_t rows) { return (kk >> 2) * rows * 128u + (kk & 3) * 32u; }

// Thread owns TMEM lane `row`; read 128 fp32 columns starting at taddr and
// write them as row `row` of a bf16 SW128 operand image in global memory
// (optionally also as fp32 to out32[0..127]).
__device__ __forceinline__ void tmem_row_to_image(uint32_t taddr, uint32_t row, uint8_t *img, float *out32)
{
#pragma unroll
    for (int h = 0; h < 4; ++h) {  // 32 columns at a time
        uint32_t a[16], b[16];
        tmem_ld16(taddr + 32 * h, a);
        tmem_ld16(taddr + 32 * h + 16, b);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(__uint_as_float(a[2 * i]), __uint_as_float(a[2 * i + 1]));
#pragma unroll
        for (int i = 0; i < 8; ++i) pk[8 + i] = pack_bf16x2(__uint_as_float(b[2 * i]), __uint_as_float(b[2 * i + 1]));
        // columns 32h..32h+31 are four 16-byte chunks (8 bf16 each)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const uint32_t k = 32 * h + 8 * cc;
            uint4 v = make_uint4(pk[4 * cc], pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
            *reinterpret_cast<uint4 *>(img + sw128_offset(row, k, 128)) = v;
        }
        if (out32) {
            float4 *o = reinterpret_cast<float4 *>(out32 + 32 * h);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[i] = make_float4(__uint_as_float(a[4 * i]), __uint_as_float(a[4 * i + 1]), __uint_as_float(a[4 * i + 2]),
                                   __uint_as_float(a[4 * i + 3]));
#pragma unroll
            for (int i = 0; i < 4; ++i)
                o[4 + i] = make_float4(__uint_as_float(b[4 * i]), __uint_as_float(b[4 * i + 1]),
                                       __uint_as_float(b[4 * i + 2]), __uint_as_float(b[4 * i + 3]));
        }
    }
}

// ============================================================================
// seg_state_tc
// ============================================================================
constexpr int kT1Threads = 192;               // warp 0 TMA, warp 1 MMA, warps 2-5 workers
constexpr uint32_t kT1Stage = 3 * kTile;      // K, V, U tiles of one chunk
constexpr size_t kT1Smem = 2 * kT1Stage + 1024;

template <bool GATED>
__global__ void __launch_bounds__(kT1Threads, 1)
    seg_state_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                 const __grid_constant__ CUtensorMap mU, TcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t full[2], empty[2], r_full, r_free, s_ready, s_read;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float ksum_s[kD];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x % a.N, bh = blockIdx.x / a.N;
    const int row0 = bh * a.L + seg * a.C;  // first token row of the segment in the [BH*L, d] view
    const int nch = a.CPS;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 256);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 4);  // MMA commit + one arrive per worker warp
        }
        mbar_init(&r_full, 1);
        mbar_init(&r_free, 128);
        mbar_init(&s_ready, 1);
        mbar_init(&s_read, 128);
        fence_mbar_init();
    }
    if (threadIdx.x >= 64) ksum_s[threadIdx.x - 64] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tR = tb, tS = tb + 128;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            if (GATED) prefetch_tensormap(&mU);
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                const uint32_t r = c >> 1;
                if (!mbar_wait(&empty[s], (r & 1) ^ 1, &abort_flag)) break;
                uint8_t *st = sm + s * kT1Stage;
                mbar_arrive_expect_tx(&full[s], GATED ? 3 * kTile : 2 * kTile);
                const int rr = row0 + c * kCT;
                tma_load_2d(st, &mK, 0, rr, &full[s]);
                tma_load_2d(st + 16384, &mK, 64, rr, &full[s]);
                tma_load_2d(st + kTile, &mV, 0, rr, &full[s]);
                tma_load_2d(st + kTile + 16384, &mV, 64, rr, &full[s]);
                if (GATED) {
                    tma_load_2d(st + 2 * kTile, &mU, 0, rr, &full[s]);
                    tma_load_2d(st + 2 * kTile + 16384, &mU, 64, rr, &full[s]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idR = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idS = idesc_bf16(128, 128, true, true);
            for (int c = 0; c < nch; ++c) {
                const int s = c & 1;
                const uint32_t r = c >> 1;
                if (!mbar_wait(&full[s], r & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(sm + s * kT1Stage), vb = kb + kTile, ub = kb + 2 * kTile;
                if (GATED) {
                    if (!mbar_wait(&r_free, (c & 1) ^ 1, &abort_flag)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tR, make_desc_sw128(ub + kmaj_off(kk, 128), 0, 1024),
                               make_desc_sw128(kb + kmaj_off(kk, 128), 0, 1024), idR, kk > 0);
                    mma_commit(&r_full);
                }
                if (!mbar_wait(&s_read, c & 1, &abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tS, make_desc_sw128(vb + kk * 2048u, 16384, 1024), make_desc_sw128(kb + kk * 2048u, 16384, 1024),
                           idS, (c > 0 || kk > 0) ? 1u : 0u);
                mma_commit(&s_ready);
                mma_commit(&empty[s]);
            }
        }
    } else {
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;  // TMEM lane = token row (R) = value row (S) = key column (sums)
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        float ks = 0.f;  // running sum of key column `row` over the segment, in token order
        // A worker that gives up (bounded wait ran out) keeps walking the loop
        // without work so that every warp reaches the same named barriers.
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1;
            const uint32_t r = c >> 1;
            if (ok && c > 0) {  // the state before chunk c, as the chunk's prefix-state image
                ok = mbar_wait(&s_ready, (c - 1) & 1, &abort_flag);
                if (ok) {
                    tc_fence_after();
                    uint8_t *img = a.spre_img + (((size_t)bh * a.N + seg) * a.CPS + c) * kTile;
                    tmem_row_to_image(tS + lane_base, row, img, nullptr);
                }
            }
            tc_fence_before();
            mbar_arrive(&s_read);
            if (ok) ok = mbar_wait(&full[s], r & 1, &abort_flag);
            const uint8_t *st = sm + s * kT1Stage;
            if (GATED && ok) {
                float dot = 0.f;  // <u_t, keys of the segment before this chunk>
                for (int k = 0; k < kD; ++k) dot = fmaf(bf16_at(st + 2 * kTile, row, k, 128), ksum_s[k], dot);
                ok = mbar_wait(&r_full, c & 1, &abort_flag);
                if (ok) {
                    tc_fence_after();
                    float w = 0.f;  // sum_{j <= t} <u_t, k_j> within the chunk
#pragma unroll
                    for (int j16 = 0; j16 < 8; ++j16) {
                        uint32_t v[16];
                        tmem_ld16(tR + lane_base + 16 * j16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if ((uint32_t)(16 * j16 + i) <= row) w += __uint_as_float(v[i]);
                    }
                    tc_fence_before();
                    mbar_arrive(&r_free);
                    const int t_in_seg = c * kCT + (int)row;
                    a.r_on[(size_t)row0 + t_in_seg] = (dot + w) / (float)(t_in_seg + 1);
                }
            }
            named_bar_sync(1, 128);  // every worker has read ksum_s
            if (ok) {
                float s2 = ks;
                for (int rr = 0; rr < kCT; ++rr) s2 += bf16_at(st, rr, row, 128);
                ks = s2;
                ksum_s[row] = ks;
            }
            named_bar_sync(1, 128);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (ok && !abort_flag && mbar_wait(&s_ready, (nch - 1) & 1, &abort_flag)) {
            tc_fence_after();
            const size_t sidx = (size_t)bh * a.N + seg;
            tmem_row_to_image(tS + lane_base, row, a.states_img + sidx * kTile, a.states + sidx * kD * kD + (size_t)row * kD);
            if (GATED) {
                const float kb = ks / (float)a.C;
                const __nv_bfloat16 hi = __float2bfloat16_rn(kb);
                const __nv_bfloat16 lo = __float2bfloat16_rn(kb - __bfloat162float(hi));
                uint8_t *img = a.kbar_img + (size_t)bh * kTile;
                *reinterpret_cast<__nv_bfloat16 *>(img + sw128_offset(seg, row, 64)) = hi;
                *reinterpret_cast<__nv_bfloat16 *>(img + 16384 + sw128_offset(seg, row, 64)) = lo;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 256);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_device_abort, 1);
}

// Residual: prefix sums of the cached states, P_n = sum_{i<n} M^(i) (fp32
// accumulate), written as bf16 operand images (P_0 is never read).
__global__ void __launch_bounds__(256) prefix_images(TcArgs a)
{
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;  // element of the d x d state
    if (e >= kD * kD) return;
    const int v = e / kD, k = e % kD;
    const float *st = a.states + (size_t)bh * a.N * kD * kD + e;
    float acc = 0.f;
    for (int n = 1; n < a.N; ++n) {
        acc += st[(size_t)(n - 1) * kD * kD];
        *reinterpret_cast<__nv_bfloat16 *>(a.prefix_img + ((size_t)bh * a.N + n) * kTile + sw128_offset(v, k, 128)) =
            __float2bfloat16_rn(acc);
    }
}

// ============================================================================
// readout_tc
// ============================================================================
constexpr int kT2Threads = 320;  // 0 TMA, 1 MMA, 2-5 A producers, 6-9 aux
constexpr int kRing = 4;
constexpr uint32_t kOffK = 0, kOffV = kTile, kOffKbar = 2 * kTile, kOffRing = 3 * kTile;
constexpr size_t kT2Smem = 3 * kTile + kRing * kTile + 1024;

struct TileInfo {
    int n, c, bh;
};

__device__ __forceinline__ TileInfo decode_tile(const TcArgs &a, int id)
{
    const int per_seg = a.BH * a.CPS;
    TileInfo t;
    t.n = a.N - 1 - id / per_seg;
    const int rem = id % per_seg;
    t.c = rem / a.BH;
    t.bh = rem % a.BH;
    return t;
}

template <bool GATED>
__device__ __forceinline__ int tile_items(const TileInfo &t)
{
    return GATED ? t.n + (t.c > 0 ? 1 : 0) : (t.n > 0 ? 1 : 0) + (t.c > 0 ? 1 : 0);
}

template <bool GATED>
__device__ __forceinline__ const uint8_t *item_image(const TcArgs &a, const TileInfo &t, int k)
{
    const size_t sb = (size_t)t.bh * a.N;
    const uint8_t *spre = a.spre_img + ((sb + t.n) * a.CPS + t.c) * kTile;
    if (GATED) {
        if (t.c > 0) {
            if (k == 0) return spre;
            --k;
        }
        return a.states_img + (sb + k) * kTile;
    } else {
        if (t.n > 0) {
            if (k == 0) return a.prefix_img + (sb + t.n) * kTile;
            --k;
        }
        return spre;
    }
}

template <bool GATED>
__global__ void __launch_bounds__(kT2Threads, 1)
    readout_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, TcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t ring_full[kRing], ring_empty[kRing];
    __shared__ uint64_t kv_full, kv_empty, kb_full, kb_empty;
    __shared__ uint64_t a_full[2], a_empty[2];
    __shared__ uint64_t r_free, g_full, g_done, u_full, sc_full, gam_full;
    __shared__ uint64_t y_full[2], y_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles_total = a.num_tiles;
    const int my_tiles = blockIdx.x < (unsigned)ntiles_total
                             ? (ntiles_total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1
                             : 0;
    auto tile_id = [&](int j) { return (int)blockIdx.x + j * (int)gridDim.x; };

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&ring_full[s], 1);
            mbar_init(&ring_empty[s], 1);
        }
        mbar_init(&kv_full, 1);
        mbar_init(&kv_empty, 1);
        mbar_init(&kb_full, 1);
        mbar_init(&kb_empty, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&a_full[s], 128);
            mbar_init(&a_empty[s], 1);
            mbar_init(&y_full[s], 1);
            mbar_init(&y_empty[s], 128);
        }
        mbar_init(&r_free, 128);
        mbar_init(&g_full, 1);
        mbar_init(&g_done, 128);
        mbar_init(&u_full, 128);
        mbar_init(&sc_full, 1);
        mbar_init(&gam_full, 128);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tY0 = tb, tR = tb + 256, tA0 = tb + 384;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        if (lane == 0 && my_tiles > 0) {
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            int kv_next = 0, kb_next = GATED ? 0 : my_tiles;  // next tile whose K/V, kbar image to load
            int it_tile = 0, it_k = 0;                          // next ring item
            uint32_t g = 0;
            TileInfo it_info = decode_tile(a, tile_id(0));
            while (tile_items<GATED>(it_info) == 0) {  // skip tiles that read no cached state
                if (++it_tile >= my_tiles) break;
                it_info = decode_tile(a, tile_id(it_tile));
            }
            uint64_t t_idle = 0;
            bool idle = false;
            while (kv_next < my_tiles || kb_next < my_tiles || it_tile < my_tiles) {
                bool did = false;
                if (kv_next < my_tiles && mbar_try_wait(&kv_empty, (kv_next & 1) ^ 1)) {
                    const TileInfo t = decode_tile(a, tile_id(kv_next));
                    const int rr = t.bh * a.L + t.n * a.C + t.c * kCT;
                    mbar_arrive_expect_tx(&kv_full, 2 * kTile);
                    tma_load_2d(sm + kOffK, &mK, 0, rr, &kv_full);
                    tma_load_2d(sm + kOffK + 16384, &mK, 64, rr, &kv_full);
                    tma_load_2d(sm + kOffV, &mV, 0, rr, &kv_full);
                    tma_load_2d(sm + kOffV + 16384, &mV, 64, rr, &kv_full);
                    ++kv_next;
                    did = true;
                }
                if (GATED && kb_next < my_tiles && mbar_try_wait(&kb_empty, (kb_next & 1) ^ 1)) {
                    const TileInfo t = decode_tile(a, tile_id(kb_next));
                    mbar_arrive_expect_tx(&kb_full, kTile);
                    bulk_load(sm + kOffKbar, a.kbar_img + (size_t)t.bh * kTile, kTile, &kb_full);
                    ++kb_next;
                    did = true;
                }
                if (it_tile < my_tiles) {
                    const int s = g % kRing;
                    const uint32_t r = g / kRing;
                    if (mbar_try_wait(&ring_empty[s], (r & 1) ^ 1)) {
                        mbar_arrive_expect_tx(&ring_full[s], kTile);
                        bulk_load(sm + kOffRing + s * kTile, item_image<GATED>(a, it_info, it_k), kTile, &ring_full[s]);
                        ++g;
                        did = true;
                        if (++it_k >= tile_items<GATED>(it_info)) {
                            it_k = 0;
                            ++it_tile;
                            while (it_tile < my_tiles) {
                                it_info = decode_tile(a, tile_id(it_tile));
                                if (tile_items<GATED>(it_info) > 0) break;
                                ++it_tile;
                            }
                        }
                    }
                }
                if (did) {
                    idle = false;
                } else {
                    if (abort_flag) break;
                    if (!idle) {
                        idle = true;
                        t_idle = globaltimer_ns();
                    } else if (globaltimer_ns() - t_idle > kWaitLimitNs) {
                        abort_flag = 1;
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && my_tiles > 0) {
            constexpr uint32_t idG = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idPV = idesc_bf16(128, 128, false, true);
            constexpr uint32_t idC = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
            const uint32_t kb_base = s_base + kOffKbar;
            auto issue_scores = [&](int jn) -> bool {
                if (!mbar_wait(&u_full, jn & 1, &abort_flag)) return false;
                if (!mbar_wait(&kb_full, jn & 1, &abort_flag)) return false;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tR, tR + 64 + kk * 8, make_desc_sw128(kb_base + kmaj_off(kk, 64), 0, 1024), idS, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ts(tR, tR + 64 + kk * 8, make_desc_sw128(kb_base + 16384 + kmaj_off(kk, 64), 0, 1024), idS, 1);
                mma_commit(&sc_full);
                mma_commit(&kb_empty);
                return true;
            };
            uint32_t g = 0, ac = 0;
            bool ok = true;
            if (GATED) ok = issue_scores(0);
            for (int j = 0; j < my_tiles && ok; ++j) {
                const TileInfo t = decode_tile(a, tile_id(j));
                const uint32_t tY = tY0 + (j & 1) * 128;
                // online: G = Q K^T into R
                if (!(ok = mbar_wait(&kv_full, j & 1, &abort_flag))) break;
                if (!(ok = mbar_wait(&r_free, j & 1, &abort_flag))) break;
                if (!(ok = mbar_wait(&a_full[ac & 1], (ac >> 1) & 1, &abort_flag))) break;
                tc_fence_after();
                {
                    const uint32_t ta = tA0 + (ac & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tR, ta + kk * 8, make_desc_sw128(s_base + kOffK + kmaj_off(kk, 128), 0, 1024), idG, kk > 0);
                    mma_commit(&g_full);
                    mma_commit(&a_empty[ac & 1]);
                    ++ac;
                }
                // online: D_Y = P V
                if (!(ok = mbar_wait(&y_empty[j & 1], ((j >> 1) & 1) ^ 1, &abort_flag))) break;
                if (!(ok = mbar_wait(&a_full[ac & 1], (ac >> 1) & 1, &abort_flag))) break;
                tc_fence_after();
                {
                    const uint32_t ta = tA0 + (ac & 1) * 64;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tY, ta + kk * 8, make_desc_sw128(s_base + kOffV + kk * 2048u, 16384, 1024), idPV, kk > 0);
                    mma_commit(&a_empty[ac & 1]);
                    mma_commit(&kv_empty);
                    ++ac;
                }
                // cached states (and the chunk's prefix state)
                bool next_scores = GATED && j + 1 < my_tiles;
                const int items = tile_items<GATED>(t);
                for (int k = 0; k < items; ++k) {
                    if (next_scores && mbar_try_wait(&u_full, (j + 1) & 1) && mbar_try_wait(&kb_full, (j + 1) & 1)) {
                        if (!(ok = issue_scores(j + 1))) break;
                        next_scores = false;
                    }
                    const int s = g % kRing;
                    if (!(ok = mbar_wait(&ring_full[s], (g / kRing) & 1, &abort_flag))) break;
                    if (!(ok = mbar_wait(&a_full[ac & 1], (ac >> 1) & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t ta = tA0 + (ac & 1) * 64;
                    const uint32_t bb = s_base + kOffRing + s * kTile;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ts(tY, ta + kk * 8, make_desc_sw128(bb + kmaj_off(kk, 128), 0, 1024), idC, 1);
                    mma_commit(&ring_empty[s]);
                    mma_commit(&a_empty[ac & 1]);
                    ++g;
                    ++ac;
                }
                if (!ok) break;
                if (next_scores && !(ok = issue_scores(j + 1))) break;
                mma_commit(&y_full[j & 1]);
            }
        }
    } else if (warp < 6) {
        // ---------------------------------------------------------- A producers
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t ac = 0;
        bool ok = true;
        auto put_a = [&](const uint32_t (&src)[64], __nv_bfloat162 gam, bool scale) -> bool {
            if (!mbar_wait(&a_empty[ac & 1], ((ac >> 1) & 1) ^ 1, &abort_flag)) return false;
            tc_fence_after();
            const uint32_t ta = tA0 + (ac & 1) * 64 + lane_base;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (scale) {
                        __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&src[16 * m + i]);
                        __nv_bfloat162 pr = __hmul2(x, gam);
                        r[i] = *reinterpret_cast<uint32_t *>(&pr);
                    } else {
                        r[i] = src[16 * m + i];
                    }
                }
                tmem_st16(ta + 16 * m, r);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&a_full[ac & 1]);
            ++ac;
            return true;
        };
        for (int j = 0; j < my_tiles && ok; ++j) {
            const TileInfo t = decode_tile(a, tile_id(j));
            uint32_t gm2[32];  // gates g_{t,i} as bf16 pairs (i even: low half)
            float g_on = 1.f;
            if (GATED) {
                if (!(ok = mbar_wait(&gam_full, j & 1, &abort_flag))) break;
                tc_fence_after();
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t v[16];
                    tmem_ld16(tR + lane_base + 16 * m, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 8; ++i) gm2[8 * m + i] = pack_bf16x2(__uint_as_float(v[2 * i]), __uint_as_float(v[2 * i + 1]));
                    if (m == 3) g_on = __uint_as_float(v[15]);
                }
            }
            tc_fence_before();
            mbar_arrive(&r_free);
            // the token's query row
            uint32_t qp[64];
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(
                    a.q + ((size_t)t.bh * a.L + (size_t)t.n * a.C + (size_t)t.c * kCT + row) * kD);
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    const uint4 x = __ldg(src + i);
                    qp[4 * i] = x.x;
                    qp[4 * i + 1] = x.y;
                    qp[4 * i + 2] = x.z;
                    qp[4 * i + 3] = x.w;
                }
            }
            const __nv_bfloat162 one2 = __float2bfloat162_rn(1.f);
            if (!(ok = put_a(qp, one2, false))) break;  // Q for G = Q K^T
            // P = g_on * mask(G): wait for G, write P as the next A operand
            if (!(ok = mbar_wait(&g_full, j & 1, &abort_flag))) break;
            tc_fence_after();
            if (!(ok = mbar_wait(&a_empty[ac & 1], ((ac >> 1) & 1) ^ 1, &abort_flag))) break;
            tc_fence_after();
            {
                const uint32_t ta = tA0 + (ac & 1) * 64 + lane_base;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t x[16], z[16];
                    tmem_ld16(tR + lane_base + 32 * h, x);
                    tmem_ld16(tR + lane_base + 32 * h + 16, z);
                    tmem_wait_ld();
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        const uint32_t c0 = 32 * h + 2 * i;
                        const float p0 = c0 <= row ? g_on * __uint_as_float(x[2 * i]) : 0.f;
                        const float p1 = c0 + 1 <= row ? g_on * __uint_as_float(x[2 * i + 1]) : 0.f;
                        pk[i] = pack_bf16x2(p0, p1);
                        const uint32_t c1 = 32 * h + 16 + 2 * i;
                        const float p2 = c1 <= row ? g_on * __uint_as_float(z[2 * i]) : 0.f;
                        const float p3 = c1 + 1 <= row ? g_on * __uint_as_float(z[2 * i + 1]) : 0.f;
                        pk[8 + i] = pack_bf16x2(p2, p3);
                    }
                    tmem_st16(ta + 16 * h, pk);
                }
                tc_fence_before();
                mbar_arrive(&g_done);  // R has been read
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&a_full[ac & 1]);
                ++ac;
            }
            // cached items
            if (GATED) {
                const __nv_bfloat162 gon2 = __float2bfloat162_rn(g_on);
                if (t.c > 0 && !(ok = put_a(qp, gon2, true))) break;
#pragma unroll
                for (int i = 0; i < 63; ++i) {
                    if (i >= t.n) break;
                    const __nv_bfloat162 pair = *reinterpret_cast<const __nv_bfloat162 *>(&gm2[i >> 1]);
                    const __nv_bfloat162 gi2 = (i & 1) ? __high2bfloat162(pair) : __low2bfloat162(pair);
                    if (!(ok = put_a(qp, gi2, true))) break;
                }
                if (!ok) break;
            } else {
                const int items = tile_items<GATED>(t);
                for (int k = 0; k < items && ok; ++k) ok = put_a(qp, one2, false);
            }
        }
    } else {
        // ---------------------------------------------------------- aux: next-tile gates, drain
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        bool ok = true;
        auto pre = [&](int jn) -> bool {
            const TileInfo t = decode_tile(a, tile_id(jn));
            const size_t tok = (size_t)t.bh * a.L + (size_t)t.n * a.C + (size_t)t.c * kCT + row;
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.u + tok * kD);
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    uint32_t r[16];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 x = __ldg(src + 4 * m + i);
                        r[4 * i] = x.x;
                        r[4 * i + 1] = x.y;
                        r[4 * i + 2] = x.z;
                        r[4 * i + 3] = x.w;
                    }
                    tmem_st16(tR + 64 + lane_base + 16 * m, r);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(&u_full);
            const float ron = a.r_on[tok];
            if (!mbar_wait(&sc_full, jn & 1, &abort_flag)) return false;
            tc_fence_after();
            float sc[64];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t v[16];
                tmem_ld16(tR + lane_base + 16 * m, v);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 16; ++i) sc[16 * m + i] = __uint_as_float(v[i]);
            }
            float mx = ron;
#pragma unroll
            for (int i = 0; i < 63; ++i)
                if (i < t.n) mx = fmaxf(mx, sc[i]);
            float z = expf(ron - mx);
#pragma unroll
            for (int i = 0; i < 63; ++i) {
                if (i < t.n) {
                    sc[i] = expf(sc[i] - mx);
                    z += sc[i];
                }
            }
            const float inv = 1.f / z;
#pragma unroll
            for (int i = 0; i < 63; ++i) sc[i] *= inv;
            sc[63] = expf(ron - mx) * inv;
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t r[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(sc[16 * m + i]);
                tmem_st16(tR + lane_base + 16 * m, r);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&gam_full);
            return true;
        };
        if (GATED && my_tiles > 0) ok = pre(0);
        for (int j = 0; j < my_tiles && ok; ++j) {
            const TileInfo t = decode_tile(a, tile_id(j));
            if (GATED && j + 1 < my_tiles) {
                if (!(ok = mbar_wait(&g_done, j & 1, &abort_flag))) break;
                tc_fence_after();
                if (!(ok = pre(j + 1))) break;
            }
            // drain D_Y of tile j into y
            if (!(ok = mbar_wait(&y_full[j & 1], (j >> 1) & 1, &abort_flag))) break;
            tc_fence_after();
            const uint32_t tY = tY0 + (j & 1) * 128 + lane_base;
            uint4 *dst = reinterpret_cast<uint4 *>(
                a.y + ((size_t)t.bh * a.L + (size_t)t.n * a.C + (size_t)t.c * kCT + row) * kD);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t x[16], z[16];
                tmem_ld16(tY + 32 * h, x);
                tmem_ld16(tY + 32 * h + 16, z);
                tmem_wait_ld();
                uint32_t pk[16];
#pragma unroll
                for (int i = 0; i < 8; ++i) pk[i] = pack_bf16x2(__uint_as_float(x[2 * i]), __uint_as_float(x[2 * i + 1]));
#pragma unroll
                for (int i = 0; i < 8; ++i) pk[8 + i] = pack_bf16x2(__uint_as_float(z[2 * i]), __uint_as_float(z[2 * i + 1]));
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[4 * h + i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
            }
            tc_fence_before();
            mbar_arrive(&y_empty[j & 1]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_device_abort, 1);
}

size_t pad256(size_t x) { return (x + 255) & ~(size_t)255; }

int g_num_sms = 0;

}  // namespace

cudaError_t take_device_abort(int *was_set)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_device_abort, sizeof(int));
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        v = 0;
        e = cudaMemcpyToSymbol(g_device_abort, &v, sizeof(int));
    }
    return e;
}

bool tc_supported(const Problem &p)
{
    return p.bf16 && p.d == kD && p.C % kCT == 0 && p.L % p.C == 0 && p.N <= 64 &&
           (p.mode == MC_GRM || p.mode == MC_SOUP || p.mode == MC_RESIDUAL);
}

size_t tc_scratch_bytes(const Problem &p)
{
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT;
    size_t b = pad256(BH * N * kTile) + pad256(BH * N * CPS * kTile) + pad256(BH * kTile) +
               pad256(sizeof(float) * BH * p.L);
    if (p.mode == MC_RESIDUAL) b += pad256(BH * N * kTile);
    return b;
}

cudaError_t launch_forward_tc(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    const bool gated = p.mode != MC_RESIDUAL;
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    TcArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(fa.q);
    a.u = static_cast<const __nv_bfloat16 *>(fa.u);
    a.y = static_cast<__nv_bfloat16 *>(fa.y);
    a.states = fa.states;
    a.states_img = base;
    base += pad256(BH * N * kTile);
    a.spre_img = base;
    base += pad256(BH * N * CPS * kTile);
    a.kbar_img = base;
    base += pad256(BH * kTile);
    a.r_on = reinterpret_cast<float *>(base);
    base += pad256(sizeof(float) * BH * p.L);
    a.prefix_img = gated ? nullptr : base;
    a.BH = p.BH;
    a.L = p.L;
    a.C = p.C;
    a.N = p.N;
    a.CPS = (int)CPS;
    a.num_tiles = (int)(BH * N * CPS);

    CUtensorMap mK, mV, mU;
    const unsigned long long rows = (unsigned long long)BH * p.L;
    if (!make_tmap_bf16_sw128(&mK, fa.k, rows, kD, 128) || !make_tmap_bf16_sw128(&mV, fa.v, rows, kD, 128))
        return cudaErrorInvalidValue;
    if (gated) {
        if (!make_tmap_bf16_sw128(&mU, fa.u, rows, kD, 128)) return cudaErrorInvalidValue;
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
    if (gated) {
        e = cudaMemsetAsync(a.kbar_img, 0, BH * kTile, s);
        if (e != cudaSuccess) return e;
    }

    profile_call_start(s);
    {
        auto k1 = gated ? seg_state_tc<true> : seg_state_tc<false>;
        e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kT1Smem);
        if (e != cudaSuccess) return e;
        k1<<<(unsigned)(BH * N), kT1Threads, kT1Smem, s>>>(mK, mV, mU, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "seg_state_tc");
    }
    if (!gated) {
        dim3 grid((kD * kD + 255) / 256, (unsigned)BH);
        prefix_images<<<grid, 256, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "prefix_images");
    }
    {
        auto k2 = gated ? readout_tc<true> : readout_tc<false>;
        e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kT2Smem);
        if (e != cudaSuccess) return e;
        const int grid = a.num_tiles < g_num_sms ? a.num_tiles : g_num_sms;
        k2<<<grid, kT2Threads, kT2Smem, s>>>(mK, mV, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "readout_tc");
    }
    return cudaSuccess;
}

}  // namespace mc
