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
constexpr int kTcMaxTopk = 16;     // SSC selections per token handled by the tensor-core path
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
    __nv_bfloat16 *gam;   // [BH][L][64] gates: g_i at column i < n, g_n at column 63
    int32_t *sel_out;     // SSC: optional [BH][L][topk] router output (rank order, -1 padded)
    int topk;             // SSC: cached segments selected per token
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
    __shared__ uint64_t full[2], empty[2], r_full[2], r_empty[2], z_full[2], z_empty[2];
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float ksum_s[kD];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int seg = blockIdx.x % a.N, bh = blockIdx.x / a.N;
    const int row0 = bh * a.L + seg * a.C;  // first token row of the segment in the [BH*L, d] view
    const int nch = a.CPS;

    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1 + 4);  // MMA commit + one arrive per worker warp
            mbar_init(&r_full[s], 1);
            mbar_init(&r_empty[s], 128);
            mbar_init(&z_full[s], 1);
            mbar_init(&z_empty[s], 128);
        }
        fence_mbar_init();
    }
    if (threadIdx.x >= 64) ksum_s[threadIdx.x - 64] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    // tensor memory: R (U K^T) x 2 | Z (chunk state V^T K) x 2, 128 columns each
    const uint32_t tR0 = tb, tZ0 = tb + 256;

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
                const int s = c & 1, b = c & 1;
                const uint32_t r = c >> 1;
                if (!mbar_wait(&full[s], r & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(sm + s * kT1Stage), vb = kb + kTile, ub = kb + 2 * kTile;
                if (GATED) {  // R = U K^T (online gate score of the chunk's tokens)
                    if (!mbar_wait(&r_empty[b], (r & 1) ^ 1, &abort_flag)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk)
                        mma_ss(tR0 + b * 128, make_desc_sw128(ub + kmaj_off(kk, 128), 0, 1024),
                               make_desc_sw128(kb + kmaj_off(kk, 128), 0, 1024), idR, kk > 0);
                    mma_commit(&r_full[b]);
                }
                // Z = V^T K, the chunk's own state (fresh accumulator)
                if (!mbar_wait(&z_empty[b], (r & 1) ^ 1, &abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tZ0 + b * 128, make_desc_sw128(vb + kk * 2048u, 16384, 1024),
                           make_desc_sw128(kb + kk * 2048u, 16384, 1024), idS, kk > 0);
                mma_commit(&z_full[b]);
                mma_commit(&empty[s]);
            }
        }
    } else {
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;  // TMEM lane = token row (R) = value row (Z, S) = key column (sums)
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        float S[kD];  // running state row: S[row][k] = sum_{j before the chunk} v_j[row] k_j[k]
#pragma unroll
        for (int k = 0; k < kD; ++k) S[k] = 0.f;
        float ks = 0.f;  // running sum of key column `row` over the segment, in token order
        // A worker that gives up (bounded wait ran out) keeps walking the loop
        // without work so that every warp reaches the same named barriers.
        bool ok = true;
        for (int c = 0; c < nch; ++c) {
            const int s = c & 1, b = c & 1;
            const uint32_t r = c >> 1;
            if (ok) ok = mbar_wait(&full[s], r & 1, &abort_flag);
            const uint8_t *st = sm + s * kT1Stage;
            if (GATED && ok) {
                float dot = 0.f;  // <u_t, keys of the segment before this chunk>
                for (int k = 0; k < kD; ++k) dot = fmaf(bf16_at(st + 2 * kTile, row, k, 128), ksum_s[k], dot);
                ok = mbar_wait(&r_full[b], r & 1, &abort_flag);
                if (ok) {
                    tc_fence_after();
                    float w = 0.f;  // sum_{j <= t} <u_t, k_j> within the chunk
#pragma unroll
                    for (int j16 = 0; j16 < 8; ++j16) {
                        uint32_t v[16];
                        tmem_ld16(tR0 + b * 128 + lane_base + 16 * j16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if ((uint32_t)(16 * j16 + i) <= row) w += __uint_as_float(v[i]);
                    }
                    tc_fence_before();
                    mbar_arrive(&r_empty[b]);
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
            // S += Z_c; then S is the prefix state of chunk c + 1
            if (ok) ok = mbar_wait(&z_full[b], r & 1, &abort_flag);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int j16 = 0; j16 < 8; ++j16) {
                    uint32_t v[16];
                    tmem_ld16(tZ0 + b * 128 + lane_base + 16 * j16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) S[16 * j16 + i] += __uint_as_float(v[i]);
                }
                tc_fence_before();
                mbar_arrive(&z_empty[b]);
                const size_t sidx = (size_t)bh * a.N + seg;
                uint8_t *img = c + 1 < nch ? a.spre_img + (sidx * a.CPS + c + 1) * kTile : a.states_img + sidx * kTile;
#pragma unroll
                for (int cc = 0; cc < 16; ++cc) {  // 16-byte chunks of 8 bf16
                    const uint4 v = make_uint4(pack_bf16x2(S[8 * cc], S[8 * cc + 1]), pack_bf16x2(S[8 * cc + 2], S[8 * cc + 3]),
                                               pack_bf16x2(S[8 * cc + 4], S[8 * cc + 5]), pack_bf16x2(S[8 * cc + 6], S[8 * cc + 7]));
                    *reinterpret_cast<uint4 *>(img + sw128_offset(row, 8 * cc, 128)) = v;
                }
                if (c + 1 == nch) {  // the segment's cached state, fp32
                    float4 *o = reinterpret_cast<float4 *>(a.states + sidx * kD * kD + (size_t)row * kD);
#pragma unroll
                    for (int i = 0; i < kD / 4; ++i) o[i] = make_float4(S[4 * i], S[4 * i + 1], S[4 * i + 2], S[4 * i + 3]);
                }
            }
        }
        if (ok && GATED && !abort_flag) {
            const float kb = ks / (float)a.C;
            const __nv_bfloat16 hi = __float2bfloat16_rn(kb);
            const __nv_bfloat16 lo = __float2bfloat16_rn(kb - __bfloat162float(hi));
            uint8_t *img = a.kbar_img + (size_t)bh * kTile;
            *reinterpret_cast<__nv_bfloat16 *>(img + sw128_offset(seg, row, 64)) = hi;
            *reinterpret_cast<__nv_bfloat16 *>(img + 16384 + sw128_offset(seg, row, 64)) = lo;
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

// Key means alone, as hi/lo bf16 image rows (for the stand-alone SSC router):
// the same sequential fp32 sum over the segment's tokens as seg_state_tc, so the
// router sees bit-identical scores.
__global__ void __launch_bounds__(kD) kbar_images_tc(const __nv_bfloat16 *__restrict__ k, TcArgs a)
{
    const int seg = blockIdx.x % a.N, bh = blockIdx.x / a.N;
    const int col = threadIdx.x;
    const __nv_bfloat16 *src = k + ((size_t)bh * a.L + (size_t)seg * a.C) * kD + col;
    float s = 0.f;
    for (int t = 0; t < a.C; ++t) s += __bfloat162float(src[(size_t)t * kD]);
    const float kb = s / (float)a.C;
    const __nv_bfloat16 hi = __float2bfloat16_rn(kb);
    const __nv_bfloat16 lo = __float2bfloat16_rn(kb - __bfloat162float(hi));
    uint8_t *img = a.kbar_img + (size_t)bh * kTile;
    *reinterpret_cast<__nv_bfloat16 *>(img + sw128_offset(seg, col, 64)) = hi;
    *reinterpret_cast<__nv_bfloat16 *>(img + 16384 + sw128_offset(seg, col, 64)) = lo;
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
// gates_tc -- the gate of every token ([MC-ja §3.1 eq. 10], normalised by a
// softmax): one CTA per 128-token chunk.  Scores r_{t,i} = <u_t, kbar_i> come
// from two MMAs (kbar as hi + lo bf16 rows, so the score carries ~16 bits of
// kbar; u is exact in bf16), then
//   g_{t,i} = exp(r_{t,i} - m) / Z (i < n),  g_{t,n} = exp(r_on[t] - m) / Z
// written as bf16: gam[token][i] for i < n and gam[token][63] for the online memory.
// ============================================================================
constexpr int kGatesThreads = 320;  // warp 0 TMA, warp 1 MMA, warps 2-9 softmax + store
constexpr size_t kGatesSmem = 3 * kTile + 1024;  // two U tiles, one kbar image

// Persistent: CTA b handles the contiguous tile range [b*per, (b+1)*per) of the
// (bh, chunk) tiles, so consecutive tiles share a head and its kbar image.
template <bool SSC>
__global__ void __launch_bounds__(kGatesThreads, 2) gates_tc(const __grid_constant__ CUtensorMap mU, TcArgs a)
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
                    mbar_arrive_expect_tx(&kb_full, kTile);
                    bulk_load(sKb, a.kbar_img + (size_t)bh * kTile, kTile, &kb_full);
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
                for (int kk = 0; kk < 8; ++kk) mma_ss(td, dU + (kmaj_off(kk, 128) >> 4), dKb + (kmaj_off(kk, 64) >> 4), idS, kk > 0);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(td, dU + (kmaj_off(kk, 128) >> 4), dKb + ((16384 + kmaj_off(kk, 64)) >> 4), idS, 1);
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
            float sc[64];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                uint32_t v[16];
                tmem_ld16(tb + b * 64 + lane_base + 16 * m, v);
                tmem_wait_ld();
#pragma unroll
                for (int k = 0; k < 16; ++k) sc[16 * m + k] = __uint_as_float(v[k]);
            }
            tc_fence_before();
            mbar_arrive(&s_empty[b]);
            const size_t tok = (size_t)bh * a.L + t0 + row;
            const float ron = a.r_on ? a.r_on[tok] : 0.f;  // no r_on: router only
            // GRM / Soup: every cached segment takes part.  SSC ([MC-sum §3.4]): the
            // topk largest scores, equal scores to the lower segment index.
            uint64_t take = n >= 64 ? ~0ull : ((1ull << n) - 1);
            if (SSC) {
                const int cnt = min(a.topk, n);
                uint64_t chosen = 0;
                int32_t *so = a.sel_out ? a.sel_out + tok * a.topk : nullptr;
                for (int r = 0; r < cnt; ++r) {
                    float best = 0.f;
                    int bi = -1;
#pragma unroll
                    for (int k = 0; k < 63; ++k)
                        if (k < n && !((chosen >> k) & 1ull) && (bi < 0 || sc[k] > best)) {
                            best = sc[k];
                            bi = k;
                        }
                    chosen |= 1ull << bi;
                    if (so) so[r] = bi;
                }
                if (so)
                    for (int r = cnt; r < a.topk; ++r) so[r] = -1;
                take = chosen;
            }
            float mx4[4] = {ron, ron, ron, ron};  // partial maxima / sums: shorter dependency chains
#pragma unroll
            for (int k = 0; k < 63; ++k)
                if ((take >> k) & 1ull) mx4[k & 3] = fmaxf(mx4[k & 3], sc[k]);
            const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
            float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int k = 0; k < 63; ++k) {
                sc[k] = ((take >> k) & 1ull) ? expf(sc[k] - mx) : 0.f;
                z4[k & 3] += sc[k];
            }
            sc[63] = expf(ron - mx);
            const float inv = 1.f / (sc[63] + (z4[0] + z4[1]) + (z4[2] + z4[3]));
            if (!a.gam) continue;  // router only (mc_ssc_select)
            uint4 *dst = reinterpret_cast<uint4 *>(a.gam + tok * 64);
#pragma unroll
            for (int k = 0; k < 8; ++k)
                dst[k] = make_uint4(pack_bf16x2(sc[8 * k] * inv, sc[8 * k + 1] * inv),
                                    pack_bf16x2(sc[8 * k + 2] * inv, sc[8 * k + 3] * inv),
                                    pack_bf16x2(sc[8 * k + 4] * inv, sc[8 * k + 5] * inv),
                                    pack_bf16x2(sc[8 * k + 6] * inv, sc[8 * k + 7] * inv));
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 128);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_device_abort, 1);
}

// ============================================================================
// readout_tc
// ============================================================================
constexpr int kT2Threads = 352;  // 0 TMA, 1 MMA issuer 0, 2-5 A producers, 6-9 aux, 10 MMA issuer 1
constexpr int kRing = 7;     // 32 KB operand slots: K, prefix state, cached states, V of each tile
constexpr int kASlots = 4;   // A operands (bf16, 64 TMEM columns each) in flight
constexpr size_t kT2Smem = kRing * kTile + 1024;

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

// Cached operands a tile reads, in order: the chunk's prefix state (c > 0), then
// the cached states M^(0..n-1) (GRM) or their prefix sum P_n (Residual, n > 0).
template <bool GATED>
__device__ __forceinline__ int tile_items(const TileInfo &t)
{
    return GATED ? t.n + (t.c > 0 ? 1 : 0) : (t.n > 0 ? 1 : 0) + (t.c > 0 ? 1 : 0);
}

template <bool GATED>
__device__ __forceinline__ const uint8_t *item_image(const TcArgs &a, const TileInfo &t, int k)
{
    const size_t sb = (size_t)t.bh * a.N;
    if (t.c > 0) {
        if (k == 0) return a.spre_img + ((sb + t.n) * a.CPS + t.c) * kTile;
        --k;
    }
    return GATED ? a.states_img + (sb + k) * kTile : a.prefix_img + (sb + t.n) * kTile;
}

// Accumulator groups of a tile: items + the P V product.  With two or more the
// two accumulators are both written (the MMA warp alternates between them).
template <bool GATED>
__device__ __forceinline__ int tile_groups(const TileInfo &t)
{
    return tile_items<GATED>(t) + 1;
}

template <bool GATED>
__global__ void __launch_bounds__(kT2Threads, 1)
    readout_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV, TcArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t ring_full[kRing], ring_empty[kRing];
    __shared__ uint64_t a_full[kASlots], a_empty[kASlots];
    __shared__ uint64_t g_full, g_done, y_full, y_empty, p_slot, p_written;
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
        for (int s = 0; s < kASlots; ++s) {
            mbar_init(&a_full[s], 128);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(&g_full, 1);
        mbar_init(&g_done, 128);
        mbar_init(&p_slot, 128);
        mbar_init(&p_written, 128);
        mbar_init(&y_full, 2);  // one commit from each MMA issuer
        mbar_init(&y_empty, 128);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    // tensor memory: D0 (128 cols) | D1 (128; holds G at the start of a tile) | A slots (4 x 64).
    // A slot sequence of a tile: g_n o Q (for G and the prefix state), one slot per
    // cached operand (A warps), then P for the P V product (aux warps).
    const uint32_t tD0 = tb, tD1 = tb + 128, tA0 = tb + 256;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        // ---------------------------------------------------------- producer
        // Ring sequence of a tile: K tile, the cached operands, V tile.  At the
        // start of each tile it also prefetches the next tile's query rows and
        // gate rows into L2 for the A warps.
        if (lane == 0 && my_tiles > 0) {
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            uint32_t g = 0;
            bool ok = true;
            auto slot = [&](uint32_t bytes) -> uint8_t * {
                const int s = g % kRing;
                if (!mbar_wait(&ring_empty[s], ((g / kRing) & 1) ^ 1, &abort_flag)) return nullptr;
                mbar_arrive_expect_tx(&ring_full[s], bytes);
                return sm + s * kTile;
            };
            for (int j = 0; j < my_tiles && ok; ++j) {
                const TileInfo t = decode_tile(a, tile_id(j));
                const int rr = t.bh * a.L + t.n * a.C + t.c * kCT;
                if (j + 1 < my_tiles) {
                    const TileInfo tn = decode_tile(a, tile_id(j + 1));
                    const size_t rn = (size_t)tn.bh * a.L + (size_t)tn.n * a.C + (size_t)tn.c * kCT;
                    prefetch_l2(a.q + rn * kD, kTile);
                    if (GATED) prefetch_l2(a.gam + rn * 64, kCT * 64 * 2);
                }
                uint8_t *dst = slot(kTile);
                if (!(ok = dst != nullptr)) break;
                tma_load_2d(dst, &mK, 0, rr, &ring_full[g % kRing]);
                tma_load_2d(dst + 16384, &mK, 64, rr, &ring_full[g % kRing]);
                ++g;
                const int items = tile_items<GATED>(t);
                for (int k = 0; k < items; ++k) {
                    if (!(dst = slot(kTile))) break;
                    bulk_load(dst, item_image<GATED>(a, t, k), kTile, &ring_full[g % kRing]);
                    ++g;
                }
                if (!(ok = dst != nullptr)) break;
                if (!(ok = (dst = slot(kTile)) != nullptr)) break;
                tma_load_2d(dst, &mV, 0, rr, &ring_full[g % kRing]);
                tma_load_2d(dst + 16384, &mV, 64, rr, &ring_full[g % kRing]);
                ++g;
            }
        }
    } else if (warp == 1 || warp == kT2Threads / 32 - 1) {
        // ---------------------------------------------------------- MMA issuers
        // Two issuing threads: a single thread cannot issue tcgen05.mma fast enough
        // to keep the tensor pipe busy once its per-group bookkeeping is counted.
        // Issuer 1 owns accumulator D1 (G, then the odd groups of a tile), issuer 0
        // owns D0 (the even groups).  Group k of a tile is the k-th cached operand
        // (prefix state first), the last group is P V.  Every ring and A slot has
        // exactly one consumer, which commits its release.
        if (lane == 0 && my_tiles > 0) {
            const int me = warp == 1 ? 0 : 1;
            constexpr uint32_t idKm = idesc_bf16(128, 128, false, false);  // B K-major
            constexpr uint32_t idPV = idesc_bf16(128, 128, false, true);   // B MN-major (V)
            const uint64_t dRing0 = make_desc_sw128(s_base, 0, 1024);
            const uint64_t dRingMN = make_desc_sw128(s_base, 16384, 1024);
            uint32_t off128[8];
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) off128[kk] = kmaj_off(kk, 128) >> 4;
            const uint32_t tD = me ? tD1 : tD0;
            uint32_t g = 0, ac = 0;  // ring / A-slot index of the tile's first slot
            bool ok = true;
            for (int j = 0; j < my_tiles && ok; ++j) {
                const TileInfo t = decode_tile(a, tile_id(j));
                const int groups = tile_items<GATED>(t) + 1;
                if (me == 1) {  // G = (g_n o Q) K^T into D1
                    const int s = g % kRing;
                    if (!(ok = mbar_wait(&ring_full[s], (g / kRing) & 1, &abort_flag))) break;
                    if (!(ok = mbar_wait(&a_full[ac % kASlots], (ac / kASlots) & 1, &abort_flag))) break;
                    if (!(ok = mbar_wait(&y_empty, (j & 1) ^ 1, &abort_flag))) break;  // tile j-1 drained
                    tc_fence_after();
                    const uint32_t ta = tA0 + (ac % kASlots) * 64;
                    const uint64_t dB = dRing0 + ((s * kTile) >> 4);
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) mma_ts(tD1, ta + kk * 8, dB + off128[kk], idKm, kk > 0);
                    mma_commit(&g_full);
                    mma_commit(&ring_empty[s]);
                    mma_commit(&a_empty[ac % kASlots]);
                }
                bool used = false;
                for (int k = me; k < groups; k += 2) {
                    const uint32_t rk = g + 1 + k, ak = ac + 1 + k;
                    const int s = rk % kRing;
                    if (!(ok = mbar_wait(&ring_full[s], (rk / kRing) & 1, &abort_flag))) break;
                    if (!(ok = mbar_wait(&a_full[ak % kASlots], (ak / kASlots) & 1, &abort_flag))) break;
                    if (!used) {
                        // D0: tile j-1 drained; D1: G has been read by the aux warps
                        if (me == 0 && !(ok = mbar_wait(&y_empty, (j & 1) ^ 1, &abort_flag))) break;
                        if (me == 1 && !(ok = mbar_wait(&g_done, j & 1, &abort_flag))) break;
                    }
                    tc_fence_after();
                    const uint32_t ta = tA0 + (ak % kASlots) * 64;
                    const uint32_t acc0 = used ? 1u : 0u;
                    if (k == groups - 1) {  // P V: the V operand is MN-major, a K step is 16 rows
                        const uint64_t dB = dRingMN + ((s * kTile) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) mma_ts(tD, ta + kk * 8, dB + kk * (2048u >> 4), idPV, acc0 | (kk > 0));
                    } else {
                        const uint64_t dB = dRing0 + ((s * kTile) >> 4);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk) mma_ts(tD, ta + kk * 8, dB + off128[kk], idKm, acc0 | (kk > 0));
                    }
                    mma_commit(&ring_empty[s]);
                    mma_commit(&a_empty[ak % kASlots]);
                    used = true;
                }
                if (!ok) break;
                mma_commit(&y_full);  // both issuers commit: the tile's sum is complete
                g += 1 + groups;
                ac += 1 + groups;
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
            if (!mbar_wait(&a_empty[ac % kASlots], ((ac / kASlots) & 1) ^ 1, &abort_flag)) return false;
            tc_fence_after();
            const uint32_t ta = tA0 + (ac % kASlots) * 64 + lane_base;
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
            mbar_arrive(&a_full[ac % kASlots]);
            ++ac;
            return true;
        };
        for (int j = 0; j < my_tiles && ok; ++j) {
            const TileInfo t = decode_tile(a, tile_id(j));
            const size_t tok = (size_t)t.bh * a.L + (size_t)t.n * a.C + (size_t)t.c * kCT + row;
            uint32_t gm2[32];  // gates g_{t,i} as bf16 pairs (i even: low half); g_{t,n} at 63
            if (GATED) {
                const uint4 *gsrc = reinterpret_cast<const uint4 *>(a.gam + tok * 64);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint4 x = __ldg(gsrc + i);
                    gm2[4 * i] = x.x;
                    gm2[4 * i + 1] = x.y;
                    gm2[4 * i + 2] = x.z;
                    gm2[4 * i + 3] = x.w;
                }
            }
            uint32_t qp[64];  // the token's query row, bf16 pairs
            {
                const uint4 *src = reinterpret_cast<const uint4 *>(a.q + tok * kD);
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
            // g_n o Q: A operand of G and of the prefix state
            __nv_bfloat162 gon2 = one2;
            if (GATED) gon2 = __high2bfloat162(*reinterpret_cast<const __nv_bfloat162 *>(&gm2[31]));
            if (!(ok = put_a(qp, gon2, GATED))) break;                  // for G
            if (t.c > 0 && !(ok = put_a(qp, gon2, GATED))) break;      // for the prefix state
            if (GATED) {
                // Rolled loop (one copy of put_a keeps the code small); the gate of
                // segment i comes from a small per-thread array.
                const __nv_bfloat16 *gl = reinterpret_cast<const __nv_bfloat16 *>(gm2);
#pragma unroll 1
                for (int i = 0; i < t.n; ++i) {
                    if (!(ok = put_a(qp, __bfloat162bfloat162(gl[i]), true))) break;
                }
                if (!ok) break;
            } else if (t.n > 0) {
                if (!(ok = put_a(qp, one2, false))) break;
            }
            // The tile's last A slot carries P.  The A warps claim it in order (so
            // every wait on a slot stays within one phase of its barrier) and hand it
            // to the aux warps, after the previous tile's P has been written.
            if (j > 0 && !(ok = mbar_wait(&p_written, (j - 1) & 1, &abort_flag))) break;
            if (!(ok = mbar_wait(&a_empty[ac % kASlots], ((ac / kASlots) & 1) ^ 1, &abort_flag))) break;
            mbar_arrive(&p_slot);
            ++ac;
        }
    } else {
        // ---------------------------------------------------------- aux: P, drain
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        bool ok = true;
        uint32_t ac = 0;  // A-slot counter, kept in step with the A warps and the MMA warp
        for (int j = 0; j < my_tiles && ok; ++j) {
            const TileInfo t = decode_tile(a, tile_id(j));
            ac += 1 + (uint32_t)tile_items<GATED>(t);  // the G slot and the cached operands' slots
            // P = mask(G): G already carries the online gate g_n through its A operand
            if (!(ok = mbar_wait(&g_full, j & 1, &abort_flag))) break;
            tc_fence_after();
            uint32_t pk[64];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t x[16], z[16];
                tmem_ld16(tD1 + lane_base + 32 * h, x);
                tmem_ld16(tD1 + lane_base + 32 * h + 16, z);
                tmem_wait_ld();
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t c0 = 32 * h + 2 * i, c1 = c0 + 16;
                    pk[16 * h + i] = pack_bf16x2(c0 <= row ? __uint_as_float(x[2 * i]) : 0.f,
                                                 c0 + 1 <= row ? __uint_as_float(x[2 * i + 1]) : 0.f);
                    pk[16 * h + 8 + i] = pack_bf16x2(c1 <= row ? __uint_as_float(z[2 * i]) : 0.f,
                                                     c1 + 1 <= row ? __uint_as_float(z[2 * i + 1]) : 0.f);
                }
            }
            tc_fence_before();
            mbar_arrive(&g_done);
            if (!(ok = mbar_wait(&p_slot, j & 1, &abort_flag))) break;  // claimed for us by the A warps
            tc_fence_after();
            {
                const uint32_t ta = tA0 + (ac % kASlots) * 64 + lane_base;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t r[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) r[i] = pk[16 * h + i];
                    tmem_st16(ta + 16 * h, r);
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&a_full[ac % kASlots]);
                mbar_arrive(&p_written);
                ++ac;
            }
            // drain: y = D0 (+ D1 when the tile wrote both accumulators)
            const bool both = tile_groups<GATED>(t) >= 2;
            if (!(ok = mbar_wait(&y_full, j & 1, &abort_flag))) break;
            tc_fence_after();
            uint4 *dst = reinterpret_cast<uint4 *>(a.y + ((size_t)t.bh * a.L + (size_t)t.n * a.C + (size_t)t.c * kCT + row) * kD);
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                uint32_t x[16], z[16], x1[16], z1[16];
                tmem_ld16(tD0 + lane_base + 32 * h, x);
                tmem_ld16(tD0 + lane_base + 32 * h + 16, z);
                if (both) {
                    tmem_ld16(tD1 + lane_base + 32 * h, x1);
                    tmem_ld16(tD1 + lane_base + 32 * h + 16, z1);
                }
                tmem_wait_ld();
                float f[32];
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    f[i] = __uint_as_float(x[i]) + (both ? __uint_as_float(x1[i]) : 0.f);
                    f[16 + i] = __uint_as_float(z[i]) + (both ? __uint_as_float(z1[i]) : 0.f);
                }
                uint32_t o[16];
#pragma unroll
                for (int i = 0; i < 16; ++i) o[i] = pack_bf16x2(f[2 * i], f[2 * i + 1]);
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[4 * h + i] = make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]);
            }
            tc_fence_before();
            mbar_arrive(&y_empty);
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
           (p.mode == MC_GRM || p.mode == MC_SOUP || p.mode == MC_RESIDUAL ||
            (p.mode == MC_SSC && p.topk >= 0 && p.topk <= kTcMaxTopk));
}

size_t tc_scratch_bytes(const Problem &p)
{
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT;
    size_t b = pad256(BH * N * kTile) + pad256(BH * N * CPS * kTile) + pad256(BH * kTile) +
               pad256(sizeof(float) * BH * p.L);
    if (p.mode == MC_RESIDUAL)
        b += pad256(BH * N * kTile);  // prefix sums of the states
    else
        b += pad256(sizeof(__nv_bfloat16) * BH * p.L * 64);  // gates
    return b;
}

// SSC router alone (mc_ssc_select) on the tensor-core path's shapes: key-mean
// images, then the SSC gates kernel with only the router output enabled.
size_t tc_select_scratch_bytes(const Problem &p) { return pad256((size_t)p.BH * kTile); }

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
    CUtensorMap mU;
    if (!make_tmap_bf16_sw128(&mU, fa.u, (unsigned long long)p.BH * p.L, kD, 128)) return cudaErrorInvalidValue;
    if (g_num_sms == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&g_num_sms, cudaDevAttrMultiProcessorCount, dev);
        if (g_num_sms <= 0) g_num_sms = 148;
    }
    cudaError_t e = cudaMemsetAsync(a.kbar_img, 0, (size_t)p.BH * kTile, s);
    if (e != cudaSuccess) return e;
    kbar_images_tc<<<(unsigned)(p.BH * p.N), kD, 0, s>>>(static_cast<const __nv_bfloat16 *>(fa.k), a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    e = cudaFuncSetAttribute(gates_tc<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGatesSmem);
    if (e != cudaSuccess) return e;
    const int gtiles = p.BH * (p.L / kCT);
    const int ggrid = gtiles < 2 * g_num_sms ? gtiles : 2 * g_num_sms;
    gates_tc<true><<<ggrid, kGatesThreads, kGatesSmem, s>>>(mU, a);
    return cudaGetLastError();
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
    a.gam = gated ? reinterpret_cast<__nv_bfloat16 *>(base) : nullptr;
    a.sel_out = fa.sel_out;
    a.topk = p.topk;
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
    } else {
        auto kg = p.mode == MC_SSC ? gates_tc<true> : gates_tc<false>;
        e = cudaFuncSetAttribute(kg, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGatesSmem);
        if (e != cudaSuccess) return e;
        const int gtiles = (int)(BH * (p.L / kCT));
        const int ggrid = gtiles < 2 * g_num_sms ? gtiles : 2 * g_num_sms;
        kg<<<ggrid, kGatesThreads, kGatesSmem, s>>>(mU, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "gates_tc");
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
