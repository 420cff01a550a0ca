// k_gen.cu -- the general tensor-core path of the Memory Caching forward (bf16, d = 64
// or 128): any segment length that is a multiple of 16 tokens, any sequence length
// (a ragged last segment), up to 512 segments; and the factorised form of the cached
// readout.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
//
// For a linear memory every read is linear in the memory, so the aggregation
//     y_t = sum_{i < s} g_{t,i} M^(i) q_t + g_{t,s} M_t^(s) q_t      ([MC-ja §3.1 eq. 9])
// regroups by token: M^(i) = sum_{j in i} v_j k_j^T ([MC-ja §3 eq. 4b]), so
//     y_t = sum_{j <= t} g_{t, seg(j)} v_j (k_j . q_t),
// the factorised form: an attention-like product with one weight per (token, segment)
// instead of a softmax.  Its cost per token is 4 d t against the state form's
// 2 d^2 (s - 1) + 4 d^2, so it wins when segments are shorter than d / 2 ([MC-sum §2.2]:
// the read is O(N) per token and the segment length sets N).  Three kernels:
//
// seg_piece_tc -- persistent; walks every head in units of lcm(C, 128) tokens (a unit
//   starts on both a segment and a 128-token chunk boundary).  Per chunk, the pieces
//   (a segment's tokens inside the chunk, whole 16-token steps) each get
//     Z = V_p^T K_p  (tcgen05, fp32 in tensor memory)
//   added to the running state of their segment; at a segment's end the state (fp32,
//   the `states` output) and its key mean (the key-mean image, hi + mid + lo rows) are
//   written.  With the routed aggregations it also forms the online score
//     r_on[t] = <u_t, sum_{j = t0..t} k_j> / (t - t0 + 1)
//   from R = U K^T masked to the token's piece, plus <u_t, keys of the segment before
//   the chunk>.
//
// gates_tc -- the gates of every token as bf16 gates[bh][i][t] (i < s cached, i = s
//   the online memory): the scores <u_t, kbar_i> on the tensor cores (kbar as hi + mid +
//   lo rows, so each score is an fp32 sum of exact products), then a softmax over the
//   cached scores and r_on (GRM; Soup is the same sum for a linear memory [MC-sum §3.3])
//   or the topk largest cached scores, equal scores to the lower index, and a softmax
//   over those and r_on ([MC-sum §3.4]); unselected segments get gate 0.
//
// readout_fact_tc -- per 128-token query tile, over every key tile up to it:
//     G = Q K^T;  P = w o mask(G), w_{t,j} = g_{t, seg(j)};  D += P V
//   (Residual: w = 1, which is causal linear attention, the collapse of [MC-ja §3.1
//   eq. 7]; Mean: w = 1 / (s + 1)).  Two CTAs per SM share the tensor pipe.
#include <cstdint>

#include "mc_internal.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"
#include "tensormap.cuh"

namespace mc {

// Set by any kernel of this file that abandoned its work after a bounded wait ran out;
// read and cleared by take_gen_abort().
__device__ int g_gen_abort;

namespace {

using namespace sm100;

struct GenArgs {
    float *states;         // [BH][N][d][d] fp32 output, or null
    uint8_t *kbar_img;     // [BH][NB] x kKbImg key-mean images
    float *r_on;           // [BH][Lp] online scores
    __nv_bfloat16 *gates;  // [BH][N][Lp] gates (routed aggregations)
    __nv_bfloat16 *y;      // [BH][L][d]
    int32_t *sel_out;      // optional SSC router output [BH][L][topk] (rank order, -1 padded)
    int BH, L, Lp, d, C, N, NB, topk;
    int UL;                // unit length of seg_piece_tc in tokens (a multiple of 128)
    int units;             // units per head
    int mean;              // readout weights 1 / (s + 1)
};

// ============================================================================
// seg_piece_tc
// ============================================================================
constexpr int kPThreads = 192;              // warp 0 TMA, warp 1 MMA, warps 2-5 workers
constexpr uint32_t kPStage = 3 * kTile;     // K, V, U tiles of one chunk
constexpr uint32_t kPStaging = 4096;        // per worker warp: 32 rows x 128 bytes of a store in flight
constexpr size_t kPSmem = 2 * kPStage + 4 * kPStaging + 1024;

struct Piece {
    int seg, a, b;  // segment, tokens [a, b) of the head inside the chunk
};

// Pieces of the chunk [T0, T1): segment sp covers [sp C, (sp + 1) C).
__device__ __forceinline__ Piece piece_of(int T0, int T1, int C, int p)
{
    Piece x;
    x.seg = T0 / C + p;
    x.a = max(x.seg * C, T0);
    x.b = min((x.seg + 1) * C, T1);
    return x;
}

template <bool GATED>
__global__ void __launch_bounds__(kPThreads, 1)
    seg_piece_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                 const __grid_constant__ CUtensorMap mU, GenArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t full[2], empty[2], r_full[2], r_empty[2], z_full[2], z_empty[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ __align__(16) float ksum_s[kD];     // keys of the segment that continues into this chunk
    __shared__ __align__(16) float red_s[8][kD];   // column sums of the chunk's 16-row groups

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int total_units = a.BH * a.units;
    // This CTA's chunks form one stream: units blockIdx.x, blockIdx.x + gridDim.x, ...,
    // each walked in order.  Unit u of head bh covers tokens [u UL, min((u + 1) UL, L)).
    auto unit_chunks = [&](int unit) {
        const int u0 = (unit % a.units) * a.UL;
        return (min(u0 + a.UL, a.L) - u0 + kCT - 1) / kCT;
    };

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
        mbar_init(&fin, 1);
        fence_mbar_init();
    }
    if (threadIdx.x < kD) ksum_s[threadIdx.x] = 0.f;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tR0 = tb, tZ0 = tb + 256;  // R x 2 | Z x 2, 128 columns each

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            if (GATED) prefetch_tensormap(&mU);
            uint32_t gch = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < total_units && ok; unit += gridDim.x) {
                const int bh = unit / a.units, u0 = (unit % a.units) * a.UL;
                const int nch = unit_chunks(unit);
                for (int c = 0; c < nch; ++c, ++gch) {
                    const int s = gch & 1;
                    const uint32_t r = gch >> 1;
                    if (!(ok = mbar_wait(&empty[s], (r & 1) ^ 1, &abort_flag))) break;
                    uint8_t *st = sm + s * kPStage;
                    const int T0 = u0 + c * kCT;
                    mbar_arrive_expect_tx(&full[s], GATED ? 3 * kTile : 2 * kTile);
                    tma_load_3d(st, &mK, 0, T0, bh, &full[s]);
                    tma_load_3d(st + kPanel, &mK, 64, T0, bh, &full[s]);
                    tma_load_3d(st + kTile, &mV, 0, T0, bh, &full[s]);
                    tma_load_3d(st + kTile + kPanel, &mV, 64, T0, bh, &full[s]);
                    if (GATED) {
                        tma_load_3d(st + 2 * kTile, &mU, 0, T0, bh, &full[s]);
                        tma_load_3d(st + 2 * kTile + kPanel, &mU, 64, T0, bh, &full[s]);
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idR = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idS = idesc_bf16(128, 128, true, true);
            uint32_t gch = 0, pc = 0;
            bool ok = true;
            for (int unit = blockIdx.x; unit < total_units && ok; unit += gridDim.x) {
                const int u0 = (unit % a.units) * a.UL;
                const int nch = unit_chunks(unit);
                for (int c = 0; c < nch && ok; ++c, ++gch) {
                    const int s = gch & 1, b = gch & 1;
                    const uint32_t r = gch >> 1;
                    if (!(ok = mbar_wait(&full[s], r & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint32_t kb = smem_u32(sm + s * kPStage), vb = kb + kTile, ub = kb + 2 * kTile;
                    if (GATED) {  // R = U K^T: the chunk's <u_t, k_j>
                        if (!(ok = mbar_wait(&r_empty[b], (r & 1) ^ 1, &abort_flag))) break;
                        tc_fence_after();
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(tR0 + b * 128, make_desc_sw128(ub + kmaj_off(kk, 128), 0, 1024),
                                   make_desc_sw128(kb + kmaj_off(kk, 128), 0, 1024), idR, kk > 0);
                        mma_commit(&r_full[b]);
                    }
                    const int T0 = u0 + c * kCT, T1 = min(T0 + kCT, a.L);
                    const int np = (T1 - 1) / a.C - T0 / a.C + 1;
                    for (int p = 0; p < np; ++p, ++pc) {  // Z = V_p^T K_p, the piece's own state
                        const Piece x = piece_of(T0, T1, a.C, p);
                        const int zb = pc & 1;
                        if (!(ok = mbar_wait(&z_empty[zb], ((pc >> 1) & 1) ^ 1, &abort_flag))) break;
                        tc_fence_after();
                        const int k0 = (x.a - T0) >> 4, k1 = (x.b - T0 + 15) >> 4;
                        for (int kk = k0; kk < k1; ++kk)
                            mma_ss(tZ0 + zb * 128, make_desc_sw128(vb + kk * 2048u, kPanel, 1024),
                                   make_desc_sw128(kb + kk * 2048u, kPanel, 1024), idS, kk > k0);
                        mma_commit(&z_full[zb]);
                    }
                    if (ok) mma_commit(&empty[s]);
                }
            }
            // leave no MMA in flight
            mma_commit(&fin);
            int give_up = 0;
            mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
        }
    } else {
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;  // token row (R) = value row (Z, S) = key column (sums)
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint8_t *wst = sm + 2 * kPStage + q4 * kPStaging;
        float S[kD];       // running state row of the segment: S[row][k] = sum v_j[row] k_j[k]
        float ks = 0.f;    // running key sum (column `row`) of the segment
        uint32_t gch = 0, pc = 0;
        bool ok = true;
        for (int unit = blockIdx.x; unit < total_units; unit += gridDim.x) {
            const int bh = unit / a.units, u0 = (unit % a.units) * a.UL;
            const int nch = unit_chunks(unit);
            for (int c = 0; c < nch; ++c, ++gch) {
                const int s = gch & 1, b = gch & 1;
                const uint32_t r = gch >> 1;
                const int T0 = u0 + c * kCT, T1 = min(T0 + kCT, a.L);
                const int np = (T1 - 1) / a.C - T0 / a.C + 1;
                if (ok) ok = mbar_wait(&full[s], r & 1, &abort_flag);
                const uint8_t *st = sm + s * kPStage;
                // column sums of the chunk's 16-row groups (rows past L are zero)
                if (ok) {
                    const int cc = row & 15, rg = row >> 4;
                    float p8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint4 x = *reinterpret_cast<const uint4 *>(st + sw128_offset(16 * rg + i, 8 * cc, 128));
                        const float2 k01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.x));
                        const float2 k23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.y));
                        const float2 k45 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.z));
                        const float2 k67 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.w));
                        p8[0] += k01.x; p8[1] += k01.y; p8[2] += k23.x; p8[3] += k23.y;
                        p8[4] += k45.x; p8[5] += k45.y; p8[6] += k67.x; p8[7] += k67.y;
                    }
                    *reinterpret_cast<float4 *>(&red_s[rg][8 * cc]) = make_float4(p8[0], p8[1], p8[2], p8[3]);
                    *reinterpret_cast<float4 *>(&red_s[rg][8 * cc + 4]) = make_float4(p8[4], p8[5], p8[6], p8[7]);
                }
                if (GATED) {  // the online score of token T0 + row
                    const int t = T0 + (int)row;
                    const int sp = min(t, a.L - 1) / a.C;  // its segment
                    const int pa = max(sp * a.C, T0) - T0;  // first chunk row of its piece
                    float dot = 0.f;
                    if (ok && sp * a.C < T0) {  // the segment began before the chunk: its earlier keys
                        float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
                        for (int cc = 0; cc < 16; ++cc) {
                            const uint4 x = *reinterpret_cast<const uint4 *>(st + 2 * kTile + sw128_offset(row, 8 * cc, 128));
                            const float4 k0 = *reinterpret_cast<const float4 *>(&ksum_s[8 * cc]);
                            const float4 k1 = *reinterpret_cast<const float4 *>(&ksum_s[8 * cc + 4]);
                            const float2 u01 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.x));
                            const float2 u23 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.y));
                            const float2 u45 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.z));
                            const float2 u67 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&x.w));
                            float &dd = d4[cc & 3];
                            dd = fmaf(u01.x, k0.x, dd); dd = fmaf(u01.y, k0.y, dd);
                            dd = fmaf(u23.x, k0.z, dd); dd = fmaf(u23.y, k0.w, dd);
                            dd = fmaf(u45.x, k1.x, dd); dd = fmaf(u45.y, k1.y, dd);
                            dd = fmaf(u67.x, k1.z, dd); dd = fmaf(u67.y, k1.w, dd);
                        }
                        dot = (d4[0] + d4[1]) + (d4[2] + d4[3]);
                    }
                    if (ok) ok = mbar_wait(&r_full[b], r & 1, &abort_flag);
                    if (ok) {
                        tc_fence_after();
                        float w4[4] = {0.f, 0.f, 0.f, 0.f};  // sum_{j in the piece, j <= t} <u_t, k_j>
#pragma unroll
                        for (int j16 = 0; j16 < 8; ++j16) {
                            if (16 * j16 > 32 * q4 + 31) break;  // columns past the warp's last row are masked
                            uint32_t v[16];
                            tmem_ld16(tR0 + b * 128 + lane_base + 16 * j16, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const int j = 16 * j16 + i;
                                if (j >= pa && j <= (int)row) w4[i & 3] += __uint_as_float(v[i]);
                            }
                        }
                        tc_fence_before();
                        mbar_arrive(&r_empty[b]);
                        if (t < a.L)
                            a.r_on[(size_t)bh * a.Lp + t] = (dot + (w4[0] + w4[1]) + (w4[2] + w4[3])) / (float)(t - sp * a.C + 1);
                    }
                }
                named_bar_sync(1, 128);  // red_s complete; ksum_s read by every worker
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[s]);  // this warp is done with the stage
                for (int p = 0; p < np; ++p, ++pc) {
                    const Piece x = piece_of(T0, T1, a.C, p);
                    const bool cont = x.seg * a.C < T0;            // the segment began in an earlier chunk
                    const int seg_end = min((x.seg + 1) * a.C, a.L);
                    const bool ends = x.b == seg_end;
                    // key sums of the piece's 16-row groups, in order
                    if (ok) {
                        float cs = 0.f;
                        const int g0 = (x.a - T0) >> 4, g1 = (x.b - T0 + 15) >> 4;
                        for (int g8 = g0; g8 < g1; ++g8) cs += red_s[g8][row];
                        ks = cont ? ks + cs : cs;
                    }
                    const int zb = pc & 1;
                    if (!cont) {  // a new segment: its memory starts from zero
#pragma unroll
                        for (int k = 0; k < kD; ++k) S[k] = 0.f;
                    }
                    if (ok) ok = mbar_wait(&z_full[zb], (pc >> 1) & 1, &abort_flag);
                    if (ok) {
                        tc_fence_after();
#pragma unroll
                        for (int j16 = 0; j16 < 8; ++j16) {
                            uint32_t v[16];
                            tmem_ld16(tZ0 + zb * 128 + lane_base + 16 * j16, v);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 16; ++i) S[16 * j16 + i] += __uint_as_float(v[i]);
                        }
                        tc_fence_before();
                        mbar_arrive(&z_empty[zb]);
                    }
                    if (ok && ends) {  // the segment's cached state (fp32) and key mean
                        const size_t sidx = (size_t)bh * a.N + x.seg;
                        const int d = a.d;
                        if (a.states) {
                            // fp32 rows (d values), 32 columns (128 bytes) at a time through the staging
                            // area (16-byte chunk c of row r at chunk c ^ (r % 8)), 4 rows per instruction;
                            // with d < 128 the padded rows and columns are not stored
                            float *o = a.states + sidx * d * d + (size_t)(32 * q4) * d;
#pragma unroll
                            for (int blk = 0; blk < 4; ++blk) {
                                if (32 * q4 >= d || 32 * blk >= d) break;  // warp-uniform
#pragma unroll
                                for (int c8 = 0; c8 < 8; ++c8) {
                                    const int e = 32 * blk + 4 * c8;
                                    *reinterpret_cast<float4 *>(wst + lane * 128 + ((c8 ^ (lane & 7)) << 4)) =
                                        make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
                                }
                                __syncwarp();
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    const int rr = 4 * i + (lane >> 3), c8 = lane & 7;
                                    const float4 v = *reinterpret_cast<const float4 *>(wst + rr * 128 + ((c8 ^ (rr & 7)) << 4));
                                    *reinterpret_cast<float4 *>(o + (size_t)rr * d + 32 * blk + 4 * c8) = v;
                                }
                                __syncwarp();
                            }
                        }
                        if (GATED)
                            store_kbar_terms(a.kbar_img + (size_t)bh * a.NB * kKbImg, x.seg, row,
                                             ks / (float)(seg_end - x.seg * a.C));
                    }
                }
                named_bar_sync(1, 128);  // every worker is done with red_s and ksum_s
                if (ok) ksum_s[row] = ks;  // the last piece's segment continues into the next chunk
                named_bar_sync(1, 128);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, 512);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_gen_abort, 1);
}

// ============================================================================
// gates_tc
// ============================================================================
constexpr int kGThreads = 576;                               // warp 0 TMA, warp 1 MMA, warps 2-17 token rows
constexpr int kGParts = 4;                                   // worker warps per quarter of the token rows
constexpr size_t kGSmem = 2 * kTile + 2 * kKbImg + 1024;     // U x 2, key-mean blocks x 2
constexpr int kGMaxN = 512;                                  // cached segments the score columns hold

// Persistent, one CTA per SM over contiguous ranges of (bh, 128-token tile).  Per tile the
// scores against every cached segment its last token sees go to tensor memory (blocks of
// 64 segments, 64 columns each); four worker warps per quarter of the token rows then form
// the gates, each over every fourth 32-column group of scores (GRM: partial maxima and
// sums combined through shared memory; SSC: the first of the four ranks alone).  With
// at most 256 segments two tiles' scores fit, so the next tile's MMAs run while the
// workers read this one's.
template <bool SSC>
__global__ void __launch_bounds__(kGThreads, 1) gates_tc(const __grid_constant__ CUtensorMap mU, GenArgs a)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sU = sm, *sKb = sm + 2 * kTile;
    __shared__ uint64_t u_full[2], u_empty[2], kb_full[2], kb_empty[2], s_full[2], t_free[2], fin;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ float red_m[2][kGParts][kCT], red_z[2][kGParts][kCT];  // per tile parity: partial maxima and sums
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int QT = a.Lp / kCT;
    const int total = a.BH * QT;
    const int per = (total + (int)gridDim.x - 1) / (int)gridDim.x;
    const int first = (int)blockIdx.x * per;
    const int last = min(total, first + per);  // tiles [first, last)
    // cached segments the tile's last token reads, in blocks of 64
    auto tile_blocks = [&](int it) {
        const int T0 = (it % QT) * kCT;
        const int ncached = (min(T0 + kCT, a.L) - 1) / a.C;
        return (ncached + 63) >> 6;
    };
    if (warp == 0) {
        tmem_alloc(&tmem_base, 512);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int i = 0; i < 2; ++i) {
            mbar_init(&u_full[i], 1);
            mbar_init(&u_empty[i], 1);
            mbar_init(&kb_full[i], 1);
            mbar_init(&kb_empty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&s_full[i], 1);
            mbar_init(&t_free[i], 32 * 4 * kGParts);
        }
        mbar_init(&fin, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const int nbuf = (a.N - 1 + 63) / 64 <= 4 ? 2 : 1;  // score buffers of 256 columns, or one of 512
    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mU);
            uint32_t kbc = 0;
            for (int it = first; it < last; ++it) {
                const int i = it - first, ub = i & 1;
                const int bh = it / QT, T0 = (it % QT) * kCT;
                if (!mbar_wait(&u_empty[ub], ((i >> 1) & 1) ^ 1, &abort_flag)) break;
                mbar_arrive_expect_tx(&u_full[ub], kTile);
                tma_load_3d(sU + ub * kTile, &mU, 0, T0, bh, &u_full[ub]);
                tma_load_3d(sU + ub * kTile + kPanel, &mU, 64, T0, bh, &u_full[ub]);
                const int nblk = tile_blocks(it);
                bool ok = true;
                for (int blk = 0; blk < nblk; ++blk, ++kbc) {
                    const int slot = kbc & 1;
                    if (!(ok = mbar_wait(&kb_empty[slot], ((kbc >> 1) & 1) ^ 1, &abort_flag))) break;
                    mbar_arrive_expect_tx(&kb_full[slot], kKbImg);
                    bulk_load(sKb + slot * kKbImg, a.kbar_img + ((size_t)bh * a.NB + blk) * kKbImg, kKbImg, &kb_full[slot]);
                }
                if (!ok) break;
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idS = idesc_bf16(128, 64, false, false);
            uint32_t kbc = 0;
            bool ok = true, issued = false;
            for (int it = first; it < last && ok; ++it) {
                const int i = it - first, ub = i & 1;
                const int sb = i % nbuf, use = i / nbuf;  // score buffer, and its use count
                if (!(ok = mbar_wait(&t_free[sb], (use & 1) ^ 1, &abort_flag))) break;  // its last scores are read
                if (!(ok = mbar_wait(&u_full[ub], (i >> 1) & 1, &abort_flag))) break;
                tc_fence_after();
                const int nblk = tile_blocks(it);
                const uint32_t ts = tb + 256 * sb;
                const uint64_t dU = make_desc_sw128(smem_u32(sU + ub * kTile), 0, 1024);
                for (int blk = 0; blk < nblk; ++blk, ++kbc) {
                    const int slot = kbc & 1;
                    if (!(ok = mbar_wait(&kb_full[slot], (kbc >> 1) & 1, &abort_flag))) break;
                    tc_fence_after();
                    const uint64_t dKb = make_desc_sw128(smem_u32(sKb + slot * kKbImg), 0, 1024);
#pragma unroll
                    for (int term = 0; term < 3; ++term)  // hi, mid, lo
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ss(ts + 64 * blk, dU + (kmaj_off(kk, 128) >> 4),
                                   dKb + ((term * kKbPanel + kmaj_off(kk, 64)) >> 4), idS, (term | kk) != 0);
                    mma_commit(&kb_empty[slot]);
                    issued = true;
                }
                if (!ok) break;
                if (nblk > 0) {
                    mma_commit(&u_empty[ub]);
                    mma_commit(&s_full[sb]);
                } else {  // no cached segment yet: nothing was issued
                    mbar_arrive(&u_empty[ub]);
                    mbar_arrive(&s_full[sb]);
                }
            }
            if (issued) {  // leave no MMA in flight
                mma_commit(&fin);
                int give_up = 0;
                mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
            }
        }
    } else {
        const int q4 = warp & 3;
        const int part = (warp - 2) >> 2;  // every fourth 32-column group of scores, from group `part`
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        // A worker that gives up (a bounded wait ran out) keeps walking the tiles without
        // work so that every worker reaches the same named barriers.
        bool ok = true;
        for (int it = first; it < last; ++it) {
            const int i = it - first;
            const int bh = it / QT, T0 = (it % QT) * kCT;
            const int t = T0 + (int)row;
            const bool valid = t < a.L;
            const int st = min(t, a.L - 1) / a.C;  // cached segments of this token
            const int nblk = tile_blocks(it);
            const float ron = valid ? a.r_on[(size_t)bh * a.Lp + t] : 0.f;
            const int sb = i % nbuf, use = i / nbuf;
            const uint32_t ts = tb + 256 * sb + lane_base;
            if (ok) ok = mbar_wait(&s_full[sb], use & 1, &abort_flag);
            if (!ok) {
                if (!SSC) named_bar_sync(1, 32 * 4 * kGParts);
                continue;
            }
            tc_fence_after();
            __nv_bfloat16 *gcol = a.gates + (size_t)bh * a.N * a.Lp + t;  // gate of segment n at gcol[n Lp]
            const int n32 = 2 * nblk;  // 32-column groups of scores
            if (!SSC) {
                // softmax over the cached scores i < st and the online score: this part's running
                // maximum and sum over its groups, combined with the other parts', then the gates
                float m = -3.402823466e38f, z = 0.f;
                for (int c = part; c < n32; c += kGParts) {
                    uint32_t v[32];
                    tmem_ld32(ts + 32 * c, v);
                    tmem_wait_ld();
                    float mc = m;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (32 * c + e < st) mc = fmaxf(mc, __uint_as_float(v[e]));
                    z *= __expf(m - mc);
                    m = mc;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (32 * c + e < st) z += __expf(__uint_as_float(v[e]) - m);
                }
                red_m[i & 1][part][row] = m;
                red_z[i & 1][part][row] = z;
                named_bar_sync(1, 32 * 4 * kGParts);
                float M = ron;
#pragma unroll
                for (int q = 0; q < kGParts; ++q) M = fmaxf(M, red_m[i & 1][q][row]);
                float Z = __expf(ron - M);
#pragma unroll
                for (int q = 0; q < kGParts; ++q) Z += red_z[i & 1][q][row] * __expf(red_m[i & 1][q][row] - M);
                const float inv = 1.f / Z;
                for (int c = part; c < n32; c += kGParts) {
                    uint32_t v[32];
                    tmem_ld32(ts + 32 * c, v);
                    tmem_wait_ld();
                    if (valid) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (32 * c + e < st)
                                gcol[(size_t)(32 * c + e) * a.Lp] = __float2bfloat16_rn(__expf(__uint_as_float(v[e]) - M) * inv);
                    }
                }
                tc_fence_before();
                mbar_arrive(&t_free[sb]);
                if (valid && part == 0) gcol[(size_t)st * a.Lp] = __float2bfloat16_rn(__expf(ron - M) * inv);
            } else if (part != 0) {  // SSC ranks in the first part alone
                tc_fence_before();
                mbar_arrive(&t_free[sb]);
            } else {
                // the topk largest cached scores (equal scores: lower index first), then a softmax
                // over them and the online score; every other cached segment gets gate 0
                float vals[kTcMaxTopk];
                int idxs[kTcMaxTopk];
                int cnt = 0;
                const int k = min(a.topk, st);
                for (int c = 0; c < n32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(ts + 32 * c, v);
                    tmem_wait_ld();
                    if (k > 0) {
                        for (int e = 0; e < 32; ++e)
                            if (32 * c + e < st) topk_insert(vals, idxs, cnt, k, __uint_as_float(v[e]), 32 * c + e);
                    }
                }
                tc_fence_before();
                mbar_arrive(&t_free[sb]);
                float m = ron;
                for (int c = 0; c < cnt; ++c) m = fmaxf(m, vals[c]);
                float z = __expf(ron - m);
                for (int c = 0; c < cnt; ++c) z += __expf(vals[c] - m);
                const float inv = 1.f / z;
                if (valid) {
                    for (int n = 0; n < st; ++n) gcol[(size_t)n * a.Lp] = __float2bfloat16_rn(0.f);
                    for (int c = 0; c < cnt; ++c) gcol[(size_t)idxs[c] * a.Lp] = __float2bfloat16_rn(__expf(vals[c] - m) * inv);
                    gcol[(size_t)st * a.Lp] = __float2bfloat16_rn(__expf(ron - m) * inv);
                    if (a.sel_out) {
                        int32_t *so = a.sel_out + ((size_t)bh * a.L + t) * a.topk;
                        for (int c = 0; c < a.topk; ++c) so[c] = c < cnt ? idxs[c] : -1;
                    }
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
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_gen_abort, 1);
}

// ============================================================================
// readout_fact_tc
// ============================================================================
constexpr int kFThreads = 320;     // warp 0 TMA, warp 1 MMA issuer, warps 2-9 token rows (two per lane quarter)
constexpr int kFRing = 4;          // 16 KB operand panels in flight (one key tile's K and V)
constexpr uint32_t kFCols = 256;   // tensor memory per CTA: D (d columns) | G (128 columns, P written over it)
constexpr int kFGRing = 4;         // key tiles whose gate rows are staged ahead
constexpr int kFGRows = 9;         // gate rows (segments) one key tile can touch: 128 / 16 + 1
constexpr uint32_t kFGStage = kFGRows * 256;  // 128 bf16 gates of the query tile per row
constexpr size_t kFSmem = 2 * kPanel + kFRing * kPanel + kFGRing * kFGStage + 1024;  // two CTAs per SM

enum { kWRouted = 0, kWOne = 1, kWMean = 2 };

// (w0 x0, w1 x1) rounded to a bf16 pair (x0 in the low half): one packed fp32 multiply and
// one conversion.
__device__ __forceinline__ uint32_t scale_pack(uint32_t x0, uint32_t x1, uint64_t w01)
{
    uint32_t r;
    asm("{\n\t.reg .b64 xx, pp;\n\t.reg .b32 lo, hi;\n\tmov.b64 xx, {%1, %2};\n\tmul.rn.f32x2 pp, xx, %3;\n\t"
        "mov.b64 {lo, hi}, pp;\n\tcvt.rn.bf16x2.f32 %0, hi, lo;\n\t}"
        : "=r"(r)
        : "r"(x0), "r"(x1), "l"(w01));
    return r;
}

__device__ __forceinline__ uint64_t pair_of(float lo, float hi)
{
    return ((uint64_t)__float_as_uint(hi) << 32) | __float_as_uint(lo);
}

// One tile = 128 query tokens of one head; for every key tile kt up to it:
//   G = Q K_kt^T;  P = w o mask(G) (written over G);  D += P V_kt.
// The producer also stages, per key tile, the query tile's gates of the segments the key
// tile touches (rows of 128 bf16) in shared memory.
// Two worker warps share each quarter of the tensor-memory lanes (token rows): warp half h
// turns columns 64h .. 64h + 63 of G into P and writes it over the first 32 of those
// columns (each warp overwrites only what it has read), so keys 64h + 16 kk' .. sit at
// column 64h + 8 kk'.
// Tiles are ordered head by head, the longest first within a head, so the CTAs running
// together share a few heads' keys and values in L2; CTA j takes positions j, 2P - 1 - j,
// 2P + j, ... of that order (P CTAs), which evens out the sums of the tiles' lengths.
template <int DP, int WMODE>
__global__ void __launch_bounds__(kFThreads, 2)
    readout_fact_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
                    const __grid_constant__ CUtensorMap mV, GenArgs a)
{
    constexpr int NP = DP / 64;  // 64-column panels of a row of q, k, v
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    uint8_t *sQ = sm, *sR = sm + 2 * kPanel;
    __shared__ uint64_t ring_full[kFRing], ring_empty[kFRing], gr_full[kFGRing], gr_empty[kFGRing];
    __shared__ uint64_t q_full, q_empty, g_full, p_full, g_free, y_full, y_empty, fin;
    uint8_t *sGr = sm + 2 * kPanel + kFRing * kPanel;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int QT = (a.L + kCT - 1) / kCT;
    const int ntiles = a.BH * QT;
    const int P = gridDim.x, j0 = blockIdx.x;
    // position of this CTA's n-th tile in the order (snake over rounds of P)
    auto pos_of = [&](int n) { return n * P + ((n & 1) ? P - 1 - j0 : j0); };
    auto tile_of = [&](int id, int &bh, int &qt) {
        bh = id / QT;
        qt = QT - 1 - id % QT;
    };
    // the query tile's last segment, and the gate rows [i0, i1] key tile kt needs
    auto gate_rows = [&](int qt, int kt, int &i0, int &i1) {
        const int smax = (min(qt * kCT + kCT, a.L) - 1) / a.C;
        i0 = kt * kCT / a.C;
        i1 = min((kt * kCT + kCT - 1) / a.C, smax);
    };
    if (warp == 0) {
        tmem_alloc(&tmem_base, kFCols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int s = 0; s < kFRing; ++s) {
            mbar_init(&ring_full[s], 1);
            mbar_init(&ring_empty[s], 1);
        }
        for (int s = 0; s < kFGRing; ++s) {
            mbar_init(&gr_full[s], 1);
            mbar_init(&gr_empty[s], 8);  // one arrive per worker warp
        }
        mbar_init(&q_full, 1);
        mbar_init(&q_empty, 1);
        mbar_init(&g_full, 1);
        mbar_init(&p_full, 256);
        mbar_init(&g_free, 1);
        mbar_init(&y_full, 1);
        mbar_init(&y_empty, 256);
        mbar_init(&fin, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tD = tb, tG = tb + 128;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mQ);
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            uint32_t g = 0, qc = 0, kc = 0;
            bool ok = true;
            auto slot = [&]() -> uint8_t * {
                const int s = g % kFRing;
                if (!mbar_wait(&ring_empty[s], ((g / kFRing) & 1) ^ 1, &abort_flag)) return nullptr;
                mbar_arrive_expect_tx(&ring_full[s], kPanel);
                return sR + s * kPanel;
            };
            for (int n = 0; pos_of(n) < ntiles && ok; ++n, ++qc) {
                int bh, qt;
                tile_of(pos_of(n), bh, qt);
                if (!(ok = mbar_wait(&q_empty, (qc & 1) ^ 1, &abort_flag))) break;
                mbar_arrive_expect_tx(&q_full, NP * kPanel);
                for (int h = 0; h < NP; ++h) tma_load_3d(sQ + h * kPanel, &mQ, 64 * h, qt * kCT, bh, &q_full);
                for (int kt = 0; kt <= qt && ok; ++kt, ++kc) {
                    uint8_t *dst;
                    if (WMODE == kWRouted) {  // the gate rows of this key tile
                        const int gs = kc % kFGRing;
                        if (!(ok = mbar_wait(&gr_empty[gs], ((kc / kFGRing) & 1) ^ 1, &abort_flag))) break;
                        int i0, i1;
                        gate_rows(qt, kt, i0, i1);
                        mbar_arrive_expect_tx(&gr_full[gs], (uint32_t)(i1 - i0 + 1) * 256u);
                        for (int i = i0; i <= i1; ++i)
                            bulk_load(sGr + gs * kFGStage + (i - i0) * 256,
                                      a.gates + ((size_t)bh * a.N + i) * a.Lp + (size_t)qt * kCT, 256u, &gr_full[gs]);
                    }
                    for (int h = 0; h < NP && ok; ++h) {  // K panels
                        if (!(ok = (dst = slot()) != nullptr)) break;
                        tma_load_3d(dst, &mK, 64 * h, kt * kCT, bh, &ring_full[g % kFRing]);
                        ++g;
                    }
                    if (DP == 128) {
                        for (int h = 0; h < 2 && ok; ++h) {  // keys 64h .. 64h + 63, both 64-wide halves of v
                            if (!(ok = (dst = slot()) != nullptr)) break;
                            tma_load_3d(dst, &mV, 0, kt * kCT + 64 * h, bh, &ring_full[g % kFRing]);
                            tma_load_3d(dst + kPanel / 2, &mV, 64, kt * kCT + 64 * h, bh, &ring_full[g % kFRing]);
                            ++g;
                        }
                    } else {  // all 128 keys, the 64 columns of v
                        if (!(ok = (dst = slot()) != nullptr)) break;
                        tma_load_3d(dst, &mV, 0, kt * kCT, bh, &ring_full[g % kFRing]);
                        ++g;
                    }
                }
            }
            // leave no copy in flight
            int give_up = 0;
            for (uint32_t i = 0; i < (uint32_t)kFRing && i < g; ++i) {
                const uint32_t u = g - 1 - i;
                mbar_wait_limit(&ring_full[u % kFRing], (u / kFRing) & 1, &give_up, kWaitLimitNs);
            }
            if (WMODE == kWRouted)
                for (uint32_t i = 0; i < (uint32_t)kFGRing && i < kc; ++i) {
                    const uint32_t u = kc - 1 - i;
                    mbar_wait_limit(&gr_full[u % kFGRing], (u / kFGRing) & 1, &give_up, kWaitLimitNs);
                }
            if (qc > 0) mbar_wait_limit(&q_full, (qc - 1) & 1, &give_up, kWaitLimitNs);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idG = idesc_bf16(128, 128, false, false);  // Q, K both K-major
            constexpr uint32_t idPV = idesc_bf16(128, DP, false, true);   // V MN-major
            uint32_t g = 0, qc = 0, gc = 0, yc = 0;
            bool ok = true;
            auto ring_ready = [&](uint32_t u) { return mbar_wait(&ring_full[u % kFRing], (u / kFRing) & 1, &abort_flag); };
            const uint32_t sQb = smem_u32(sQ), sRb = smem_u32(sR);
            for (int n = 0; pos_of(n) < ntiles && ok; ++n, ++qc, ++yc) {
                int bh, qt;
                tile_of(pos_of(n), bh, qt);
                if (!(ok = mbar_wait(&q_full, qc & 1, &abort_flag))) break;
                for (int kt = 0; kt <= qt && ok; ++kt, ++gc) {
                    if (!(ok = mbar_wait(&g_free, (gc & 1) ^ 1, &abort_flag))) break;  // P of the previous key tile read
                    tc_fence_after();
                    for (int h = 0; h < NP; ++h) {  // G = Q K^T
                        if (!(ok = ring_ready(g + h))) break;
                        tc_fence_after();
                        const uint64_t dq = make_desc_sw128(sQb + h * kPanel, 0, 1024);
                        const uint64_t dk = make_desc_sw128(sRb + ((g + h) % kFRing) * kPanel, 0, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) mma_ss(tG, dq + 2 * kk, dk + 2 * kk, idG, (h | kk) != 0);
                    }
                    if (!ok) break;
                    for (int h = 0; h < NP; ++h) mma_commit(&ring_empty[(g + h) % kFRing]);
                    g += NP;
                    mma_commit(&g_full);
                    if (kt == qt) mma_commit(&q_empty);
                    if (!(ok = mbar_wait(&p_full, gc & 1, &abort_flag))) break;
                    if (kt == 0 && !(ok = mbar_wait(&y_empty, (yc & 1) ^ 1, &abort_flag))) break;  // D drained
                    tc_fence_after();
                    if (DP == 128) {
                        for (int h = 0; h < 2; ++h) {  // D += P V, keys 64h .. 64h + 63
                            if (!(ok = ring_ready(g))) break;
                            tc_fence_after();
                            const uint64_t dv = make_desc_sw128(sRb + (g % kFRing) * kPanel, kPanel / 2, 1024);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ts(tD, tG + 64 * h + 8 * kk, dv + kk * (2048u >> 4), idPV, (kt | h | kk) != 0);
                            mma_commit(&ring_empty[g % kFRing]);
                            ++g;
                        }
                    } else {
                        if (!(ok = ring_ready(g))) break;
                        tc_fence_after();
                        const uint64_t dv = make_desc_sw128(sRb + (g % kFRing) * kPanel, 0, 1024);
#pragma unroll
                        for (int kk = 0; kk < 8; ++kk)
                            mma_ts(tD, tG + 64 * (kk >> 2) + 8 * (kk & 3), dv + kk * (2048u >> 4), idPV, (kt | kk) != 0);
                        mma_commit(&ring_empty[g % kFRing]);
                        ++g;
                    }
                    if (!ok) break;
                    mma_commit(&g_free);
                }
                if (!ok) break;
                mma_commit(&y_full);
            }
            mma_commit(&fin);
            int give_up = 0;
            mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
        }
    } else {
        const int q4 = warp & 3;
        const int half = (warp - 2) >> 2;  // columns 64 half .. 64 half + 63 of G; column half of D
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        uint32_t gc = 0, yc = 0;
        bool ok = true;
        for (int n = 0; pos_of(n) < ntiles && ok; ++n, ++yc) {
            int bh, qt;
            tile_of(pos_of(n), bh, qt);
            const int t = qt * kCT + (int)row;
            const bool valid = t < a.L;
            const int st = min(t, a.L - 1) / a.C;  // the token's segment
            const float wmean = valid ? (WMODE == kWMean ? 1.f / (float)(st + 1) : 1.f) : 0.f;
            for (int kt = 0; kt <= qt && ok; ++kt, ++gc) {
                // weights of this warp's 64 columns, per 32-column block: segment sa up to
                // column bnd, then segment sa + 1 (segments are whole 16-token steps)
                float ga[2], gb[2];
                int bnd[2];
                int i0 = 0, i1 = 0;
                const __nv_bfloat16 *grow = nullptr;
                if (WMODE == kWRouted) {
                    const int gs = gc % kFGRing;
                    gate_rows(qt, kt, i0, i1);
                    if (!(ok = mbar_wait(&gr_full[gs], (gc / kFGRing) & 1, &abort_flag))) break;
                    grow = reinterpret_cast<const __nv_bfloat16 *>(sGr + gs * kFGStage) + row;
                }
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    const int j0 = kt * kCT + 64 * half + 32 * h;
                    const int sa = j0 / a.C;
                    bnd[h] = min(32, (sa + 1) * a.C - j0);
                    if (WMODE == kWRouted) {
                        ga[h] = valid ? __bfloat162float(grow[(min(sa, st) - i0) * kCT]) : 0.f;
                        gb[h] = valid && bnd[h] < 32 ? __bfloat162float(grow[(min(sa + 1, st) - i0) * kCT]) : ga[h];
                    } else {
                        ga[h] = gb[h] = wmean;
                    }
                }
                if (WMODE == kWRouted) {  // the gate rows are in registers: hand the stage back
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&gr_empty[gc % kFGRing]);
                }
                if (!(ok = mbar_wait(&g_full, gc & 1, &abort_flag))) break;
                tc_fence_after();
                uint32_t x[64];
                tmem_ld32(tG + lane_base + 64 * half, *reinterpret_cast<uint32_t(*)[32]>(x));
                tmem_ld32(tG + lane_base + 64 * half + 32, *reinterpret_cast<uint32_t(*)[32]>(x + 32));
                tmem_wait_ld();
                const int rel = (int)row - 64 * half;  // columns c <= rel are at or before the token
                if (kt < qt) {  // every key precedes the token
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t o[16];
                        const uint64_t wa = pair_of(ga[h], ga[h]), wb = pair_of(gb[h], gb[h]);
#pragma unroll
                        for (int i = 0; i < 16; ++i)  // bnd is a multiple of 16: a pair never straddles it
                            o[i] = scale_pack(x[32 * h + 2 * i], x[32 * h + 2 * i + 1], 2 * i < bnd[h] ? wa : wb);
                        tmem_st16(tG + lane_base + 64 * half + 16 * h, o);  // P over G columns this warp has read
                    }
                } else {  // the diagonal tile: keys after the token are masked
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        uint32_t o[16];
                        const uint64_t wa = pair_of(ga[h], ga[h]), wb = pair_of(gb[h], gb[h]);
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const int c0 = 32 * h + 2 * i;
                            const uint32_t pk = scale_pack(x[c0], x[c0 + 1], 2 * i < bnd[h] ? wa : wb);
                            o[i] = c0 + 1 <= rel ? pk : (c0 <= rel ? (pk & 0xffffu) : 0u);
                        }
                        tmem_st16(tG + lane_base + 64 * half + 16 * h, o);
                    }
                }
                tmem_wait_st();
                tc_fence_before();
                mbar_arrive(&p_full);
            }
            if (!ok) break;
            // drain this warp's column half of D: the 16x256b layout (a quad of threads holds
            // 8 consecutive columns of a row), then a 4 x 4 transpose within the quad so that
            // every thread stores 16 contiguous bytes
            if (!(ok = mbar_wait(&y_full, yc & 1, &abort_flag))) break;
            tc_fence_after();
            const bool drains = half < NP;
            uint32_t yb[32];
            if (drains) {
#pragma unroll
                for (int hl = 0; hl < 2; ++hl) {
                    uint32_t x[32];
                    tmem_ld_16x256b_x8(tD + ((uint32_t)(32 * q4 + 16 * hl) << 16) + 64 * half, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int b = 0; b < 8; ++b) {
                        yb[16 * hl + b] = pack_bf16x2(__uint_as_float(x[4 * b]), __uint_as_float(x[4 * b + 1]));
                        yb[16 * hl + 8 + b] = pack_bf16x2(__uint_as_float(x[4 * b + 2]), __uint_as_float(x[4 * b + 3]));
                    }
                }
            }
            tc_fence_before();
            mbar_arrive(&y_empty);
            if (drains) {
                const int c = lane & 3;
                __nv_bfloat16 *ytile = a.y + ((size_t)bh * a.L + (size_t)qt * kCT) * DP;
#pragma unroll
                for (int g4 = 0; g4 < 8; ++g4) {  // (lane half, row A/B, block group) groups of 4 pairs
                    const int hl = g4 >> 2, rb = (g4 >> 1) & 1, bg = g4 & 1;
                    uint32_t *xv = yb + 4 * g4;
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const uint32_t send = (c & 2) ? xv[k2] : xv[k2 + 2];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 2);
                        if (c & 2) xv[k2] = recv; else xv[k2 + 2] = recv;
                    }
#pragma unroll
                    for (int b2 = 0; b2 < 2; ++b2) {
                        const uint32_t send = (c & 1) ? xv[2 * b2] : xv[2 * b2 + 1];
                        const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1);
                        if (c & 1) xv[2 * b2] = recv; else xv[2 * b2 + 1] = recv;
                    }
                    const int r = 32 * q4 + 16 * hl + 8 * rb + (lane >> 2);
                    if (qt * kCT + r < a.L)
                        *reinterpret_cast<uint4 *>(ytile + (size_t)r * DP + 64 * half + 8 * (4 * bg + c)) =
                            make_uint4(xv[0], xv[1], xv[2], xv[3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, kFCols);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_gen_abort, 1);
}

unsigned lcm128(unsigned C)
{
    unsigned a = C, b = 128;
    while (b) {
        const unsigned r = a % b;
        a = b;
        b = r;
    }
    return C / a * 128;
}

}  // namespace

cudaError_t take_gen_abort(int *was_set)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_gen_abort, sizeof(int));
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        v = 0;
        e = cudaMemcpyToSymbol(g_gen_abort, &v, sizeof(int));
    }
    return e;
}

bool gen_supported(const Problem &p)
{
    const bool routed = mode_uses_u(p.mode);
    return p.bf16 && (p.d == 64 || p.d == 128) && p.C % 16 == 0 && (!routed || p.N <= kGMaxN) &&
           (p.mode != MC_SSC || (p.topk >= 0 && p.topk <= kTcMaxTopk));
}

namespace {
struct GenPlan {
    size_t kbar, ron, gates, total;
    int Lp, NB;
};
GenPlan gen_plan(const Problem &p)
{
    GenPlan g{};
    g.Lp = (p.L + kCT - 1) / kCT * kCT;
    g.NB = (p.N + 63) / 64;
    const bool routed = mode_uses_u(p.mode);
    g.kbar = routed ? pad256((size_t)p.BH * g.NB * kKbImg) : 0;
    g.ron = routed ? pad256(sizeof(float) * (size_t)p.BH * g.Lp) : 0;
    g.gates = routed ? pad256(sizeof(__nv_bfloat16) * (size_t)p.BH * p.N * g.Lp) : 0;
    g.total = g.kbar + g.ron + g.gates;
    return g;
}

// The state kernel and, for the routed aggregations, the gate kernel.
cudaError_t launch_gen_front(const Problem &p, const FwdArgs &fa, GenArgs &a, uint8_t *base, cudaStream_t s)
{
    if (!fa.k || !fa.v || (mode_uses_u(p.mode) && !fa.u)) return cudaErrorInvalidValue;
    const bool routed = mode_uses_u(p.mode);
    const GenPlan g = gen_plan(p);
    a.kbar_img = routed ? base : nullptr;
    a.r_on = routed ? reinterpret_cast<float *>(base + g.kbar) : nullptr;
    a.gates = routed ? reinterpret_cast<__nv_bfloat16 *>(base + g.kbar + g.ron) : nullptr;
    a.states = fa.states;
    a.BH = p.BH; a.L = p.L; a.Lp = g.Lp; a.d = p.d; a.C = p.C; a.N = p.N; a.NB = g.NB;
    a.topk = p.topk;
    a.UL = (int)lcm128((unsigned)p.C);
    a.units = (p.L + a.UL - 1) / a.UL;
    a.mean = p.mode == MC_MEAN;
    const int sms = sm_count();
    cudaError_t e;
    if (routed && (e = cudaMemsetAsync(a.kbar_img, 0, g.kbar, s)) != cudaSuccess) return e;
    if (routed || fa.states) {
        CUtensorMap mK, mV, mU;
        if (!make_tmap_bf16_3d_sw128(&mK, fa.k, p.BH, p.L, p.d, 128) ||
            !make_tmap_bf16_3d_sw128(&mV, fa.v, p.BH, p.L, p.d, 128))
            return cudaErrorInvalidValue;
        if (routed) {
            if (!make_tmap_bf16_3d_sw128(&mU, fa.u, p.BH, p.L, p.d, 128)) return cudaErrorInvalidValue;
        } else {
            mU = mK;
        }
        auto k1 = routed ? seg_piece_tc<true> : seg_piece_tc<false>;
        if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kPSmem)) != cudaSuccess)
            return e;
        const int units = p.BH * a.units;
        k1<<<units < sms ? units : sms, kPThreads, kPSmem, s>>>(mK, mV, mU, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "seg_piece_tc");
    }
    if (routed) {
        CUtensorMap mU;
        if (!make_tmap_bf16_3d_sw128(&mU, fa.u, p.BH, p.L, p.d, 128)) return cudaErrorInvalidValue;
        auto k2 = p.mode == MC_SSC ? gates_tc<true> : gates_tc<false>;
        if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem)) != cudaSuccess)
            return e;
        const int tiles = p.BH * (g.Lp / kCT);
        k2<<<tiles < sms ? tiles : sms, kGThreads, kGSmem, s>>>(mU, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "gates_tc");
    }
    return cudaSuccess;
}
}  // namespace

size_t gen_scratch_bytes(const Problem &p) { return gen_plan(p).total; }

// The gate kernel alone, on the state-form path's key-mean images ([BH][ceil(N/64)] blocks)
// and online scores ([BH][L], L a multiple of 128): gates [BH][N][L] bf16.
cudaError_t launch_gates_gen(const Problem &p, const void *u, uint8_t *kbar_img, float *r_on, __nv_bfloat16 *gates,
                             cudaStream_t s)
{
    if (p.L % kCT != 0 || p.N > kGMaxN) return cudaErrorInvalidValue;
    GenArgs a{};
    a.kbar_img = kbar_img;
    a.r_on = r_on;
    a.gates = gates;
    a.BH = p.BH; a.L = p.L; a.Lp = p.L; a.d = p.d; a.C = p.C; a.N = p.N; a.NB = (p.N + 63) / 64;
    a.topk = p.topk;
    CUtensorMap mU;
    if (!make_tmap_bf16_3d_sw128(&mU, u, p.BH, p.L, p.d, 128)) return cudaErrorInvalidValue;
    auto k2 = p.mode == MC_SSC ? gates_tc<true> : gates_tc<false>;
    cudaError_t e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kGSmem);
    if (e != cudaSuccess) return e;
    const int tiles = p.BH * (p.L / kCT), sms = sm_count();
    k2<<<tiles < sms ? tiles : sms, kGThreads, kGSmem, s>>>(mU, a);
    return cudaGetLastError();
}

cudaError_t launch_forward_gen(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    GenArgs a{};
    a.y = static_cast<__nv_bfloat16 *>(fa.y);
    profile_call_start(s);
    cudaError_t e = launch_gen_front(p, fa, a, static_cast<uint8_t *>(scratch), s);
    if (e != cudaSuccess) return e;
    CUtensorMap mQ, mK, mV;
    const unsigned vbox = p.d == 128 ? 64 : 128;  // d = 128: v in 64-key halves of both column panels
    if (!make_tmap_bf16_3d_sw128(&mQ, fa.q, p.BH, p.L, p.d, 128) || !make_tmap_bf16_3d_sw128(&mK, fa.k, p.BH, p.L, p.d, 128) ||
        !make_tmap_bf16_3d_sw128(&mV, fa.v, p.BH, p.L, p.d, vbox))
        return cudaErrorInvalidValue;
    const int w = mode_uses_u(p.mode) ? kWRouted : p.mode == MC_MEAN ? kWMean : kWOne;
    void (*k3)(const CUtensorMap, const CUtensorMap, const CUtensorMap, GenArgs);
    if (p.d == 128) k3 = w == kWRouted ? readout_fact_tc<128, kWRouted> : w == kWMean ? readout_fact_tc<128, kWMean> : readout_fact_tc<128, kWOne>;
    else k3 = w == kWRouted ? readout_fact_tc<64, kWRouted> : w == kWMean ? readout_fact_tc<64, kWMean> : readout_fact_tc<64, kWOne>;
    if ((e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kFSmem)) != cudaSuccess) return e;
    const int tiles = p.BH * ((p.L + kCT - 1) / kCT);
    const int slots = 2 * sm_count();
    k3<<<tiles < slots ? tiles : slots, kFThreads, kFSmem, s>>>(mQ, mK, mV, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_after_kernel(s, "readout_fact_tc");
    return cudaSuccess;
}

// The router alone on the general path: the state kernel (no states) and the SSC gate
// kernel, whose selections go to idx.
size_t gen_select_scratch_bytes(const Problem &p) { return gen_plan(p).total; }

cudaError_t launch_ssc_select_gen(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    GenArgs a{};
    a.sel_out = fa.sel_out;
    FwdArgs f = fa;
    f.states = nullptr;
    // The router reads no values (the caller passes none): the state kernel's value tiles,
    // whose products are discarded when no states are written, are read from k.
    f.v = fa.k;
    return launch_gen_front(p, f, a, static_cast<uint8_t *>(scratch), s);
}

}  // namespace mc
