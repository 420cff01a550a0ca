// tc_state_form.cuh -- the state-form kernels of the tensor-core forward (tcgen05 /
// TMEM / TMA), for bf16 inputs with seg_len a multiple of 128, templated on the head
// dimension D (64 or 128: every operand tile is D wide).  Included by the translation
// units that launch them (k_tc.cu for D = 128, k_tc64.cu for D = 64); each has its own
// copy of the kernels and of the abort flag.
//
// seg_state_tc -- persistent; each CTA walks its segments in chunks of 128 tokens
//   with the running state S = sum v_j k_j^T (fp32, one row per worker thread):
//     S += V_c^T K_c                        (update rule, [MC-ja §3 eq. 4b])
//   Before each chunk's update it writes S (the state before the chunk) as a bf16
//   operand image (the "prefix state" of the chunk); at the end S is the
//   segment's cached state M^(n) ([MC-ja §3, after eq. 4b]), written as fp32
//   (the states output) and as a bf16 image.  It also forms the key mean
//   kbar_n ([MC-ja §3.1 eq. 10], pooled keys) as hi + mid + lo bf16 rows of a
//   per-head operand image (the three terms sum to the fp32 mean exactly), and
//   the online gate score
//     r_on[t] = <u_t, sum_{j=t0..t} k_j> / (t - t0 + 1)
//   from R = U_c K_c^T (tensor core) masked to j <= t plus <u_t, keys before the chunk>.
//
// readout_tc -- persistent, two CTAs per SM; a tile is (bh, segment n, chunk c)
//   of 128 tokens, heaviest tiles first.  For the tile's tokens it computes
//     y_t = g_{t,n} [ S_pre(c) q_t + sum_{j in chunk, j<=t} v_j (k_j . q_t) ]
//         + sum_{i<n} g_{t,i} M^(i) q_t                      ([MC-ja §3.1 eq. 9])
//   (Residual: g = 1, [MC-ja §3.1 eq. 7], where the cached sum collapses to one
//   prefix state; Mean: the same with g = 1 / (n + 1)) as MMAs into one fp32 accumulator D per CTA:
//     G = Q K_c^T;  D = (g_n * mask(G)) V_c;  D += (g_i o Q) X_i^T
//   for X_i in {S_pre(c) (weight g_n), M^(0..n-1)}.  The gates come from the
//   scores <u_t, kbar_i> (three MMA sets per tile, kbar as hi, mid and lo rows:
//   every product is exact and only the fp32 accumulation rounds) and r_on[t]:
//   g = softmax over {scores_i}_{i<n} and r_on[t] (GRM; Soup is the same sum for
//   a linear memory, [MC-sum §3.3]); SSC keeps the topk largest cached scores
//   ([MC-sum §3.4]) and gives the others gate 0.  With more than 64 segments (GG) the
//   gates come from HBM instead, written by the general path's gate kernel.
//
// Over given segment boundaries (VAR) the state kernel's units are pieces of whole-chunk
// segments from a host table (a first launch in `totals` mode forms the pieces' own states,
// the second starts each piece from their sums) and the readout's tiles come from a
// (segment, chunk) table.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
#pragma once
#include <cstdint>

#include "mc_internal.cuh"
#include "sm100.cuh"
#include "tc_common.cuh"
#include "tensormap.cuh"

namespace mc {
namespace {

using namespace sm100;

// Set by any kernel of this translation unit that abandoned its work after a bounded
// wait ran out; read and cleared through the unit's take function (mc_check_device).
__device__ int g_tc_abort;

struct TcArgs {
    const __nv_bfloat16 *q, *u;
    __nv_bfloat16 *y;
    float *states;        // [BH][N][128][128] fp32 (output)
    uint8_t *states_img;  // [BH][N] x 32 KB  bf16 operand images of M^(n)
    uint8_t *spre_img;    // [BH][N][CPS] x 32 KB  prefix state before chunk c (c >= 1)
    uint8_t *kbar_img;    // [BH][NB] x 48 KB: hi, mid, lo rows (16 KB each), row = segment % 64
    uint8_t *prefix_img;  // [BH][N] x 32 KB  sum_{i<n} M^(i) (Residual)
    float *r_on;          // [BH][L]
    float *gam_out;       // backward gates: [BH][N][L] g_{t,i}, or null
    float *tok_out;       // backward gates: [BH][L][kBwdTokWords], word 2 = the online gate
    float *kbar_out;      // backward: fp32 key means [BH][N][d], or null
    float *kpre_out;      // backward: keys of the segment before each 64-token tile [BH][N][2 CPS][d], or null
    int32_t *sel_out;     // SSC: optional [BH][L][topk] router output (rank order, -1 padded)
    const __nv_bfloat16 *gates;  // gates from HBM (more than 64 segments): [BH][N][L] bf16, or null
    int topk;             // SSC: cached segments selected per token
    int mean;             // Mean aggregation: the Residual path with every weight 1 / (n + 1)
    const float *alpha, *beta, *lam;  // SWLA per-token scalars [BH][L] (SWLA kernels only)
    int BH, L, C, N, CPS;
    int d;                // head dimension of q, k, v, u, y and the states (64 or 128: the tiles' width D)
    int NB;               // blocks of 64 segments in a head's key-mean image (1 when N <= 64)
    int num_tiles;
    int hg;               // readout: heads per group (tiles go group by group, the heaviest first within one)
    // Given segment boundaries (the VAR kernels): segments 0 .. Nseg-1 of every head start at
    // sg_off[n] (a multiple of 128) and are whole 128-token chunks; sg_cbase[n] is the segment's
    // first chunk among the head's NC chunks (prefix-state images [BH][NC]); the readout's tiles
    // are vtiles[id / BH] = (segment, chunk), heaviest first.
    const int32_t *sg_off, *sg_cbase;
    const int2 *vtiles;
    int Nseg, NC;
    // The state kernel's units over given boundaries: pieces (segment, first chunk within it, chunks,
    // aux) of the whole-chunk segments, the longest first.  With `totals` set the kernel only forms
    // each unit's own state and key sum (aux = its slot in ptot / pks); otherwise a unit starts
    // from the sum of the totals of the pieces before it (aux = first slot << 8 | their count).
    const int4 *units;
    int NU, totals, nslots;
    float *ptot;  // [BH][nslots][d][d] fp32
    float *pks;   // [BH][nslots][d] fp32
};

// A head's segment as the kernels see it: constant length C, or from the tables.
struct SegInfo {
    int bh, seg, nch, off, len, cbase;
    int pc0, aux;  // VAR: the unit's first chunk within its segment, and its table word
    bool last;     // the unit ends its segment
};

template <bool VAR>
__device__ __forceinline__ SegInfo seg_info(const TcArgs &a, int uid)
{
    SegInfo u;
    if (!VAR) {  // units head by head
        u.bh = uid / a.N;
        u.seg = uid % a.N;
        u.nch = a.CPS;
        u.off = u.seg * a.C;
        u.len = a.C;
        u.cbase = u.seg * a.CPS;
        u.pc0 = 0;
        u.aux = 0;
        u.last = true;
    } else {  // units from the table (the longest first), every head of a unit together
        const int4 t = a.units[uid / a.BH];
        u.seg = t.x;
        u.bh = uid % a.BH;
        u.pc0 = t.y;
        u.nch = t.z;
        u.aux = t.w;
        u.len = a.sg_off[u.seg + 1] - a.sg_off[u.seg];
        u.off = a.sg_off[u.seg] + t.y * kCT;
        u.cbase = a.sg_cbase[u.seg] + t.y;
        u.last = t.y + t.z == u.len / kCT;
    }
    return u;
}

// SWLA (sliding-window linear attention, c = 2, [MC-ja §3.1 eq. 28]) within one
// 128-token chunk whose first token is t_c:
//   M_t = A(t_c, t) S^_c + sum_{j = t_c..t} c_{t,j} v_j k_j^T,
//   c_{t,j} = lambda_j A(j, t) + [j < t] beta_{j+1} A(j+1, t),  A(a, t) = prod_{i=a+1..t} alpha_i,
//   S^_c = alpha_{t_c} M_{t_c - 1} + beta_{t_c} v_{t_c - 1} k_{t_c - 1}^T   (0 at a segment's start).
// A(a, t) = exp(ell_t - ell_a) with ell the running sum of log alpha over the chunk
// (ell = 0 at t_c).  Every warp holds the whole chunk, lane l tokens 4l .. 4l + 3.
struct ChunkDecay {
    float ell[4], lam[4], bet[4];
};

__device__ __forceinline__ ChunkDecay load_chunk_decay(const float *alpha, const float *beta, const float *lam,
                                                        size_t tok0, int lane)
{
    ChunkDecay cd;
    const float4 al = *reinterpret_cast<const float4 *>(alpha + tok0 + 4 * lane);
    const float4 be = *reinterpret_cast<const float4 *>(beta + tok0 + 4 * lane);
    const float4 la = *reinterpret_cast<const float4 *>(lam + tok0 + 4 * lane);
    float x0 = lane == 0 ? 0.f : logf(fmaxf(al.x, 1e-30f));  // the chunk's first token carries no decay
    float x1 = logf(fmaxf(al.y, 1e-30f)), x2 = logf(fmaxf(al.z, 1e-30f)), x3 = logf(fmaxf(al.w, 1e-30f));
    x1 += x0;
    x2 += x1;
    x3 += x2;
    float tot = x3;  // inclusive scan of the lanes' sums
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, tot, o);
        if (lane >= o) tot += y;
    }
    const float ex = tot - x3;
    cd.ell[0] = x0 + ex;
    cd.ell[1] = x1 + ex;
    cd.ell[2] = x2 + ex;
    cd.ell[3] = x3 + ex;
    cd.lam[0] = la.x; cd.lam[1] = la.y; cd.lam[2] = la.z; cd.lam[3] = la.w;
    cd.bet[0] = be.x; cd.bet[1] = be.y; cd.bet[2] = be.z; cd.bet[3] = be.w;
    return cd;
}

// Value of chunk token j (0..127) from the lane that holds it; every lane of the warp calls it.
__device__ __forceinline__ float chunk_pick(const float (&v)[4], int j)
{
    const int src = j >> 2, e = j & 3;
    const float v0 = __shfl_sync(0xffffffffu, v[0], src), v1 = __shfl_sync(0xffffffffu, v[1], src);
    const float v2 = __shfl_sync(0xffffffffu, v[2], src), v3 = __shfl_sync(0xffffffffu, v[3], src);
    return e == 0 ? v0 : e == 1 ? v1 : e == 2 ? v2 : v3;
}


// ============================================================================
// seg_state_tc
// ============================================================================
constexpr int kT1Threads = 192;               // warp 0 TMA, warp 1 MMA, warps 2-5 workers
constexpr uint32_t kT1Stage2 = 4096;           // per worker warp: 32 rows x 128 bytes of a store in flight
// A stage holds the K, V, U tiles of one chunk; with the SWLA update also alpha and
// beta of the chunk's tokens plus the next one (132 floats each) and lambda (128).
// K, V and U of a chunk are D / 64 panels each (128 tokens x 64 columns, 16 KB).
template <int D>
__host__ __device__ constexpr uint32_t t1_dec_off() { return 3u * (D / 64) * kPanel; }
constexpr uint32_t kT1DecBytes = 2 * 132 * 4 + 128 * 4;
template <bool DECAY, int D = 128>
__host__ __device__ constexpr uint32_t t1_stage_bytes() { return t1_dec_off<D>() + (DECAY ? 2048u : 0u); }  // tiles stay 1024-aligned
static_assert(kT1DecBytes <= 2048, "the SWLA scalars fit the stage's tail");
// D = 128: two stages, one CTA per SM.  D = 64: one stage and a 16 KB zero panel (the upper 64 rows of
// the M = 128 operand V^T), two CTAs per SM.
template <int D>
__host__ __device__ constexpr int t1_stages() { return D == 64 ? 1 : 2; }
template <bool DECAY, int D = 128>
__host__ __device__ constexpr size_t t1_smem_bytes()
{
    return t1_stages<D>() * t1_stage_bytes<DECAY, D>() + 4 * kT1Stage2 + (D == 64 ? kPanel : 0) + 1024;
}

template <bool GATED, bool DECAY, bool VAR = false, int D = 128>
__global__ void __launch_bounds__(kT1Threads, D == 64 ? 2 : 1)
    seg_state_tc(const __grid_constant__ CUtensorMap mK, const __grid_constant__ CUtensorMap mV,
                 const __grid_constant__ CUtensorMap mU, TcArgs a)
{
    static_assert(D == 64 || D == 128, "head dimension");
    constexpr int NP = D / 64;              // 64-column panels of an operand tile
    constexpr uint32_t kOp = NP * kPanel;   // one chunk's K, V or U tile
    constexpr uint32_t kImg = D * D * 2;    // a D x D bf16 operand image
    constexpr uint32_t kStage = t1_stage_bytes<DECAY, D>();
    constexpr int NS = t1_stages<D>();       // operand stages
    constexpr int NR = D == 64 ? 1 : 2;      // U K^T buffers in tensor memory
    constexpr uint32_t kCols = D == 64 ? 256 : 512;  // R x NR | Z x 2 (D columns each, 128 apart at D = 128)
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t full[2], empty[2], r_full[2], r_empty[2], z_full[2], z_empty[2];
    __shared__ uint64_t v_scaled;  // SWLA: the workers have weighted the chunk's value rows
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;
    __shared__ __align__(16) float ksum_s[kD];
    __shared__ __align__(16) float red_s[8][kD];  // column-sum partials of 16-row groups

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // Persistent: this CTA walks segments (units) blockIdx.x, blockIdx.x + gridDim.x, ...;
    // its chunks form one stream (global chunk counter g) so loads run ahead
    // across segment boundaries.
    const int nseg_total = a.BH * (VAR ? a.NU : a.N);
    const bool totals = VAR && a.totals;  // units form their own state only (no images, no scores)
    const int my_segs = (int)blockIdx.x < nseg_total ? (nseg_total - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    int my_chunks = 0;
    for (int k = 0; k < my_segs; ++k) my_chunks += seg_info<VAR>(a, (int)blockIdx.x + k * (int)gridDim.x).nch;
    const int NCH = VAR ? a.NC : a.N * a.CPS;  // prefix-state images per head
    if (GATED && !totals) {
        // The key-mean image's rows past the last segment (segments N .. 64 NB - 1, which no unit writes)
        // are zero when the readout's score MMAs read them: every thread clears a strided share of them.
        const int nrow = VAR ? a.Nseg : a.N;
        const int tail = a.NB * 64 - nrow;
        if (tail > 0) {
            const long long per_head = 3LL * NP * tail * 8;  // terms x panels x rows x 16-byte chunks
            const long long total = per_head * a.BH;
            for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
                 i += (long long)gridDim.x * blockDim.x) {
                const int bh = (int)(i / per_head);
                long long r = i % per_head;
                const int ch = (int)(r & 7);
                r >>= 3;
                const int row = nrow + (int)(r % tail);
                r /= tail;
                const int panel = (int)(r % NP), term = (int)(r / NP);
                uint8_t *p = a.kbar_img + ((size_t)bh * a.NB + (row >> 6)) * kKbImg + (size_t)term * kKbPanel +
                             panel * (64 * 128) + (row & 63) * 128 + ch * 16;
                *reinterpret_cast<uint4 *>(p) = make_uint4(0u, 0u, 0u, 0u);
            }
        }
    }
    // each role walks the chunk stream with a cursor: the unit, and the chunk within it
    struct Cursor {
        int k, c;
        SegInfo u;
    };
    auto start = [&]() {
        Cursor q;
        q.k = 0;
        q.c = 0;
        q.u = seg_info<VAR>(a, (int)blockIdx.x);
        return q;
    };
    auto advance = [&](Cursor &q) {
        if (++q.c == q.u.nch) {
            q.c = 0;
            ++q.k;
            if (q.k < my_segs) q.u = seg_info<VAR>(a, (int)blockIdx.x + q.k * (int)gridDim.x);
        }
    };

    if (warp == 0) {
        tmem_alloc(&tmem_base, kCols);
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
        mbar_init(&v_scaled, 128);
        fence_mbar_init();
    }
    uint8_t *const zero_panel = sm + NS * kStage + 4 * kT1Stage2;  // D = 64 only
    if (D == 64) {
        for (int i = threadIdx.x; i < (int)(kPanel / 16); i += kT1Threads)
            reinterpret_cast<uint4 *>(zero_panel)[i] = make_uint4(0u, 0u, 0u, 0u);
        fence_async_smem();  // visible to the tensor cores
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    // tensor memory: R (U K^T) x NR, 128 columns each | Z (chunk state V^T K) x 2
    const uint32_t tR0 = tb, tZ0 = tb + 128 * NR;
    constexpr uint32_t kZStride = D == 64 ? 64 : 128;

    if (warp == 0) {
        if (lane == 0) {
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            if (GATED) prefetch_tensormap(&mU);
            Cursor cu = start();
            for (int gch = 0; gch < my_chunks; ++gch, advance(cu)) {
                const int c = cu.c, nch = cu.u.nch;
                const int rr = cu.u.bh * a.L + cu.u.off + c * kCT;
                const int s = gch % NS;
                const uint32_t r = gch / NS;
                if (!mbar_wait(&empty[s], (r & 1) ^ 1, &abort_flag)) break;
                uint8_t *st = sm + s * kStage;
                // SWLA: alpha and beta reach one token into the next chunk when it is in the same segment
                const uint32_t dec_ab = (c + 1 < nch ? 132u : 128u) * 4u;
                // the first segment's tokens have no cached memory: their single gate is 1 and
                // their online score is not needed, so u is not read there
                const bool scored = GATED && cu.u.seg != 0 && !totals;
                mbar_arrive_expect_tx(&full[s], (scored ? 3 * kOp : 2 * kOp) + (DECAY ? 2 * dec_ab + 512u : 0u));
                if (DECAY) {
                    float *dec = reinterpret_cast<float *>(st + t1_dec_off<D>());
                    bulk_load(dec, a.alpha + rr, dec_ab, &full[s]);
                    bulk_load(dec + 132, a.beta + rr, dec_ab, &full[s]);
                    bulk_load(dec + 264, a.lam + rr, 512u, &full[s]);
                }
#pragma unroll
                for (int h = 0; h < NP; ++h) {
                    tma_load_2d(st + h * kPanel, &mK, 64 * h, rr, &full[s]);
                    tma_load_2d(st + kOp + h * kPanel, &mV, 64 * h, rr, &full[s]);
                    if (scored) tma_load_2d(st + 2 * kOp + h * kPanel, &mU, 64 * h, rr, &full[s]);
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idR = idesc_bf16(128, 128, false, false);
            constexpr uint32_t idS = idesc_bf16(128, D, true, true);
            uint32_t rc = 0;  // chunks with online scores (not in a head's first segment)
            Cursor cu = start();
            for (int gch = 0; gch < my_chunks; ++gch, advance(cu)) {
                const int s = gch % NS, b = gch & 1;
                const uint32_t r = gch / NS, rz = gch >> 1;
                if (!mbar_wait(&full[s], r & 1, &abort_flag)) break;
                tc_fence_after();
                const uint32_t kb = smem_u32(sm + s * kStage), vb = kb + kOp, ub = kb + 2 * kOp;
                // V^T is M = 128 rows: the two 64-row halves of V (D = 128), or V and the zero panel
                const uint32_t v_lbo = D == 128 ? kPanel : smem_u32(zero_panel) - vb;
                if (GATED && cu.u.seg != 0 && !totals) {  // R = U K^T (online gate score of the chunk's tokens)
                    const int rb = rc % NR;
                    if (!mbar_wait(&r_empty[rb], ((rc / NR) & 1) ^ 1, &abort_flag)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 4 * NP; ++kk)
                        mma_ss(tR0 + rb * 128, make_desc_sw128(ub + kmaj_off(kk, 128), 0, 1024),
                               make_desc_sw128(kb + kmaj_off(kk, 128), 0, 1024), idR, kk > 0);
                    mma_commit(&r_full[rb]);
                    ++rc;
                }
                // Z = V^T K, the chunk's own state (fresh accumulator); SWLA: V^T diag(w) K
                if (!mbar_wait(&z_empty[b], (rz & 1) ^ 1, &abort_flag)) break;
                if (DECAY && !mbar_wait(&v_scaled, gch & 1, &abort_flag)) break;
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < 8; ++kk)
                    mma_ss(tZ0 + b * kZStride, make_desc_sw128(vb + kk * 2048u, v_lbo, 1024),
                           make_desc_sw128(kb + kk * 2048u, 16384, 1024), idS, kk > 0);
                mma_commit(&z_full[b]);
                mma_commit(&empty[s]);
            }
        }
    } else {
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;  // TMEM lane = token row (R) = value row (Z, S) = key column (sums)
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        float S[D];  // running state row: S[row][k] = sum_{j before the chunk} v_j[row] k_j[k]
        uint8_t *wst = sm + NS * kStage + q4 * kT1Stage2;  // this warp's staging area for global stores
        float ks = 0.f;  // running sum of key column `row` over the segment, in token order
        // A worker that gives up (bounded wait ran out) keeps walking the loop
        // without work so that every warp reaches the same named barriers.
        bool ok = true;
        uint32_t rc = 0;  // chunks with online scores, in step with the MMA issuer
        Cursor cu = start();
        for (int gch = 0; gch < my_chunks; ++gch, advance(cu)) {
            const int c = cu.c, nch = cu.u.nch;
            const int bh = cu.u.bh, seg = cu.u.seg;
            const int row0 = bh * a.L + cu.u.off;
            const int s = gch % NS, b = gch & 1;
            const uint32_t r = gch / NS, rz = gch >> 1;
            if (c == 0) {  // a new unit: memory restarts at zero, or at the sum of the earlier pieces' totals
#pragma unroll
                for (int k = 0; k < D; ++k) S[k] = 0.f;
                ks = 0.f;
                if (VAR && !totals && (int)row < D) {
                    const int slot0 = cu.u.aux >> 8, npre = cu.u.aux & 255;
                    for (int pp = 0; pp < npre; ++pp) {
                        const size_t sl = (size_t)bh * a.nslots + slot0 + pp;
                        const float4 *tp = reinterpret_cast<const float4 *>(a.ptot + (sl * D + row) * D);
#pragma unroll
                        for (int k4 = 0; k4 < D / 4; ++k4) {
                            const float4 x = tp[k4];
                            S[4 * k4] += x.x; S[4 * k4 + 1] += x.y; S[4 * k4 + 2] += x.z; S[4 * k4 + 3] += x.w;
                        }
                        ks += a.pks[sl * D + row];
                    }
                }
                ksum_s[row] = ks;
                named_bar_sync(1, 128);
            }
            if (ok) ok = mbar_wait(&full[s], r & 1, &abort_flag);
            const uint8_t *st = sm + s * kStage;
            // SWLA: the chunk's state is S_{c+1} = zdecay * S^_c + V^T diag(w) K, where w_j is
            // token j's weight at the chunk's end, carried one step on (alpha', beta' of the
            // next token) when that token is in the same segment -- so S is S^_{c+1}.
            float zdecay = 1.f;
            if (DECAY) {
                const float *dec = reinterpret_cast<const float *>(st + t1_dec_off<D>());  // alpha | beta | lambda
                const ChunkDecay cd = load_chunk_decay(dec, dec + 132, dec + 264, 0, lane);
                const int jt = (int)row, jn = jt < kCT - 1 ? jt + 1 : jt;
                const float ell_end = __shfl_sync(0xffffffffu, cd.ell[3], 31);
                const float ell_j = chunk_pick(cd.ell, jt), lam_j = chunk_pick(cd.lam, jt);
                const float ell_n = chunk_pick(cd.ell, jn), bet_n = chunk_pick(cd.bet, jn);
                float a_next = 1.f, b_next = 0.f;
                if (c + 1 < nch) {
                    a_next = dec[kCT];
                    b_next = dec[132 + kCT];
                }
                float w = lam_j * __expf(ell_end - ell_j);
                if (jt < kCT - 1) w += bet_n * __expf(ell_end - ell_n);
                w = a_next * w + (jt == kCT - 1 ? b_next : 0.f);
                zdecay = a_next * __expf(ell_end);
                if (ok) {  // value row of token jt, in place (the tile is MN-major, 128-byte swizzled)
                    uint8_t *vt = const_cast<uint8_t *>(st) + kOp;
#pragma unroll
                    for (int cc = 0; cc < D / 8; ++cc) {
                        uint4 *pv = reinterpret_cast<uint4 *>(vt + sw128_offset(jt, 8 * cc, 128));
                        uint4 x = *pv;
                        uint32_t *xw = reinterpret_cast<uint32_t *>(&x);
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&xw[e]));
                            xw[e] = pack_bf16x2(w * f.x, w * f.y);
                        }
                        *pv = x;
                    }
                    fence_async_smem();
                }
                mbar_arrive(&v_scaled);
            }
            if (GATED && seg == 0 && ok && !totals) a.r_on[(size_t)row0 + c * kCT + row] = 0.f;  // single gate: the score is unused
            if (GATED && seg != 0 && ok && !totals) {
                const int rb = rc % NR;
                float d4[4] = {0.f, 0.f, 0.f, 0.f};  // <u_t, keys of the segment before this chunk>
#pragma unroll
                for (int cc = 0; cc < D / 8; ++cc) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(st + 2 * kOp + sw128_offset(row, 8 * cc, 128));
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
                const float dot = (d4[0] + d4[1]) + (d4[2] + d4[3]);
                ok = mbar_wait(&r_full[rb], (rc / NR) & 1, &abort_flag);
                if (ok) {
                    tc_fence_after();
                    float w4[4] = {0.f, 0.f, 0.f, 0.f};  // sum_{j <= t} <u_t, k_j> within the chunk
#pragma unroll
                    for (int j16 = 0; j16 < 8; ++j16) {
                        if (16 * j16 > 32 * q4 + 31) break;  // columns past the warp's last row are masked
                        uint32_t v[16];
                        tmem_ld16(tR0 + rb * 128 + lane_base + 16 * j16, v);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            if ((uint32_t)(16 * j16 + i) <= row) w4[i & 3] += __uint_as_float(v[i]);
                    }
                    const float w = (w4[0] + w4[1]) + (w4[2] + w4[3]);
                    tc_fence_before();
                    mbar_arrive(&r_empty[rb]);
                    const int t_in_seg = (cu.u.pc0 + c) * kCT + (int)row;
                    a.r_on[(size_t)row0 + c * kCT + row] = (dot + w) / (float)(t_in_seg + 1);
                }
            }
            if (GATED && seg != 0 && !totals) ++rc;
            // Key column sums of the chunk, in a fixed order: thread (rg, cc) sums
            // columns 8cc..8cc+7 over rows 16rg..16rg+15 in row order; then column
            // `row` adds the eight group sums in rg order to the running sum.
            if (ok) {
                const int cc = row & 15, rg = row >> 4;
                float p8[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // columns past D stay 0
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    if (8 * cc >= D) break;
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
            named_bar_sync(1, 128);  // every worker has read ksum_s and written its partials
            if (ok) {
                float cs = 0.f, ch = 0.f;
#pragma unroll
                for (int g8 = 0; g8 < 8; ++g8) {
                    cs += red_s[g8][row];
                    if (g8 == 3) ch = cs;  // the chunk's first 64 rows
                }
                if (!VAR && GATED && a.kpre_out && (int)row < a.d) {  // keys before the chunk's two 64-token halves
                    float *kp = a.kpre_out + (((size_t)bh * a.N + seg) * (2 * nch) + 2 * c) * a.d + row;
                    kp[0] = ks;
                    kp[a.d] = ks + ch;
                }
                ks += cs;
                ksum_s[row] = ks;
            }
            named_bar_sync(1, 128);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
            // S += Z_c; then S is the prefix state of chunk c + 1
            if (ok) ok = mbar_wait(&z_full[b], rz & 1, &abort_flag);
            if (ok) {
                tc_fence_after();
#pragma unroll
                for (int j16 = 0; j16 < D / 16; ++j16) {
                    uint32_t v[16];
                    tmem_ld16(tZ0 + b * kZStride + lane_base + 16 * j16, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) S[16 * j16 + i] = fmaf(zdecay, S[16 * j16 + i], __uint_as_float(v[i]));
                }
                tc_fence_before();
                mbar_arrive(&z_empty[b]);
                const size_t sidx = (size_t)bh * a.N + seg;
                const bool seg_end = c + 1 == nch && cu.u.last;
                if (totals && c + 1 == nch && (int)row < D) {  // the piece's own state and key sums
                    const size_t sl = (size_t)bh * a.nslots + cu.u.aux;
                    float4 *tp = reinterpret_cast<float4 *>(a.ptot + (sl * D + row) * D);
#pragma unroll
                    for (int k4 = 0; k4 < D / 4; ++k4) tp[k4] = make_float4(S[4 * k4], S[4 * k4 + 1], S[4 * k4 + 2], S[4 * k4 + 3]);
                    a.pks[sl * D + row] = ks;
                }
                uint8_t *img = !seg_end ? a.spre_img + ((size_t)bh * NCH + cu.u.cbase + c + 1) * kImg
                                        : a.states_img + sidx * kImg;
                // Through the warp's 4 KB staging area, one 64-column panel at a time: the
                // warp's 32 rows of a panel are 4 KB contiguous in the image, stored 512
                // contiguous bytes per instruction.  (D = 64: rows 64.. are zero and not stored.)
#pragma unroll
                for (int p = 0; p < NP; ++p) {
                    if (32 * q4 >= D || totals) break;  // warp-uniform
#pragma unroll
                    for (int c8 = 0; c8 < 8; ++c8) {  // 16-byte chunk c8 of the row's panel p
                        const int cc = 8 * p + c8;
                        const uint4 v = make_uint4(pack_bf16x2(S[8 * cc], S[8 * cc + 1]), pack_bf16x2(S[8 * cc + 2], S[8 * cc + 3]),
                                                   pack_bf16x2(S[8 * cc + 4], S[8 * cc + 5]), pack_bf16x2(S[8 * cc + 6], S[8 * cc + 7]));
                        *reinterpret_cast<uint4 *>(wst + sw128_offset(lane, 8 * c8, 32)) = v;
                    }
                    __syncwarp();
                    uint4 *dst = reinterpret_cast<uint4 *>(img + p * (D * 128) + (32 * q4) * 128);
#pragma unroll
                    for (int i = 0; i < 8; ++i) dst[32 * i + lane] = reinterpret_cast<const uint4 *>(wst)[32 * i + lane];
                    __syncwarp();
                }
                if (seg_end && !totals) {  // the segment's cached state (fp32) and key mean
                    // fp32 rows (d values), 32 columns (128 bytes) at a time through the staging
                    // area (16-byte chunk c of row r at chunk c ^ (r % 8)), 4 rows per instruction;
                    // with d < 128 the padded rows and columns are not stored
                    const int d = a.d;
                    float *o = a.states + sidx * d * d + (size_t)(32 * q4) * d;
#pragma unroll
                    for (int blk = 0; blk < D / 32; ++blk) {
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
                            const int r = 4 * i + (lane >> 3), c8 = lane & 7;
                            const float4 v = *reinterpret_cast<const float4 *>(wst + r * 128 + ((c8 ^ (r & 7)) << 4));
                            *reinterpret_cast<float4 *>(o + (size_t)r * d + 32 * blk + 4 * c8) = v;
                        }
                        __syncwarp();
                    }
                    if (GATED) {
                        const float kbv = ks / (float)cu.u.len;
                        if (a.kbar_out && (int)row < a.d) a.kbar_out[sidx * a.d + row] = kbv;
                        store_kbar_terms(a.kbar_img + (size_t)bh * a.NB * kKbImg, seg, row, kbv);
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, kCols);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_tc_abort, 1);
}

// Residual: prefix sums of the cached states, P_n = sum_{i<n} M^(i) (fp32
// accumulate), written as bf16 D x D operand images (P_0 is never read).
template <int D>
__global__ void __launch_bounds__(256) prefix_images(TcArgs a)
{
    const int bh = blockIdx.y;
    const int e = blockIdx.x * blockDim.x + threadIdx.x;  // element of the D x D image
    if (e >= D * D) return;
    const int v = e / D, k = e % D, d = a.d;
    const bool inside = v < d && k < d;  // padding (d < D) stays zero
    const float *st = a.states + (size_t)bh * a.N * d * d + (inside ? v * d + k : 0);
    float acc = 0.f;
    for (int n = 1; n < a.N; ++n) {
        if (inside) acc += st[(size_t)(n - 1) * d * d];
        *reinterpret_cast<__nv_bfloat16 *>(a.prefix_img + ((size_t)bh * a.N + n) * (D * D * 2) + sw128_offset(v, k, D)) =
            __float2bfloat16_rn(acc);
    }
}

// The gates of one token ([MC-ja §3.1 eq. 10], normalised by a softmax) from its
// scores sc[0..n) against the cached segments and its online score ron.  GRM / Soup:
// every cached segment takes part; SSC ([MC-sum §3.4]): the topk largest scores,
// equal scores to the lower segment index (their indices, in rank order and -1
// padded, go to so when given).  On return sc[i] (i < 63) holds the unnormalised
// weight of segment i (0 when not taken or i >= n), sc[63] the online one; the
// result is 1 / Z.  n is the same for every thread of a warp, so the loops skip
// whole groups of 8 segments uniformly.
template <bool SSC>
__device__ __forceinline__ float token_gates(float (&sc)[64], int n, float ron, int topk, int32_t *so)
{
    uint64_t take = n >= 64 ? ~0ull : ((1ull << n) - 1);
    if (SSC) {
        const int cnt = min(topk, n);
        uint64_t chosen = 0;
        for (int r = 0; r < cnt; ++r) {
            float best = 0.f;
            int bi = -1;
#pragma unroll
            for (int g8 = 0; g8 < 8; ++g8) {
                if (8 * g8 >= n) break;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const int k = 8 * g8 + kk;
                    if (k < 63 && k < n && !((chosen >> k) & 1ull) && (bi < 0 || sc[k] > best)) {
                        best = sc[k];
                        bi = k;
                    }
                }
            }
            chosen |= 1ull << bi;
            if (so) so[r] = bi;
        }
        if (so)
            for (int r = cnt; r < topk; ++r) so[r] = -1;
        take = chosen;
    }
    float mx4[4] = {ron, ron, ron, ron};  // partial maxima / sums: shorter dependency chains
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) {
        if (8 * g8 >= n) break;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int k = 8 * g8 + kk;
            if (k < 63 && ((take >> k) & 1ull)) mx4[kk & 3] = fmaxf(mx4[kk & 3], sc[k]);
        }
    }
    const float mx = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3]));
    float z4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int g8 = 0; g8 < 8; ++g8) {
        if (8 * g8 >= n) break;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            const int k = 8 * g8 + kk;
            if (k < 63) {
                sc[k] = ((take >> k) & 1ull) ? __expf(sc[k] - mx) : 0.f;
                z4[kk & 3] += sc[k];
            }
        }
    }
    sc[63] = __expf(ron - mx);
    return 1.f / (sc[63] + (z4[0] + z4[1]) + (z4[2] + z4[3]));
}

// ============================================================================
// readout_tc
// ============================================================================
constexpr int kT2Threads = 192;    // warp 0 TMA, warp 1 MMA issuer, warps 2-5 token-row workers
constexpr int kT2CtasPerSm = 2;    // two CTAs share each SM's tensor pipe
constexpr int kRing = 6;           // operand panels in flight per CTA
constexpr uint32_t kT2Cols = 256;  // tensor memory per CTA: D (128 columns) | A slot 0 | A slot 1 (64 each)
constexpr uint32_t kT2Decay = 4 * 5 * kCT * 4;   // SWLA: per worker warp, ell | lambda | beta_next | E | F of a chunk
constexpr size_t kT2Smem = kRing * kPanel + kT2Decay + 1024;  // two CTAs fit in an SM's 228 KB

struct TileInfo {
    int n, c, bh;
    int off;    // the segment's first token within the head
    int cbase;  // the segment's first chunk among the head's chunks
};

template <bool VAR>
__device__ __forceinline__ TileInfo decode_tile(const TcArgs &a, int id)
{
    TileInfo t;
    if (!VAR) {
        // groups of hg heads (the last one smaller), so that the cached images the tiles in flight
        // read stay within the L2; inside a group the segments with the most cached states first
        const int per_group = a.hg * a.N * a.CPS;
        const int grp = id / per_group;
        const int first = grp * a.hg;
        const int heads = min(a.hg, a.BH - first);
        const int rem0 = id - grp * per_group;
        const int per_seg = heads * a.CPS;
        t.n = a.N - 1 - rem0 / per_seg;
        const int rem = rem0 % per_seg;
        t.c = rem / heads;
        t.bh = first + rem % heads;
        t.off = t.n * a.C;
        t.cbase = t.n * a.CPS;
    } else {
        const int2 nc = a.vtiles[id / a.BH];
        t.n = nc.x;
        t.c = nc.y;
        t.bh = id % a.BH;
        t.off = a.sg_off[t.n];
        t.cbase = a.sg_cbase[t.n];
    }
    return t;
}

// Cached operands a tile reads, in order: the chunk's prefix state (c > 0), then
// the cached states M^(0..n-1) (GRM) or their prefix sum P_n (Residual, n > 0).
template <bool GATED>
__device__ __forceinline__ int tile_items(const TileInfo &t)
{
    return GATED ? t.n + (t.c > 0 ? 1 : 0) : (t.n > 0 ? 1 : 0) + (t.c > 0 ? 1 : 0);
}

template <bool GATED, bool VAR, int D>
__device__ __forceinline__ const uint8_t *item_image(const TcArgs &a, const TileInfo &t, int k)
{
    constexpr size_t kImg = D * D * 2;
    const size_t sb = (size_t)t.bh * a.N;
    if (t.c > 0) {
        const size_t nch_head = VAR ? (size_t)a.NC : (size_t)a.N * a.CPS;
        if (k == 0) return a.spre_img + ((size_t)t.bh * nch_head + t.cbase + t.c) * kImg;
        --k;
    }
    return GATED ? a.states_img + (sb + k) * kImg : a.prefix_img + (sb + t.n) * kImg;
}


// One tile = 128 tokens (bh, segment n, chunk c).  Per tile, in this order, into
// one fp32 accumulator D[t][v]:
//   G   = Q K_c^T                      (both operands in shared memory)
//   D   = P V_c,  P = g_n * mask(G)    (P written into tensor memory by the workers)
//   D  += (g_i o Q) X_i^T              for X_i in {S_pre(c), M^(0..n-1)} (GRM / Soup)
//                                      or {S_pre(c), sum_{i<n} M^(i)} (Residual, g = 1)
// Operands stream through a ring of 16 KB panels (a K-half of a 128 x 128 tile;
// V in key halves).  The workers take their query rows from the Q panels (and
// release those panels once G is done), read the gate rows in the tile-transposed
// layout (coalesced), and write y from a quad-transposed register layout.  Two CTAs run on each SM, so while one waits on its G -> P step or its
// drain the other keeps the tensor pipe busy.
// GG: the gates come from HBM (gates[bh][i][t], the online gate at i = n), written by
// the gate kernel, instead of being formed here from scores in tensor memory; the tile then
// reads no U or key-mean panels, and any number of cached segments works.
template <bool GATED, bool DECAY, bool SSC, bool GG = false, bool VAR = false, int D = 128>
__global__ void __launch_bounds__(kT2Threads, kT2CtasPerSm)
    readout_tc(const __grid_constant__ CUtensorMap mQ, const __grid_constant__ CUtensorMap mK,
               const __grid_constant__ CUtensorMap mV, const __grid_constant__ CUtensorMap mU, TcArgs a)
{
    static_assert(D == 64 || D == 128, "head dimension");
    constexpr int NP = D / 64;  // 64-column panels of a Q, K, U tile or of an image
    constexpr uint32_t kImg = D * D * 2;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *sm = align1024(smem_raw);
    __shared__ uint64_t ring_full[kRing], ring_empty[kRing];
    __shared__ uint64_t a_full[2], a_empty[2];
    __shared__ uint64_t g_full, y_full, y_empty, fin, q_read, s_full;
    __shared__ uint32_t tmem_base;
    __shared__ int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntiles = a.num_tiles;
    const int my_tiles =
        blockIdx.x < (unsigned)ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    auto tile_id = [&](int j) { return (int)blockIdx.x + j * (int)gridDim.x; };  // heaviest tiles first

    if (warp == 0) {
        tmem_alloc(&tmem_base, kT2Cols);
        tmem_relinquish();
    }
    if (threadIdx.x == 32) {
        abort_flag = 0;
        for (int s = 0; s < kRing; ++s) {
            mbar_init(&ring_full[s], 1);
            mbar_init(&ring_empty[s], 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(&a_full[s], 128);
            mbar_init(&a_empty[s], 1);
        }
        mbar_init(&g_full, 1);
        mbar_init(&s_full, 1);
        mbar_init(&y_full, 1);
        mbar_init(&y_empty, 128);
        mbar_init(&fin, 1);
        mbar_init(&q_read, 128);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tb = tmem_base;
    const uint32_t tD = tb, tA0 = tb + 128;
    const uint32_t s_base = smem_u32(sm);

    if (warp == 0) {
        // ---------------------------------------------------------- TMA producer
        // Panel sequence of a tile: (gated) U0 U1 KBhi KBmid KBlo (gate scores), Q0 K0 Q1 K1
        // (G), V0 V1 (P V), then both K panels of every cached operand.  The workers
        // release the Q panels.
        if (lane == 0 && my_tiles > 0) {
            prefetch_tensormap(&mQ);
            prefetch_tensormap(&mK);
            prefetch_tensormap(&mV);
            if (GATED && !GG) prefetch_tensormap(&mU);
            uint32_t g = 0;
            bool ok = true;
            auto slot = [&](uint32_t bytes) -> uint8_t * {
                const int s = g % kRing;
                if (!mbar_wait(&ring_empty[s], ((g / kRing) & 1) ^ 1, &abort_flag)) return nullptr;
                mbar_arrive_expect_tx(&ring_full[s], bytes);
                return sm + s * kPanel;
            };
            for (int j = 0; j < my_tiles && ok; ++j) {
                const TileInfo t = decode_tile<VAR>(a, tile_id(j));
                const int rr = t.bh * a.L + t.off + t.c * kCT;
                if (((GATED && !GG) || DECAY) && j + 1 < my_tiles) {  // rows the workers read directly
                    const TileInfo tn = decode_tile<VAR>(a, tile_id(j + 1));
                    const size_t tn_id = ((size_t)tn.bh * a.L + (size_t)tn.off + (size_t)tn.c * kCT) / kCT;
                    if (GATED && !GG) prefetch_l2(a.r_on + tn_id * kCT, kCT * 4);
                    if (DECAY) {
                        prefetch_l2(a.alpha + tn_id * kCT, kCT * 4);
                        prefetch_l2(a.beta + tn_id * kCT, kCT * 4);
                        prefetch_l2(a.lam + tn_id * kCT, kCT * 4);
                    }
                }
                uint8_t *dst = nullptr;
                // U (two K panels) and the head's key-mean image (hi, mid, lo rows); tiles of a
                // head's first segment have one memory, gate 1, and need neither
                if (GATED && !GG && t.n > 0) {
                    for (int h = 0; h < NP && ok; ++h) {
                        if (!(ok = (dst = slot(kPanel)) != nullptr)) break;
                        tma_load_2d(dst, &mU, 64 * h, rr, &ring_full[g % kRing]);
                        ++g;
                    }
                    // the key-mean rows' first D columns (a 64 x 128 panel's first D / 64 halves)
                    for (int h = 0; h < 3 && ok; ++h) {
                        if (!(ok = (dst = slot(NP * kPanel / 2)) != nullptr)) break;
                        bulk_load(dst, a.kbar_img + (size_t)t.bh * kKbImg + h * kKbPanel, NP * kPanel / 2,
                                  &ring_full[g % kRing]);
                        ++g;
                    }
                }
                for (int h = 0; h < NP && ok; ++h) {
                    if (!(ok = (dst = slot(kPanel)) != nullptr)) break;
                    tma_load_2d(dst, &mQ, 64 * h, rr, &ring_full[g % kRing]);
                    ++g;
                    if (!(ok = (dst = slot(kPanel)) != nullptr)) break;
                    tma_load_2d(dst, &mK, 64 * h, rr, &ring_full[g % kRing]);
                    ++g;
                }
                if (D == 128) {
                    for (int h = 0; h < 2 && ok; ++h) {  // keys 64h .. 64h + 63, both 64-wide halves of v
                        if (!(ok = (dst = slot(kPanel)) != nullptr)) break;
                        tma_load_2d(dst, &mV, 0, rr + 64 * h, &ring_full[g % kRing]);
                        tma_load_2d(dst + kPanel / 2, &mV, 64, rr + 64 * h, &ring_full[g % kRing]);
                        ++g;
                    }
                } else if (ok) {  // all 128 keys of the 64-wide v in one panel
                    if ((ok = (dst = slot(kPanel)) != nullptr)) {
                        tma_load_2d(dst, &mV, 0, rr, &ring_full[g % kRing]);
                        tma_load_2d(dst + kPanel / 2, &mV, 0, rr + 64, &ring_full[g % kRing]);
                        ++g;
                    }
                }
                const int items = tile_items<GATED>(t);
                for (int k = 0; k < items && ok; ++k) {
                    const uint8_t *src = item_image<GATED, VAR, D>(a, t, k);
                    for (int h = 0; h < NP && ok; ++h) {
                        if (!(ok = (dst = slot(kImg / NP)) != nullptr)) break;
                        bulk_load(dst, src + h * (kImg / NP), kImg / NP, &ring_full[g % kRing]);
                        ++g;
                    }
                }
            }
            // leave no copy in flight: the last use of every slot has landed
            int give_up = 0;
            for (uint32_t i = 0; i < (uint32_t)kRing && i < g; ++i) {
                const uint32_t u = g - 1 - i;
                mbar_wait_limit(&ring_full[u % kRing], (u / kRing) & 1, &give_up, kWaitLimitNs);
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA issuer
        if (lane == 0 && my_tiles > 0) {
            constexpr uint32_t idKm = idesc_bf16(128, 128, false, false);  // G: A and B K-major
            constexpr uint32_t idX = idesc_bf16(128, D, false, false);     // cached reads: N = D
            constexpr uint32_t idPV = idesc_bf16(128, D, false, true);     // B MN-major (V)
            uint32_t g = 0, ac = 0;
            bool ok = true;
            auto ring_ready = [&](uint32_t u) {
                return mbar_wait(&ring_full[u % kRing], (u / kRing) & 1, &abort_flag);
            };
            for (int j = 0; j < my_tiles && ok; ++j) {
                const TileInfo t = decode_tile<VAR>(a, tile_id(j));
                if (GATED && !GG && t.n > 0) {
                    // gate scores S = U (kbar_hi + kbar_mid + kbar_lo)^T into the tile's first A slot
                    // (the workers read S there, then write P over it); the slot's last readers
                    // were issued before this.  Only the first n columns are read: N = n rounded up to 16.
                    const uint32_t idS = idesc_bf16(128, 16 * ((t.n + 15) / 16), false, false);
                    const uint32_t ts = tA0 + (ac % 2) * 64;
                    bool ready = true;
                    for (int i = 0; i < NP + 3 && ready; ++i) ready = ring_ready(g + i);
                    if (!(ok = ready)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kb = 0; kb < 3; ++kb) {  // hi rows, mid rows, lo rows
                        const uint64_t dkb = make_desc_sw128(s_base + ((g + NP + kb) % kRing) * kPanel, 0, 1024);
#pragma unroll
                        for (int h = 0; h < NP; ++h) {
                            const uint64_t du = make_desc_sw128(s_base + ((g + h) % kRing) * kPanel, 0, 1024);
#pragma unroll
                            for (int kk = 0; kk < 4; ++kk)
                                mma_ss(ts, du + 2 * kk, dkb + ((8192u * h) >> 4) + 2 * kk, idS, (kb | h | kk) != 0);
                        }
                    }
                    for (int i = 0; i < NP + 3; ++i) mma_commit(&ring_empty[(g + i) % kRing]);
                    mma_commit(&s_full);
                    g += NP + 3;
                }
                if (!(ok = mbar_wait(&y_empty, (j & 1) ^ 1, &abort_flag))) break;  // D of tile j-1 drained
                // G = Q K^T
                for (int h = 0; h < NP; ++h) {
                    const uint32_t sq = g % kRing, sk = (g + 1) % kRing;
                    if (!(ok = ring_ready(g) && ring_ready(g + 1))) break;
                    tc_fence_after();
                    const uint64_t dq = make_desc_sw128(s_base + sq * kPanel, 0, 1024);
                    const uint64_t dk = make_desc_sw128(s_base + sk * kPanel, 0, 1024);
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) mma_ss(tD, dq + 2 * kk, dk + 2 * kk, idKm, (h | kk) != 0);
                    mma_commit(&ring_empty[sk]);  // the Q panel is released by the workers
                    g += 2;
                }
                if (!ok) break;
                mma_commit(&g_full);
                // D = P V once the workers have read G and written P
                const uint32_t ps = ac % 2;
                if (!(ok = mbar_wait(&a_full[ps], (ac / 2) & 1, &abort_flag))) break;
                for (int h = 0; h < NP; ++h) {  // V panels: 128 / NP keys each
                    const uint32_t s = g % kRing;
                    if (!(ok = ring_ready(g))) break;
                    tc_fence_after();
                    const uint64_t dv = make_desc_sw128(s_base + s * kPanel, kPanel / 2, 1024);
#pragma unroll
                    for (int kk = 0; kk < 8 / NP; ++kk)
                        mma_ts(tD, tA0 + ps * 64 + ((8 / NP) * h + kk) * 8, dv + kk * (2048u >> 4), idPV, (h | kk) != 0);
                    mma_commit(&ring_empty[s]);
                    ++g;
                }
                if (!ok) break;
                mma_commit(&a_empty[ps]);
                ++ac;
                // D += (g_i o Q) X_i^T
                const int items = tile_items<GATED>(t);
                for (int k = 0; k < items && ok; ++k) {
                    const uint32_t as = ac % 2;
                    if (!(ok = mbar_wait(&a_full[as], (ac / 2) & 1, &abort_flag))) break;
                    for (int h = 0; h < NP; ++h) {
                        const uint32_t s = g % kRing;
                        if (!(ok = ring_ready(g))) break;
                        tc_fence_after();
                        const uint64_t db = make_desc_sw128(s_base + s * kPanel, 0, 1024);
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) mma_ts(tD, tA0 + as * 64 + (4 * h + kk) * 8, db + 2 * kk, idX, 1);
                        mma_commit(&ring_empty[s]);
                        ++g;
                    }
                    if (!ok) break;
                    mma_commit(&a_empty[as]);
                    ++ac;
                }
                if (!ok) break;
                mma_commit(&y_full);
            }
            // leave no MMA in flight
            mma_commit(&fin);
            int give_up = 0;
            mbar_wait_limit(&fin, 0, &give_up, kWaitLimitNs);
        }
    } else {
        // ---------------------------------------------------------- workers (thread = token row)
        const int q4 = warp & 3;
        const uint32_t row = 32 * q4 + lane;
        const uint32_t lane_base = (uint32_t)(32 * q4) << 16;
        const bool leader = warp == 2 && lane == 0;  // releases the Q panels
        uint32_t ac = 0, g = 0;  // A-slot / ring counters, in step with the MMA issuer
        uint32_t scn = 0;        // tiles whose gate scores the issuer computed
        bool ok = true;
        uint32_t gm2[32];  // gate pairs of the token: (g_{2p}, g_{2p+1}); g_n is element 63
        auto claim = [&]() -> bool {  // the next A slot is free
            if (!mbar_wait(&a_empty[ac % 2], ((ac / 2) & 1) ^ 1, &abort_flag)) return false;
            tc_fence_after();
            return true;
        };
        auto publish = [&]() {  // hand the A slot to the issuer
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(&a_full[ac % 2]);
            ++ac;
        };
        float *dsm = reinterpret_cast<float *>(sm + kRing * kPanel) + q4 * 5 * kCT;  // SWLA: ell | lambda | beta_{j+1} | E | F
        for (int j = 0; j < my_tiles && ok; ++j) {
            const TileInfo t = decode_tile<VAR>(a, tile_id(j));
            const int items = tile_items<GATED>(t);
            float gn = a.mean ? 1.f / (float)(t.n + 1) : 1.f;  // Residual: 1
            // GG: this token's gates in HBM, gcol[i L] for memory i (the online one at i = n)
            const __nv_bfloat16 *gcol =
                a.gates + (size_t)t.bh * a.N * a.L + (size_t)t.off + (size_t)t.c * kCT + row;
            if (GG) gn = __bfloat162float(gcol[(size_t)t.n * a.L]);
            if (GATED && !GG && t.n > 0) {
                // the token's gates from the scores S in this tile's first A slot
                g += NP + 3;  // the U and key-mean panels, released by the issuer
                const size_t tok = (size_t)t.bh * a.L + (size_t)t.off + (size_t)t.c * kCT + row;
                const float ron = __ldg(a.r_on + tok);
                if (!(ok = mbar_wait(&s_full, scn & 1, &abort_flag))) break;
                ++scn;
                tc_fence_after();
                float sc[64];
#pragma unroll
                for (int m = 0; m < 4; ++m) {
                    if (16 * m < t.n) {
                        tmem_ld16f(tA0 + (ac % 2) * 64 + lane_base + 16 * m, sc + 16 * m);
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; ++k) sc[16 * m + k] = 0.f;
                    }
                }
                tmem_wait_ld();
                const float inv = token_gates<SSC>(sc, t.n, ron, a.topk, nullptr);
#pragma unroll
                for (int k = 0; k < 32; ++k) gm2[k] = pack_bf16x2(sc[2 * k] * inv, sc[2 * k + 1] * inv);
                gn = __bfloat162float(__high2bfloat16(*reinterpret_cast<const __nv_bfloat162 *>(&gm2[31])));
            }
            float ellt = 0.f;  // SWLA: log of A(t_c, t) for this token row
            if (DECAY) {
                const size_t tok0 = (size_t)t.bh * a.L + (size_t)t.off + (size_t)t.c * kCT;
                const ChunkDecay cd = load_chunk_decay(a.alpha, a.beta, a.lam, tok0, lane);
                const float b_up = __shfl_down_sync(0xffffffffu, cd.bet[0], 1);  // beta of token 4 (lane + 1)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    dsm[4 * lane + e] = cd.ell[e];
                    dsm[kCT + 4 * lane + e] = cd.lam[e];
                    dsm[2 * kCT + 4 * lane + e] = e < 3 ? cd.bet[e + 1] : (lane < 31 ? b_up : 0.f);
                }
                __syncwarp();
                // Per 32-column block h with reference m_h = ell_{32h}: E_j = lambda_j exp(m_h - ell_j),
                // F_j = beta_{j+1} exp(m_h - ell_{j+1}), so c_{t,j} = exp(ell_t - m_h) (E_j + [j<t] F_j).
#pragma unroll
                for (int hb = 0; hb < 4; ++hb) {
                    const int cj = 32 * hb + lane;
                    const float m = dsm[32 * hb];
                    dsm[3 * kCT + cj] = dsm[kCT + cj] * __expf(m - dsm[cj]);
                    dsm[4 * kCT + cj] = cj < kCT - 1 ? dsm[2 * kCT + cj] * __expf(m - dsm[cj + 1]) : 0.f;
                }
                __syncwarp();
                ellt = dsm[row];
            }
            // the token's query row from the Q panels (SWIZZLE_128B: 16-byte chunk c of
            // row r sits at chunk c ^ (r % 8)), read while G runs
            uint32_t qp[32 * NP];
            if (!(ok = mbar_wait(&ring_full[g % kRing], (g / kRing) & 1, &abort_flag) &&
                       (NP == 1 || mbar_wait(&ring_full[(g + 2) % kRing], ((g + 2) / kRing) & 1, &abort_flag))))
                break;
#pragma unroll
            for (int h = 0; h < NP; ++h) {
                const uint8_t *pq = sm + ((g + 2 * h) % kRing) * kPanel + row * 128;
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint4 x = *reinterpret_cast<const uint4 *>(pq + ((c ^ (row & 7)) << 4));
                    qp[32 * h + 4 * c] = x.x;
                    qp[32 * h + 4 * c + 1] = x.y;
                    qp[32 * h + 4 * c + 2] = x.z;
                    qp[32 * h + 4 * c + 3] = x.w;
                }
            }
            mbar_arrive(&q_read);
            if (!(ok = mbar_wait(&g_full, j & 1, &abort_flag))) break;
            tc_fence_after();
            if (leader) {  // G and every worker are done with the Q panels
                if (!(ok = mbar_wait(&q_read, j & 1, &abort_flag))) break;
                mbar_arrive(&ring_empty[g % kRing]);
                if (NP == 2) mbar_arrive(&ring_empty[(g + 2) % kRing]);
            }
            // P = g_n * mask(G), key column c <= token row
            if (!(ok = claim())) break;
            {
                const uint32_t ta = tA0 + (ac % 2) * 64 + lane_base;
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    uint32_t x[32], o[16];
                    tmem_ld32(tD + lane_base + 32 * h, x);
                    tmem_wait_ld();
                    if (!DECAY) {
#pragma unroll
                        for (int i = 0; i < 16; ++i) {
                            const uint32_t c0 = 32 * h + 2 * i;
                            o[i] = pack_bf16x2(c0 <= row ? gn * __uint_as_float(x[2 * i]) : 0.f,
                                               c0 + 1 <= row ? gn * __uint_as_float(x[2 * i + 1]) : 0.f);
                        }
                    } else if (32 * h > 32 * q4 + 31) {  // the whole block is above every row of the warp
#pragma unroll
                        for (int i = 0; i < 16; ++i) o[i] = 0u;
                    } else {
                        // P_tj = g_n c_{t,j} G_tj, c_{t,j} = lambda_j A(j,t) + [j<t] beta_{j+1} A(j+1,t).
                        // Factored through the block's reference when the block's decay range keeps
                        // E and F finite; element by element otherwise (strong decay).
                        const float m = dsm[32 * h];
                        const bool factored = m - dsm[32 * h + 32 < kCT ? 32 * h + 32 : kCT - 1] <= 80.f &&
                                              dsm[kCT - 1] - m <= 80.f;  // warp-uniform
                        if (factored) {
                            const float et = gn * __expf(ellt - m);
                            auto coef = [&](uint32_t cj) -> float {
                                if (cj > row) return 0.f;
                                return dsm[3 * kCT + cj] + (cj < row ? dsm[4 * kCT + cj] : 0.f);
                            };
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const uint32_t c0 = 32 * h + 2 * i;
                                o[i] = pack_bf16x2(et * coef(c0) * __uint_as_float(x[2 * i]),
                                                   et * coef(c0 + 1) * __uint_as_float(x[2 * i + 1]));
                            }
                        } else {
                            auto coef = [&](uint32_t cj) -> float {
                                if (cj > row) return 0.f;
                                float cf = dsm[kCT + cj] * __expf(ellt - dsm[cj]);
                                if (cj < row) cf += dsm[2 * kCT + cj] * __expf(ellt - dsm[cj + 1]);
                                return cf;
                            };
#pragma unroll
                            for (int i = 0; i < 16; ++i) {
                                const uint32_t c0 = 32 * h + 2 * i;
                                o[i] = pack_bf16x2(gn * coef(c0) * __uint_as_float(x[2 * i]),
                                                   gn * coef(c0 + 1) * __uint_as_float(x[2 * i + 1]));
                            }
                        }
                    }
                    tmem_st16(ta + 16 * h, o);
                }
            }
            publish();
            // cached operands: g_i o Q
            const __nv_bfloat16 *gl = reinterpret_cast<const __nv_bfloat16 *>(gm2);
            // GG: item k's gate from HBM, loaded one item ahead
            auto item_gate = [&](int k) -> __nv_bfloat16 {
                const int i = t.c > 0 ? k - 1 : k;
                return gcol[(size_t)(i < 0 ? t.n : i) * a.L];
            };
            __nv_bfloat16 gnext = GG && items > 0 ? item_gate(0) : __float2bfloat16_rn(0.f);
#pragma unroll 1
            for (int k = 0; k < items; ++k) {
                __nv_bfloat162 gam2 = __float2bfloat162_rn(gn);  // Residual: 1, Mean: 1 / (n + 1)
                const bool prefix = t.c > 0 && k == 0;  // item 0 of a chunk c > 0 is its prefix state (gate g_n)
                if (GG) {
                    gam2 = __bfloat162bfloat162(gnext);
                    if (k + 1 < items) gnext = item_gate(k + 1);
                } else if (GATED) {
                    const int i = t.c > 0 ? k - 1 : k;
                    gam2 = __bfloat162bfloat162(i < 0 ? __float2bfloat16_rn(gn) : gl[i]);
                }
                if (DECAY && prefix) gam2 = __float2bfloat162_rn(gn * __expf(ellt));  // A(t_c, t) S^_c q_t
                const bool scale = GATED || (DECAY && prefix) || a.mean;
                if (!(ok = claim())) break;
                const uint32_t ta = tA0 + (ac % 2) * 64 + lane_base;
#pragma unroll
                for (int m = 0; m < NP; ++m) {
                    uint32_t r[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        if (scale) {
                            __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162 *>(&qp[32 * m + i]);
                            __nv_bfloat162 pr = __hmul2(x, gam2);
                            r[i] = *reinterpret_cast<uint32_t *>(&pr);
                        } else {
                            r[i] = qp[32 * m + i];
                        }
                    }
                    tmem_st32(ta + 32 * m, r);
                }
                publish();
            }
            if (!ok) break;
            g += NP * (3 + items);  // Q, K, V and the cached operands
            // drain: read D in the 16x256b layout (a quad of threads holds 8 consecutive
            // columns of a row), release it, then transpose within each quad by shuffles
            // so that every thread stores 16 contiguous bytes: 8 rows x 64 bytes per store
            if (!(ok = mbar_wait(&y_full, j & 1, &abort_flag))) break;
            tc_fence_after();
            uint32_t yb[64];  // [lane half][column half]: 8 pairs of row A, then 8 of row B
#pragma unroll
            for (int hl = 0; hl < 2; ++hl)
#pragma unroll
                for (int ch = 0; ch < NP; ++ch) {
                    uint32_t x[32];
                    tmem_ld_16x256b_x8(tD + ((uint32_t)(32 * q4 + 16 * hl) << 16) + 64 * ch, x);
                    tmem_wait_ld();
#pragma unroll
                    for (int b = 0; b < 8; ++b) {
                        yb[16 * (2 * hl + ch) + b] = pack_bf16x2(__uint_as_float(x[4 * b]), __uint_as_float(x[4 * b + 1]));
                        yb[16 * (2 * hl + ch) + 8 + b] = pack_bf16x2(__uint_as_float(x[4 * b + 2]), __uint_as_float(x[4 * b + 3]));
                    }
                }
            tc_fence_before();
            mbar_arrive(&y_empty);
            {
                const int c = lane & 3;
                __nv_bfloat16 *ytile = a.y + ((size_t)t.bh * a.L + (size_t)t.off + (size_t)t.c * kCT) * a.d;
#pragma unroll
                for (int g4 = 0; g4 < 16; ++g4) {  // (lane half, column half, row A/B, block group) groups of 4 pairs
                    if (((g4 >> 2) & 1) >= NP) continue;  // D = 64: one column half
                    uint32_t *xv = yb + 4 * g4;
                    // 4 x 4 transpose across the quad: thread c ends with block (4 (g4 % 2) + c)
                    // of its row, columns in order
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
                    const int hl = g4 >> 3, ch = (g4 >> 2) & 1, rb = (g4 >> 1) & 1, bg = g4 & 1;
                    const int r = 32 * q4 + 16 * hl + 8 * rb + (lane >> 2);
                    *reinterpret_cast<uint4 *>(ytile + (size_t)r * a.d + 64 * ch + 8 * (4 * bg + c)) =
                        make_uint4(xv[0], xv[1], xv[2], xv[3]);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tb, kT2Cols);
    }
    if (threadIdx.x == 0 && abort_flag) atomicExch(&g_tc_abort, 1);
}

// ============================================================================
// Host launchers, one instantiation per head dimension D (= d).
// ============================================================================

// Gates through HBM: the routed aggregations with more than 64 segments.
inline bool tc_hbm_gates(const Problem &p) { return mode_uses_u(p.mode) && p.N > 64; }

inline size_t img_bytes(const Problem &p) { return (size_t)p.d * p.d * 2; }

// Scratch of the forward over constant segments: state images [BH][N], prefix-state
// images [BH][N][CPS], key-mean images [BH][NB], r_on [BH][L], then the prefix sums of
// the states [BH][N] (Residual / Mean) or the gates [BH][N][L] bf16 (more than 64 segments).
inline size_t forward_scratch_bytes(const Problem &p)
{
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT, NB = (N + 63) / 64, im = img_bytes(p);
    size_t b = pad256(BH * N * im) + pad256(BH * N * CPS * im) + pad256(BH * NB * kKbImg) +
               pad256(sizeof(float) * BH * p.L);
    if (!mode_uses_u(p.mode)) b += pad256(BH * N * im);
    if (tc_hbm_gates(p)) b += pad256(sizeof(__nv_bfloat16) * BH * N * p.L);
    return b;
}

// Tensor maps of the forward: 64-column boxes of 128 rows (V also of 64 rows).
struct FwdMaps {
    CUtensorMap q, k, v, v64, u;
};

inline bool make_fwd_maps(const Problem &p, const FwdArgs &fa, FwdMaps *m)
{
    const unsigned long long rows = (unsigned long long)p.BH * p.L;
    if (!make_tmap_bf16_sw128(&m->q, fa.q, rows, p.d, 128) || !make_tmap_bf16_sw128(&m->k, fa.k, rows, p.d, 128) ||
        !make_tmap_bf16_sw128(&m->v, fa.v, rows, p.d, 128) || !make_tmap_bf16_sw128(&m->v64, fa.v, rows, p.d, 64))
        return false;
    if (mode_uses_u(p.mode)) return make_tmap_bf16_sw128(&m->u, fa.u, rows, p.d, 128);
    m->u = m->k;
    return true;
}

template <int D>
cudaError_t forward_impl(const Problem &p, const FwdArgs &fa, void *scratch, cudaStream_t s)
{
    const bool gated = mode_uses_u(p.mode);
    const size_t BH = p.BH, N = p.N, CPS = p.C / kCT, im = img_bytes(p);
    uint8_t *base = static_cast<uint8_t *>(scratch);
    TcArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(fa.q);
    a.u = static_cast<const __nv_bfloat16 *>(fa.u);
    a.y = static_cast<__nv_bfloat16 *>(fa.y);
    a.states = fa.states;
    a.states_img = base;
    base += pad256(BH * N * im);
    a.spre_img = base;
    base += pad256(BH * N * CPS * im);
    a.kbar_img = base;
    base += pad256(BH * ((N + 63) / 64) * kKbImg);
    a.r_on = reinterpret_cast<float *>(base);
    base += pad256(sizeof(float) * BH * p.L);
    a.prefix_img = gated ? nullptr : base;
    const bool gg = tc_hbm_gates(p);  // routed, so there are no prefix-sum images
    __nv_bfloat16 *gates = gg ? reinterpret_cast<__nv_bfloat16 *>(base) : nullptr;
    a.gates = gates;
    a.sel_out = fa.sel_out;
    a.topk = p.topk;
    a.mean = p.mode == MC_MEAN;
    a.BH = p.BH;
    a.L = p.L;
    a.C = p.C;
    a.N = p.N;
    a.CPS = (int)CPS;
    a.d = p.d; a.NB = (p.N + 63) / 64;
    a.num_tiles = (int)(BH * N * CPS);
    // heads per readout group: when every head's state images (read by every later tile of their head;
    // the prefix images are read once) exceed 48 MB, groups whose images take about 32 MB of the L2,
    // as equal as possible
    {
        const size_t per_head = N * im;
        int hg = (int)((size_t)32 * 1024 * 1024 / (per_head > 0 ? per_head : 1));
        hg = hg < 8 ? 8 : hg > p.BH ? p.BH : hg;
        if (BH * per_head <= (size_t)48 * 1024 * 1024) hg = p.BH;
        const int groups = (p.BH + hg - 1) / hg;
        a.hg = (p.BH + groups - 1) / groups;
    }
    FwdMaps m;
    if (!make_fwd_maps(p, fa, &m)) return cudaErrorInvalidValue;
    const int sms = sm_count();
    cudaError_t e;

    profile_call_start(s);
    const bool decay = fa.alpha != nullptr;
    a.alpha = fa.alpha;
    a.beta = fa.beta;
    a.lam = fa.lam;
    {
        auto k1 = gated ? (decay ? seg_state_tc<true, true, false, D> : seg_state_tc<true, false, false, D>)
                        : (decay ? seg_state_tc<false, true, false, D> : seg_state_tc<false, false, false, D>);
        const size_t smem1 = decay ? t1_smem_bytes<true, D>() : t1_smem_bytes<false, D>();
        e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
        if (e != cudaSuccess) return e;
        const int nseg = (int)(BH * N), slots1 = (D == 64 ? 2 : 1) * sms;  // D = 64: two CTAs per SM
        k1<<<nseg < slots1 ? nseg : slots1, kT1Threads, smem1, s>>>(m.k, m.v, m.u, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "seg_state_tc");
    }
    if (!gated) {
        dim3 grid((D * D + 255) / 256, (unsigned)BH);
        prefix_images<D><<<grid, 256, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "prefix_images");
    }
    if (gg) {  // more than 64 segments: every token's gates through HBM
        if (decay) return cudaErrorInvalidValue;
        if ((e = launch_gates_gen(p, fa.u, a.kbar_img, a.r_on, gates, s)) != cudaSuccess) return e;
        profile_after_kernel(s, "gates_tc");
    }
    {
        const bool ssc = p.mode == MC_SSC;
        auto k2 = !gated ? (decay ? readout_tc<false, true, false, false, false, D> : readout_tc<false, false, false, false, false, D>)
                  : gg   ? (ssc ? readout_tc<true, false, true, true, false, D> : readout_tc<true, false, false, true, false, D>)
                  : ssc  ? (decay ? readout_tc<true, true, true, false, false, D> : readout_tc<true, false, true, false, false, D>)
                         : (decay ? readout_tc<true, true, false, false, false, D> : readout_tc<true, false, false, false, false, D>);
        e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kT2Smem);
        if (e != cudaSuccess) return e;
        const int slots = kT2CtasPerSm * sms;
        const int grid = a.num_tiles < slots ? a.num_tiles : slots;
        k2<<<grid, kT2Threads, kT2Smem, s>>>(m.q, m.k, m.v64, m.u, a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "readout_tc");
    }
    return cudaSuccess;
}

// ---------------------------------------------------------------------------
// The state form over given segment boundaries: segments 0 .. Nseg-1 of every head
// are whole 128-token chunks (start and length multiples of 128).  Scratch layout:
// state images [BH][N], prefix-state images [BH][NC], key-mean image [BH], the online
// scores [BH][L], for Residual / Mean the prefix sums of the states [BH][N], then the pieces'
// own states [BH][nslots][d][d] and key sums [BH][nslots][d] (fp32).
// ---------------------------------------------------------------------------
inline size_t segments_scratch_bytes(const Problem &p, int NC, int nslots)
{
    const size_t BH = p.BH, N = p.N, im = img_bytes(p);
    size_t b = pad256(BH * N * im) + pad256(BH * (size_t)NC * im) + pad256(BH * kKbImg) +
               pad256(sizeof(float) * BH * p.L);
    if (!mode_uses_u(p.mode)) b += pad256(BH * N * im);
    b += pad256(sizeof(float) * BH * nslots * p.d * p.d) + pad256(sizeof(float) * BH * nslots * p.d);
    return b;
}

inline TcArgs segments_args(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch)
{
    const size_t BH = p.BH, N = p.N, im = img_bytes(p);
    uint8_t *base = static_cast<uint8_t *>(scratch);
    TcArgs a{};
    a.q = static_cast<const __nv_bfloat16 *>(fa.q);
    a.u = static_cast<const __nv_bfloat16 *>(fa.u);
    a.y = static_cast<__nv_bfloat16 *>(fa.y);
    a.states = fa.states;
    a.states_img = base;
    base += pad256(BH * N * im);
    a.spre_img = base;
    base += pad256(BH * (size_t)tb.NC * im);
    a.kbar_img = base;
    base += pad256(BH * kKbImg);
    a.r_on = reinterpret_cast<float *>(base);
    base += pad256(sizeof(float) * BH * p.L);
    a.prefix_img = mode_uses_u(p.mode) ? nullptr : base;
    if (!mode_uses_u(p.mode)) base += pad256(BH * N * im);
    a.ptot = reinterpret_cast<float *>(base);
    base += pad256(sizeof(float) * BH * tb.nslots * p.d * p.d);
    a.pks = reinterpret_cast<float *>(base);
    a.nslots = tb.nslots;
    a.kbar_out = mode_uses_u(p.mode) ? fa.kbar : nullptr;  // fp32 key means, for the segments after
    a.topk = p.topk;
    a.mean = p.mode == MC_MEAN;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.CPS = 0; a.d = p.d; a.NB = 1;
    a.sg_off = tb.off;
    a.sg_cbase = tb.cbase;
    a.vtiles = tb.tiles;
    a.Nseg = tb.Nseg;
    a.NC = tb.NC;
    a.num_tiles = p.BH * tb.NC;
    return a;
}

template <int D>
cudaError_t state_segments_impl(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch,
                                cudaStream_t s)
{
    const bool gated = mode_uses_u(p.mode);
    TcArgs a = segments_args(p, fa, tb, scratch);
    FwdMaps m;
    if (!make_fwd_maps(p, fa, &m)) return cudaErrorInvalidValue;
    cudaError_t e;
    auto k1 = gated ? seg_state_tc<true, false, true, D> : seg_state_tc<false, false, true, D>;
    const size_t smem1 = t1_smem_bytes<false, D>();
    if ((e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1)) != cudaSuccess) return e;
    const int sms = (D == 64 ? 2 : 1) * sm_count();  // state CTAs at once (D = 64: two per SM)
    if (tb.n1 > 0) {  // the pieces' own states first: every later piece starts from their sums
        TcArgs a1 = a;
        a1.units = tb.units1;
        a1.NU = tb.n1;
        a1.totals = 1;
        const int units = p.BH * tb.n1;
        k1<<<units < sms ? units : sms, kT1Threads, smem1, s>>>(m.k, m.v, m.u, a1);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "seg_piece_sums_tc");
    }
    a.units = tb.units2;
    a.NU = tb.n2;
    a.totals = 0;
    const int units = p.BH * tb.n2;
    k1<<<units < sms ? units : sms, kT1Threads, smem1, s>>>(m.k, m.v, m.u, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_after_kernel(s, "seg_state_tc");
    return cudaSuccess;
}

// After every segment's state exists (fp32, fa.states): the Residual prefix sums and the
// readout of the tokens of segments 0 .. Nseg-1.
template <int D>
cudaError_t readout_segments_impl(const Problem &p, const FwdArgs &fa, const TcSegTables &tb, void *scratch,
                                  cudaStream_t s)
{
    const bool gated = mode_uses_u(p.mode);
    TcArgs a = segments_args(p, fa, tb, scratch);
    FwdMaps m;
    if (!make_fwd_maps(p, fa, &m)) return cudaErrorInvalidValue;
    cudaError_t e;
    if (!gated) {
        dim3 grid((D * D + 255) / 256, (unsigned)p.BH);
        prefix_images<D><<<grid, 256, 0, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "prefix_images");
    }
    auto k2 = !gated ? readout_tc<false, false, false, false, true, D>
              : p.mode == MC_SSC ? readout_tc<true, false, true, false, true, D> : readout_tc<true, false, false, false, true, D>;
    if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kT2Smem)) != cudaSuccess) return e;
    const int slots = kT2CtasPerSm * sm_count();
    k2<<<a.num_tiles < slots ? a.num_tiles : slots, kT2Threads, kT2Smem, s>>>(m.q, m.k, m.v64, m.u, a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_after_kernel(s, "readout_tc");
    return cudaSuccess;
}

// Read and clear this translation unit's abort flag.
inline cudaError_t take_tc_abort(int *was_set)
{
    int v = 0;
    cudaError_t e = cudaMemcpyFromSymbol(&v, g_tc_abort, sizeof(int));
    if (e != cudaSuccess) return e;
    *was_set = v;
    if (v) {
        v = 0;
        e = cudaMemcpyToSymbol(g_tc_abort, &v, sizeof(int));
    }
    return e;
}

}  // namespace
}  // namespace mc
