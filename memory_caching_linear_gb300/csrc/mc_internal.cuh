// mc_internal.cuh -- shared declarations of the CUDA path of the Memory Caching
// forward (device helpers, launch argument blocks, kernel launchers).
//
// Data flow of one forward (per batch*head "bh", segment n, token t):
//   seg_scan   : per (bh, segment) -- the segment's final state M^(n) (fp32,
//                the `states` output), its key mean kbar_n, the online read
//                O_on[t] = M_t^(n) q_t, and the online gate score
//                r_on[t] = <u_t, mean of the segment's keys up to t>.
//   readout    : per (bh, segment, token tile) -- gates over the cached
//                segments and the online memory, and
//                y_t = g_{t,n} O_on[t] + sum_{i<n} g_{t,i} M^(i) q_t.
//   ssc_select : the SSC router alone (the same score and ranking code).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "mc.h"

namespace mc {

constexpr int kMaxTopk = 64;  // SSC selections kept per token on the device
constexpr int kPieceLen = 512;  // tokens per piece when the FFMA scan splits a long segment

// Aggregations whose gates come from the router <u_t, pooled keys>; Residual and
// Mean weigh every memory the same and never read u.
__host__ __device__ inline bool mode_uses_u(int mode) { return mode == MC_GRM || mode == MC_SOUP || mode == MC_SSC; }

struct Problem {
    int B, H, L, d, C, N, mode, topk;
    int BH;
    bool bf16;
};

// Everything one forward needs on the device.  Pointers are device pointers.
struct FwdArgs {
    const void *q, *k, *v, *u;  // [BH][L][d], element type per Problem::bf16
    void *y;                    // [BH][L][d]
    float *states;              // [BH][N][d][d]
    float *O_on;                // [BH][L][d]   scratch
    float *r_on;                // [BH][L]      scratch
    float *kbar;                // [BH][N][d]   scratch
    int32_t *sel_out;           // [BH][L][topk] (ssc_select only)
    const float *alpha, *beta, *lam;  // SWLA per-token scalars [BH][L]; all null = plain update
    const int32_t *seg_off;     // optional [N+1] segment boundaries (device); then C is the longest segment
    float *kpre_tiles;          // backward state kernel only: keys before each 64-token tile [BH][N][C/64][d]
    // Optional split of long segments for the FFMA scan (null: one CTA walks a whole segment).
    // Segment n is pieces [seg_pieces[n], seg_pieces[n+1]) of piece_len tokens (the last ragged).
    const int32_t *seg_pieces;  // [N+1] first piece of each segment (device)
    const int32_t *piece_seg;   // [npieces] segment of each piece (device)
    int npieces, piece_len;
    float *piece_state;         // [BH][npieces][d][d] scratch: a piece's own state, then the state before it
    float *piece_ksum;          // [BH][npieces][d] scratch: the same for the key sums
    int BH, L, C, N, mode, topk;
};

// Segment n's tokens [seg_begin, seg_end): constant length C, or the given boundaries.
__device__ __forceinline__ int seg_begin(const FwdArgs &a, int n) { return a.seg_off ? a.seg_off[n] : n * a.C; }
__device__ __forceinline__ int seg_end(const FwdArgs &a, int n)
{
    return a.seg_off ? a.seg_off[n + 1] : min((n + 1) * a.C, a.L);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(__nv_bfloat16 x) { return __bfloat162float(x); }
template <typename T> __device__ __forceinline__ T from_f(float x);
template <> __device__ __forceinline__ float from_f<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float x) { return __float2bfloat16_rn(x); }

// Gate score <u_t, kbar_i> in fp32 on the CUDA cores: four interleaved partial sums
// (columns 4j + r into p_r, j ascending) added as (p0 + p1) + (p2 + p3), i.e. four
// independent dependency chains; d is a multiple of 4.  Every CUDA-core kernel that
// needs a router score calls this one function, so the SSC ranking seen by
// mc_ssc_select is bit-identical to the one the forward uses.  u_row and kb may each be
// in shared or global memory.
__device__ __forceinline__ float gate_score(const float *__restrict__ u_row, const float *__restrict__ kb, int d)
{
    float p0 = 0.f, p1 = 0.f, p2 = 0.f, p3 = 0.f;
#pragma unroll 4
    for (int c = 0; c < d; c += 4) {
        p0 = fmaf(u_row[c], kb[c], p0);
        p1 = fmaf(u_row[c + 1], kb[c + 1], p1);
        p2 = fmaf(u_row[c + 2], kb[c + 2], p2);
        p3 = fmaf(u_row[c + 3], kb[c + 3], p3);
    }
    return (p0 + p1) + (p2 + p3);
}

// Insert (val, idx) into a top-k list kept sorted by value descending, index
// ascending.  Candidates arrive in increasing idx, so an equal value goes after
// the ones already there (equal scores -> lower segment index first).
__device__ __forceinline__ void topk_insert(float *vals, int *idxs, int &count, int k, float val, int idx)
{
    int p = count;
    while (p > 0 && vals[p - 1] < val) --p;
    if (p >= k) return;
    int last = count < k ? count : k - 1;
    for (int j = last; j > p; --j) {
        vals[j] = vals[j - 1];
        idxs[j] = idxs[j - 1];
    }
    vals[p] = val;
    idxs[p] = idx;
    if (count < k) ++count;
}

// One decoding step (k_decode.cu).  Caches: states [BH][nmax][d][d], kbar
// [BH][nmax][d], online [BH][d][d], ksum [BH][d] (fp32); the token's q, k, v, u
// and y are [BH][d] (bf16 or fp32); gates is scratch [BH][kDecGateWords].
constexpr int kDecMaxN = 65;        // cached segments (at most 64) plus the online memory
constexpr int kDecGateWords = 132;  // per-head gate record of the decoding step (k_decode.cu)
struct DecodeArgs {
    const void *q, *k, *v, *u;
    void *y;
    float *states, *kbar, *online, *ksum, *gates;
    int BH, d, C, mode, topk, t, nmax;
    bool bf16;
};
cudaError_t launch_decode_step(const DecodeArgs &a, cudaStream_t s);

// Stream-ordered scratch from the library's per-device pool (mc_api.cu).
cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t s);

// Kernel-boundary profiling (mc_profile_begin): call_start() before the first
// kernel of a forward, after_kernel(name) after each launch.
void profile_call_start(cudaStream_t s);
void profile_after_kernel(cudaStream_t s, const char *name);

// Tensor-core state-form path (k_tc.cu): bf16, d = 64 or 128, seg_len % 128 == 0,
// L % seg_len == 0; the routed aggregations up to 512 segments (beyond 64 the gates go
// through HBM), SSC topk <= 16.  tc_fused_gates: N <= 64, the gates formed in the readout
// (the SWLA update, the stand-alone router and the backward need this).
bool tc_supported(const Problem &p);
bool tc_fused_gates(const Problem &p);
// The state form over given segment boundaries (mc_forward_segments): segments 0 .. Nseg-1
// are whole 128-token chunks; off [Nseg + 1] their first tokens (device), cbase [Nseg] their
// first chunks (off / 128), tiles [NC] the readout's (segment, chunk) slots heaviest first.
// units1 [n1] are the pieces whose own state and key sums the first pass forms (slots 0 .. nslots-1),
// units2 [n2] every piece, each starting from the totals of the pieces before it (state form walk).
struct TcSegTables {
    const int32_t *off, *cbase;
    const int2 *tiles;
    int Nseg, NC;
    const int4 *units1, *units2;
    int n1, n2, nslots;
};
size_t tc_segments_scratch_bytes(const Problem &p, int NC, int nslots);
cudaError_t launch_state_tc_segments(const Problem &p, const FwdArgs &a, const TcSegTables &tb, void *scratch,
                                     cudaStream_t s);
cudaError_t launch_readout_tc_segments(const Problem &p, const FwdArgs &a, const TcSegTables &tb, void *scratch,
                                       cudaStream_t s);
size_t tc_scratch_bytes(const Problem &p);
cudaError_t launch_forward_tc(const Problem &p, const FwdArgs &a, void *scratch, cudaStream_t s);
// The d = 64 instantiations of the forward and segment launchers (k_tc64.cu).
cudaError_t launch_forward_tc64(const Problem &p, const FwdArgs &a, void *scratch, cudaStream_t s);
cudaError_t launch_state_tc_segments64(const Problem &p, const FwdArgs &a, const TcSegTables &tb, void *scratch,
                                       cudaStream_t s);
cudaError_t launch_readout_tc_segments64(const Problem &p, const FwdArgs &a, const TcSegTables &tb, void *scratch,
                                         cudaStream_t s);
cudaError_t take_tc64_abort(int *was_set);
// The readout of the tokens [t_tail, L) (fewer than 128, the segments after the tensor-core
// ones of a given segmentation; k_tail.cu): needs O_on, r_on of those tokens and the fp32
// states and key means of every segment; bf16 inputs, d = 64 or 128, N <= 64.
size_t tail_scratch_bytes(const Problem &p, int t_tail);
cudaError_t launch_tail_readout(const Problem &p, const FwdArgs &a, int t_tail, void *scratch, cudaStream_t s);
size_t tc_select_scratch_bytes(const Problem &p);
cudaError_t launch_ssc_select_tc(const Problem &p, const FwdArgs &a, void *scratch, cudaStream_t s);
// The forward's state kernel alone, for the tensor-core backward: images of the cached
// states [BH][N] and of the chunks' prefix states [BH][N][C/128] (32 KB each, 128x128
// bf16, two 64-column 128-byte-swizzled panels, row = value dim), and r_on [BH][L];
// routed aggregations also get the fp32 key means (fa.kbar) and the keys before each
// 64-token tile (fa.kpre_tiles).
struct TcImages {
    const uint8_t *states_img, *spre_img, *kbar_img;
    const float *r_on;
};
size_t tc_state_scratch_bytes(const Problem &p);
cudaError_t launch_state_tc(const Problem &p, const FwdArgs &fa, void *scratch, TcImages *out, cudaStream_t s);
// The backward's gates on the tensor cores (routed modes): g_{t,i} to gam [BH][N][L] and the
// online gate to word 2 of tok [BH][L][kBwdTokWords].
cudaError_t launch_bwd_gates_tc(const Problem &p, const void *u, const TcImages &img, float *gam, float *tok, cudaStream_t s);
// Reads and clears the device-side record of an abandoned bounded wait.
cudaError_t take_device_abort(int *was_set);

// General tensor-core path (k_gen.cu): bf16, d in {64, 128}, seg_len a multiple of 16,
// any L (a ragged last segment), N <= 512 for the routed aggregations, SSC topk <= 16.
// The cached readout runs in the factorised form sum_j g_{t,seg(j)} v_j (k_j . q_t).
bool gen_supported(const Problem &p);
size_t gen_scratch_bytes(const Problem &p);
cudaError_t launch_forward_gen(const Problem &p, const FwdArgs &a, void *scratch, cudaStream_t s);
size_t gen_select_scratch_bytes(const Problem &p);
cudaError_t launch_ssc_select_gen(const Problem &p, const FwdArgs &a, void *scratch, cudaStream_t s);
cudaError_t take_gen_abort(int *was_set);
// The general path's gate kernel for the state form with more than 64 segments.
cudaError_t launch_gates_gen(const Problem &p, const void *u, uint8_t *kbar_img, float *r_on, __nv_bfloat16 *gates,
                             cudaStream_t s);

// SIMT kernels (any d in {16,32,64,128}, fp32 or bf16 inputs).
cudaError_t launch_seg_scan_simt(const Problem &p, const FwdArgs &a, cudaStream_t s);
cudaError_t launch_readout_simt(const Problem &p, const FwdArgs &a, cudaStream_t s);
cudaError_t launch_kbar_simt(const Problem &p, const FwdArgs &a, cudaStream_t s);
cudaError_t launch_ssc_select_simt(const Problem &p, const FwdArgs &a, cudaStream_t s);

// Backward pass (k_bwd_simt.cu).  Inputs q, k, v, u, dy and outputs dq, dk, dv, du
// are [BH][L][d] (element type per Problem::bf16); the rest is fp32 scratch.
constexpr int kBwdTokWords = 5;  // per token: softmax max m, sum z, online gate, delta = sum g dg, pool weight w
struct BwdArgs {
    const void *q, *k, *v, *u, *dy;
    void *dq, *dk, *dv, *du;
    const float *states;  // [BH][N][d][d] cached states (recomputed forward)
    const float *kbar;    // [BH][N][d]
    const float *r_on;    // [BH][L]
    const float *O_on;    // [BH][L][d]  M_t q_t (online read)
    const float *X_on;    // [BH][L][d]  M_t^T dy_t
    float *G;             // [BH][N][d][d]  sum_t g_{t,i} dy_t q_t^T per cached segment (tensor-core path:
                          // [BH][N] x 32 KB bf16 operand images)
    float *dkbar;         // [BH][N][d]  gradient of the key means (accumulated)
    float *tok;           // [BH][L][kBwdTokWords]
    int32_t *sel_idx;     // SSC: [BH][L][topk] selected segments (segment order, -1 padded)
    float *sel_g;         // SSC: [BH][L][topk] their gates
    float *gam;           // [BH][N][L] gates of the cached segments, for the tensor-core G (routed modes), or null
    const float *dg_in;   // [BH][N][L] dy_t . M^(i) q_t from the tensor cores, or null (computed here)
    const float *dq_in;   // [BH][L][d] dq from the tensor cores (all of it when X_on is null), or null (written already)
    const float *dgon_in; // [BH][L] dy_t . M_t q_t from the tensor cores, or null (from O_on)
    const float *dg_in2, *dgon_in2;  // second partial sums of dg_in and dgon_in (added to them), or null
    float *dr;            // [BH][N][L] the score gradients g (dg - delta) (may alias dg_in), or null
    __nv_bfloat16 *dr_hi, *dr_lo;  // tensor-core path: dr as two exact bf16 terms [BH][Np][L] (rows n .. Np of a
                                   // segment-n token zero up to the next multiple of 16), or null
    int Np;               // N rounded up to a multiple of 16
    float *kpre_tiles;    // [BH][N][ceil(C/64)][d] keys of each segment before each 64-token tile, or null
    float *kv_gw;         // [2][BH][L] the online gate and the pooled-key weight w per token (tensor-core path)
    int BH, L, C, N, mode, topk;
};
size_t backward_scratch_bytes(const Problem &p);
// Tensor-core pieces of the backward (k_bwd_tc.cu): bf16, d in {64, 128}, seg_len % 128 == 0,
// L % seg_len == 0, N <= 64.
bool bwd_tc_supported(const Problem &p);
cudaError_t launch_bwd_G_tc(const Problem &p, const void *dy, const void *q, const float *gam, uint8_t *G, cudaStream_t s);
// gw: [2][BH][L], the online gate of every token, then its pooled-key weight w (routed aggregations).
cudaError_t launch_bwd_kv_tc(const Problem &p, const void *q, const void *k, const void *v, const void *u, const void *dy,
                             const uint8_t *G, const float *gw, const float *dkbar, void *dk, void *dv, cudaStream_t s);
size_t bwd_cached_scratch_bytes(const Problem &p);
// dq (bf16 [BH][L][d]) is written whole; dg ([BH][N][L]) and dg_on ([BH][L]) go to scratch as two
// partial sums each (one per column half), the second BH*N*L (BH*L) floats after the first.
cudaError_t launch_bwd_cached_tc(const Problem &p, const void *q, const void *k, const void *v, const void *dy,
                                 const TcImages &img, const float *gam, const float *tok, void *dq, void *scratch,
                                 float **dg_out, float **dgon_out, cudaStream_t s);
cudaError_t take_bwd_abort(int *was_set);
// The key-mean gradients on the tensor cores: dkbar [BH][N][d] += sum_t dr_{t,i} u_t from the
// route kernel's hi / lo planes of dr.
cudaError_t launch_bwd_dkbar_tc(const Problem &p, const void *u, const __nv_bfloat16 *dr_hi,
                                const __nv_bfloat16 *dr_lo, int Np, float *dkbar, cudaStream_t s);
cudaError_t launch_backward_simt(const Problem &p, const void *q, const void *k, const void *v, const void *u,
                                 const void *dy, void *dq, void *dk, void *dv, void *du, void *scratch,
                                 cudaStream_t s);

}  // namespace mc
