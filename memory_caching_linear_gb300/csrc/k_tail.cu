// k_tail.cu -- the readout of the last tokens of a given segmentation: the tokens after
// the segments that are whole 128-token chunks (the short segments that end the
// logarithmic segmentation of Log-Linear++, [MC-sum §4.2]), fewer than 128 per head.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
//
// Three CUDA-core kernels, after the segment scan has written O_on and r_on of these
// tokens and every segment's fp32 state and key mean exists:
//   tail_gates_simt   one thread per tail token: the gate of every memory it reads
//                     ([MC-ja §3.1 eq. 9-10]: softmax over the cached scores <u_t, kbar_i> and
//                     r_on; SSC keeps the top-k cached scores, [MC-sum §3.4]; Residual 1, Mean
//                     1 / (n + 1))
//   tail_cached_simt  one CTA per (head, cached segment i): g_{t,i} M^(i) q_t for every tail
//                     token t after segment i, as a partial per (i, t)
//   tail_finish_simt  y_t = g_on(t) O_on[t] + the partials of t's cached segments, in segment order
// Each cached state is read once per head (not once per tail segment), and the sum is
// deterministic.
#include <cstdint>

#include "mc_internal.cuh"

namespace mc {
namespace {

constexpr int kTailTok = 128;  // tail tokens per head, at most (fewer than one chunk)
constexpr int kThreads = 256;  // partial and finishing kernels
constexpr int kTcTopk = 16;    // SSC selections per token on this path (the tensor-core limit)
constexpr int kTailHalf = 64;  // tail tokens per CTA of the partial kernel
constexpr int kGT = 32;        // tail tokens per CTA of the gate kernel

size_t pad(size_t x) { return (x + 255) & ~(size_t)255; }

// Segment of token t: the last n with seg_off[n] <= t.
__device__ __forceinline__ int segment_of(const int32_t *seg_off, int N, int t)
{
    int s = N - 1;
    while (seg_off[s] > t) --s;
    return s;
}

// G[bh][tt][i] = g_{t,i} (0 for a segment t does not read), gon[bh][tt] = the online gate.
// A CTA takes kGT tokens of one head: it stages the head's key means and the tokens' u rows
// in shared memory (16-byte loads), computes the scores with four threads per token (thread
// j of a token takes segments j, j + 4, ...), then one thread per token forms the gates.
template <typename T, int D>
__global__ void __launch_bounds__(4 * kGT) tail_gates_simt(FwdArgs a, int t_tail, float *G, float *gon)
{
    constexpr int P = D + 4;  // u rows, 16-byte aligned, staggered by 4 banks
    extern __shared__ float gsm[];
    float *Us = gsm;                       // kGT x P
    float *Kb = Us + kGT * P;              // 64 x D key means
    float *Sc = Kb + 64 * D;               // kGT x 65 scores
    float *vals_all = Sc + kGT * 65;       // SSC: kGT x kTcTopk
    int *idx_all = reinterpret_cast<int *>(vals_all + kGT * kTcTopk);
    const int bh = blockIdx.y, TT = a.L - t_tail, tt0 = blockIdx.x * kGT;
    const int tid = threadIdx.x, nt = min(kGT, TT - tt0);
    const bool gated = mode_uses_u(a.mode);
    const int nmax = segment_of(a.seg_off, a.N, t_tail + tt0 + nt - 1);  // the CTA's largest cached count
    if (gated) {
        static_assert(sizeof(T) == 2, "bf16 rows");
        const uint4 *u = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.u) + ((size_t)bh * a.L + t_tail + tt0) * D);
        for (int e = tid; e < nt * (D / 8); e += 4 * kGT) {  // 8 values per load
            const uint4 x = u[e];
            const int r = e / (D / 8), c = 8 * (e % (D / 8));
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&x);
            float *dst = Us + r * P + c;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h[j]);
                dst[2 * j] = f.x;
                dst[2 * j + 1] = f.y;
            }
        }
        const float4 *kb = reinterpret_cast<const float4 *>(a.kbar + (size_t)bh * a.N * D);
        for (int e = tid; e < nmax * (D / 4); e += 4 * kGT) reinterpret_cast<float4 *>(Kb)[e] = kb[e];
    }
    __syncthreads();
    if (gated) {
        const int r = tid >> 2, j = tid & 3;
        if (r < nt)
            for (int i = j; i < nmax; i += 4) Sc[r * 65 + i] = gate_score(Us + r * P, Kb + i * D, D);
    }
    __syncthreads();
    if (tid >= nt) return;
    const int tt = tt0 + tid, t = t_tail + tt;
    const int n = segment_of(a.seg_off, a.N, t);  // cached segments 0 .. n-1
    float *g = G + ((size_t)bh * TT + tt) * a.N;
    if (!gated) {
        const float w = a.mode == MC_MEAN ? 1.f / (float)(n + 1) : 1.f;
        for (int i = 0; i < a.N; ++i) g[i] = i < n ? w : 0.f;
        gon[(size_t)bh * TT + tt] = w;
        return;
    }
    const float ron = a.r_on[(size_t)bh * a.L + t];
    const float *sc = Sc + tid * 65;
    float m = ron, z;
    if (a.mode == MC_SSC) {
        float *vals = vals_all + tid * kTcTopk;
        int *idxs = idx_all + tid * kTcTopk;
        int count = 0;
        const int kk = min(a.topk, kTcTopk);
        if (kk > 0)
            for (int i = 0; i < n; ++i) topk_insert(vals, idxs, count, kk, sc[i], i);
        for (int c = 0; c < count; ++c) m = fmaxf(m, vals[c]);
        z = expf(ron - m);
        for (int c = 0; c < count; ++c) z += expf(vals[c] - m);
        for (int i = 0; i < a.N; ++i) g[i] = 0.f;
        for (int c = 0; c < count; ++c) g[idxs[c]] = expf(vals[c] - m) / z;
    } else {
        for (int i = 0; i < n; ++i) m = fmaxf(m, sc[i]);
        z = expf(ron - m);
        for (int i = 0; i < n; ++i) z += expf(sc[i] - m);
        for (int i = 0; i < a.N; ++i) g[i] = i < n ? expf(sc[i] - m) / z : 0.f;
    }
    gon[(size_t)bh * TT + tt] = expf(ron - m) / z;
}

// part[bh][i][tt] = g_{t,i} M^(i) q_t for the tail tokens after segment i.  Thread (tx, ty)
// holds tokens ty + 16 p and value rows tx + 16 r; the state goes through shared memory
// 32 key columns at a time.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) tail_cached_simt(FwdArgs a, int t_tail, const float *G, float *part)
{
    constexpr int P = D + 1, KC = 32, KP = KC + 1, RB = D / 16, TPT = kTailHalf / 16;
    extern __shared__ float sm[];
    float *Qs = sm;                  // kTailHalf x P: g_{t,i} q_t
    float *Ms = Qs + kTailHalf * P;  // D x KP: a column block of M^(i)
    const int i = blockIdx.x, bh = blockIdx.y, TT = a.L - t_tail;
    // the tokens of later segments read segment i; this CTA takes its half (blockIdx.z) of them
    const int tseg = max(t_tail, (int)a.seg_off[i + 1]);
    const int tfirst = tseg + (int)blockIdx.z * kTailHalf;
    if (tfirst >= a.L) return;
    const int r0 = tfirst - t_tail, cnt = min(a.L - tfirst, kTailHalf);
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    __shared__ float gs[kTailHalf];
    const float gt = tid < cnt ? G[((size_t)bh * TT + r0 + tid) * a.N + i] : 0.f;
    if (tid < kTailHalf) gs[tid] = gt;
    if (!__syncthreads_or(gt != 0.f)) return;  // no tail token reads segment i (SSC)
    static_assert(sizeof(T) == 2, "bf16 rows");
    const uint4 *q = reinterpret_cast<const uint4 *>(static_cast<const T *>(a.q) + ((size_t)bh * a.L + tfirst) * D);
    for (int e = tid; e < kTailHalf * (D / 8); e += kThreads) {  // 8 values per load
        const int r = e / (D / 8), c = 8 * (e % (D / 8));
        float *dst = Qs + r * P + c;
        if (r < cnt) {
            const uint4 x = q[e];
            const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&x);
            const float w = gs[r];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float2 f = __bfloat1622float2(h[j]);
                dst[2 * j] = w * f.x;
                dst[2 * j + 1] = w * f.y;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 8; ++j) dst[j] = 0.f;
        }
    }
    __syncthreads();
    float z[TPT][RB];
#pragma unroll
    for (int p = 0; p < TPT; ++p)
#pragma unroll
        for (int r = 0; r < RB; ++r) z[p][r] = 0.f;
    const float *Mi = a.states + ((size_t)bh * a.N + i) * D * D;
    for (int kc = 0; kc < D; kc += KC) {
        for (int e = tid; e < D * KC; e += kThreads) {
            const int vr = e / KC, c = e % KC;
            Ms[vr * KP + c] = __ldg(Mi + (size_t)vr * D + kc + c);
        }
        __syncthreads();
#pragma unroll 4
        for (int c = 0; c < KC; ++c) {
            float qv[TPT];
#pragma unroll
            for (int p = 0; p < TPT; ++p) qv[p] = Qs[(ty + 16 * p) * P + kc + c];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float mv = Ms[(tx + 16 * r) * KP + c];
#pragma unroll
                for (int p = 0; p < TPT; ++p) z[p][r] = fmaf(qv[p], mv, z[p][r]);
            }
        }
        __syncthreads();
    }
    float *out = part + (((size_t)bh * (a.N - 1) + i) * TT + r0) * D;
#pragma unroll
    for (int p = 0; p < TPT; ++p) {
        const int t = ty + 16 * p;
        if (t < cnt) {
#pragma unroll
            for (int r = 0; r < RB; ++r) out[(size_t)t * D + tx + 16 * r] = z[p][r];
        }
    }
}

// y_t = g_on O_on[t] + sum over t's cached segments i (ascending) of part[i][t]; a thread per element.
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
    tail_finish_simt(FwdArgs a, int t_tail, const float *G, const float *gon, const float *part)
{
    const int TT = a.L - t_tail;
    const size_t e = (size_t)blockIdx.x * kThreads + threadIdx.x;
    if (e >= (size_t)a.BH * TT * D) return;
    const int v = (int)(e % D);
    const size_t rem = e / D;
    const int tt = (int)(rem % TT), bh = (int)(rem / TT);
    const int t = t_tail + tt;
    const int n = segment_of(a.seg_off, a.N, t);
    const size_t tok = (size_t)bh * a.L + t;
    float acc = gon[(size_t)bh * TT + tt] * a.O_on[tok * D + v];
    const float *g = G + ((size_t)bh * TT + tt) * a.N;
    for (int i = 0; i < n; ++i)
        if (g[i] != 0.f) acc += part[(((size_t)bh * (a.N - 1) + i) * TT + tt) * D + v];
    static_cast<T *>(a.y)[tok * D + v] = from_f<T>(acc);
}

template <typename T, int D>
cudaError_t tail_impl(const Problem &p, const FwdArgs &a, int t_tail, void *scratch, cudaStream_t s)
{
    const size_t TT = p.L - t_tail, BH = p.BH;
    uint8_t *base = static_cast<uint8_t *>(scratch);
    float *G = reinterpret_cast<float *>(base);
    float *gon = reinterpret_cast<float *>(base + pad(sizeof(float) * BH * TT * p.N));
    float *part = reinterpret_cast<float *>(base + pad(sizeof(float) * BH * TT * p.N) + pad(sizeof(float) * BH * TT));
    constexpr size_t gsmem = sizeof(float) * (kGT * (D + 4) + 64 * D + kGT * 65 + kGT * kTcTopk) +
                             sizeof(int) * kGT * kTcTopk;
    auto k1 = tail_gates_simt<T, D>;
    cudaError_t e = cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gsmem);
    if (e != cudaSuccess) return e;
    k1<<<dim3((unsigned)((TT + kGT - 1) / kGT), (unsigned)BH), 4 * kGT, gsmem, s>>>(a, t_tail, G, gon);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (p.N > 1) {
        constexpr size_t smem = sizeof(float) * (kTailHalf * (D + 1) + D * 33);
        auto k2 = tail_cached_simt<T, D>;
        if ((e = cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        k2<<<dim3((unsigned)(p.N - 1), (unsigned)BH, (unsigned)(kTailTok / kTailHalf)), kThreads, smem, s>>>(a, t_tail, G,
                                                                                                          part);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
    const size_t elems = BH * TT * D;
    tail_finish_simt<T, D><<<(unsigned)((elems + kThreads - 1) / kThreads), kThreads, 0, s>>>(a, t_tail, G, gon, part);
    return cudaGetLastError();
}

}  // namespace

size_t tail_scratch_bytes(const Problem &p, int t_tail)
{
    const size_t TT = p.L - t_tail, BH = p.BH;
    return pad(sizeof(float) * BH * TT * p.N) + pad(sizeof(float) * BH * TT) +
           pad(sizeof(float) * BH * (p.N > 1 ? p.N - 1 : 0) * TT * p.d);
}

cudaError_t launch_tail_readout(const Problem &p, const FwdArgs &a, int t_tail, void *scratch, cudaStream_t s)
{
    if (!p.bf16 || p.L - t_tail <= 0 || p.L - t_tail > kTailTok || p.N > 64 ||
        (p.mode == MC_SSC && p.topk > kTcTopk))
        return cudaErrorInvalidValue;
    if (p.d == 64) return tail_impl<__nv_bfloat16, 64>(p, a, t_tail, scratch, s);
    if (p.d == 128) return tail_impl<__nv_bfloat16, 128>(p, a, t_tail, scratch, s);
    return cudaErrorInvalidValue;
}

}  // namespace mc
