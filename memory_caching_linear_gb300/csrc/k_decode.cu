// k_decode.cu -- one recurrent decoding step of Memory Caching over a linear
// memory: the new token updates the online memory of its segment, reads it and
// the cached segment memories through the gates, and, at a segment's last token,
// the online memory is appended to the cache.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
//
// For token t of segment s (segments of constant length C, t0 = sC):
//   online:  M_t^(s) = M_{t-1}^(s) + v_t k_t^T (empty at t0)        [MC-ja §3, eq. 4b]
//   pool:    p_t = (sum_{j=t0..t} k_j) / (t - t0 + 1)              [MC-ja §3.1, eq. 10]
//   scores:  r_i = <u_t, kbar_i> (i < s), r_s = <u_t, p_t>         [MC-ja §3.1, eq. 10]
//   gates:   GRM / Soup softmax over r_0..r_s; SSC the topk largest cached scores
//            (ties to the lower index) and the online one; Residual all 1; Mean
//            all 1 / (s + 1) (memory caching added after training, no router)
//                                                                   [MC-ja §3.1 eq. 7-10; MC-sum §3.3-3.4]
//   read:    y_t = g_s M_t^(s) q_t + sum_{i<s} g_i M^(i) q_t        [MC-ja §3.1, eq. 9]
//   at t = t0 + C - 1: M^(s) = M_t^(s), kbar_s = p_t               [MC-ja §3, after eq. 4b]
// Run from t = 0 with empty caches, the steps reproduce the forward pass token by
// token.
//
// Two kernels: decode_gates (one CTA per head: key sum, scores, gates, and the
// list of cached segments with a non-zero gate) and decode_read (one CTA per head
// and block of 8 value rows: online update, read, cache append).  The read is
// bound by the cached fp32 memories, s d^2 floats per head; splitting the rows
// spreads that over BH * d / 8 CTAs, and a warp reads one 512-byte row of four
// states per step.
//
// Per-head gate record (kDecGateWords words): [0, 64) gates of the listed cached
// segments, [64, 128) their indices, 128: the online gate, 129: the list length.
#include <cstdint>

#include "mc_internal.cuh"

namespace mc {
namespace {

constexpr int kDecThreads = 256;  // 8 warps
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMaxD = 128;

template <typename T>
__global__ void __launch_bounds__(kDecThreads) decode_gates(DecodeArgs a)
{
    const int bh = blockIdx.x;
    const int d = a.d, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = a.t / a.C, t0 = s * a.C;
    const bool seg_start = a.t == t0, seg_end = a.t == t0 + a.C - 1;
    __shared__ float us[kDecMaxD], psum[kDecMaxD];
    __shared__ float sc[kDecMaxN];
    __shared__ int chosen[kDecMaxN];

    const T *k = static_cast<const T *>(a.k) + (size_t)bh * d;
    const T *u = a.u ? static_cast<const T *>(a.u) + (size_t)bh * d : nullptr;
    float *ksum = a.ksum + (size_t)bh * d;
    for (int i = tid; i < d; i += kDecThreads) {
        us[i] = u ? to_f(u[i]) : 0.f;
        const float p = (seg_start ? 0.f : ksum[i]) + to_f(k[i]);  // keys of the segment so far
        psum[i] = p;
        ksum[i] = p;
        if (seg_end) a.kbar[((size_t)bh * a.nmax + s) * d + i] = p / (float)a.C;
    }
    __syncthreads();
    float *gout = a.gates + (size_t)bh * kDecGateWords;
    int *gidx = reinterpret_cast<int *>(gout + 64);
    if (a.mode == MC_RESIDUAL || a.mode == MC_MEAN) {
        const float w = a.mode == MC_MEAN ? 1.f / (float)(s + 1) : 1.f;
        for (int i = tid; i < s; i += kDecThreads) {
            gout[i] = w;
            gidx[i] = i;
        }
        if (tid == 0) {
            gout[128] = w;
            gidx[65] = s;
        }
        return;
    }
    // scores: one warp per segment, the online one last
    const float *kbar = a.kbar + (size_t)bh * a.nmax * d;
    for (int i = warp; i <= s; i += kDecWarps) {
        float part = 0.f;
        if (i < s) {
            for (int c = lane; c < d; c += 32) part = fmaf(us[c], kbar[(size_t)i * d + c], part);
        } else {
            for (int c = lane; c < d; c += 32) part = fmaf(us[c], psum[c], part);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        if (lane == 0) sc[i] = i < s ? part : part / (float)(a.t - t0 + 1);
    }
    __syncthreads();
    if (tid == 0) {
        for (int i = 0; i <= s; ++i) chosen[i] = 1;
        if (a.mode == MC_SSC && a.topk < s) {  // keep the topk largest cached scores
            for (int i = 0; i < s; ++i) chosen[i] = 0;
            for (int r = 0; r < a.topk; ++r) {
                int best = -1;
                for (int i = 0; i < s; ++i)
                    if (!chosen[i] && (best < 0 || sc[i] > sc[best])) best = i;  // ties: lower index
                chosen[best] = 1;
            }
        }
        float m = sc[s];
        for (int i = 0; i < s; ++i)
            if (chosen[i]) m = fmaxf(m, sc[i]);
        float z = 0.f;
        for (int i = 0; i <= s; ++i) {
            sc[i] = chosen[i] ? expf(sc[i] - m) : 0.f;
            z += sc[i];
        }
        const float inv = 1.f / z;
        int n = 0;
        for (int i = 0; i < s; ++i)
            if (chosen[i]) {
                gout[n] = sc[i] * inv;
                gidx[n] = i;
                ++n;
            }
        gout[128] = sc[s] * inv;
        gidx[65] = n;
    }
}

template <typename T>
__global__ void __launch_bounds__(kDecThreads) decode_read(DecodeArgs a)
{
    const int d = a.d, rblocks = d / kDecWarps;
    const int bh = blockIdx.x / rblocks, rb = blockIdx.x % rblocks;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int s = a.t / a.C, t0 = s * a.C;
    const bool seg_start = a.t == t0, seg_end = a.t == t0 + a.C - 1;
    __shared__ __align__(16) float qs[kDecMaxD];
    __shared__ __align__(16) float ks[kDecMaxD];
    __shared__ float gv[64];
    __shared__ int gi[64];
    __shared__ float g_on;
    __shared__ int n_list;
    const T *q = static_cast<const T *>(a.q) + (size_t)bh * d, *k = static_cast<const T *>(a.k) + (size_t)bh * d;
    for (int i = tid; i < d; i += kDecThreads) {
        qs[i] = to_f(q[i]);
        ks[i] = to_f(k[i]);
    }
    const float *grec = a.gates + (size_t)bh * kDecGateWords;
    const int n = reinterpret_cast<const int *>(grec + 64)[65];
    for (int i = tid; i < n; i += kDecThreads) {
        gv[i] = grec[i];
        gi[i] = reinterpret_cast<const int *>(grec + 64)[i];
    }
    if (tid == 0) {
        g_on = grec[128];
        n_list = n;
    }
    __syncthreads();
    // one warp per value row r
    const int r = rb * kDecWarps + warp;
    const float vr = to_f(static_cast<const T *>(a.v)[(size_t)bh * d + r]);
    float *online = a.online + ((size_t)bh * d + r) * d;
    float *append = seg_end ? a.states + (((size_t)bh * a.nmax + s) * d + r) * d : nullptr;
    const float *st = a.states + ((size_t)bh * a.nmax * d + r) * d;  // row r of cached state 0
    const size_t sstride = (size_t)d * d;
    float acc = 0.f;
    if (d == kDecMaxD) {  // a lane holds 4 consecutive columns; a warp reads a 512-byte row
        const float4 qv = reinterpret_cast<const float4 *>(qs)[lane];
        const float4 kv = reinterpret_cast<const float4 *>(ks)[lane];
        float4 o = seg_start ? make_float4(0.f, 0.f, 0.f, 0.f) : reinterpret_cast<const float4 *>(online)[lane];
        o.x = fmaf(vr, kv.x, o.x);
        o.y = fmaf(vr, kv.y, o.y);
        o.z = fmaf(vr, kv.z, o.z);
        o.w = fmaf(vr, kv.w, o.w);
        reinterpret_cast<float4 *>(online)[lane] = o;
        if (append) reinterpret_cast<float4 *>(append)[lane] = o;
        auto dot4 = [&](const float4 m) { return fmaf(m.x, qv.x, fmaf(m.y, qv.y, fmaf(m.z, qv.z, m.w * qv.w))); };
        acc = g_on * dot4(o);
        int j = 0;
        for (; j + 4 <= n_list; j += 4) {  // four rows in flight per lane
            const float4 m0 = reinterpret_cast<const float4 *>(st + gi[j] * sstride)[lane];
            const float4 m1 = reinterpret_cast<const float4 *>(st + gi[j + 1] * sstride)[lane];
            const float4 m2 = reinterpret_cast<const float4 *>(st + gi[j + 2] * sstride)[lane];
            const float4 m3 = reinterpret_cast<const float4 *>(st + gi[j + 3] * sstride)[lane];
            acc = fmaf(gv[j], dot4(m0), acc);
            acc = fmaf(gv[j + 1], dot4(m1), acc);
            acc = fmaf(gv[j + 2], dot4(m2), acc);
            acc = fmaf(gv[j + 3], dot4(m3), acc);
        }
        for (; j < n_list; ++j) acc = fmaf(gv[j], dot4(reinterpret_cast<const float4 *>(st + gi[j] * sstride)[lane]), acc);
    } else {
        float on = 0.f;
        for (int c = lane; c < d; c += 32) {
            const float o = (seg_start ? 0.f : online[c]) + vr * ks[c];
            online[c] = o;
            if (append) append[c] = o;
            on = fmaf(o, qs[c], on);
        }
        acc = g_on * on;
        for (int j = 0; j < n_list; ++j) {
            float part = 0.f;
            for (int c = lane; c < d; c += 32) part = fmaf(st[gi[j] * sstride + c], qs[c], part);
            acc = fmaf(gv[j], part, acc);
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) static_cast<T *>(a.y)[(size_t)bh * d + r] = from_f<T>(acc);
}

}  // namespace

cudaError_t launch_decode_step(const DecodeArgs &a, cudaStream_t s)
{
    const unsigned rgrid = (unsigned)(a.BH * (a.d / kDecWarps));
    if (a.bf16) {
        decode_gates<__nv_bfloat16><<<(unsigned)a.BH, kDecThreads, 0, s>>>(a);
        decode_read<__nv_bfloat16><<<rgrid, kDecThreads, 0, s>>>(a);
    } else {
        decode_gates<float><<<(unsigned)a.BH, kDecThreads, 0, s>>>(a);
        decode_read<float><<<rgrid, kDecThreads, 0, s>>>(a);
    }
    return cudaGetLastError();
}

}  // namespace mc
