// k_simt.cu -- CUDA-core (FFMA) kernels of the Memory Caching forward.
//
// These serve every shape the tensor-core path does not take: fp32 inputs
// (fp32 arithmetic end to end), d in {16, 32}, and any segment length.  All
// accumulation is fp32.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
#include <cfloat>

#include "mc_internal.cuh"

namespace mc {
namespace {

constexpr int kThreads = 256;

// ---------------------------------------------------------------------------
// seg_scan: one CTA per (bh, segment).  Walks the segment in chunks of TC
// tokens, keeping the running state S = sum_{j<chunk} v_j k_j^T (fp32) and the
// running key sum.  Per chunk (tokens c0..c0+cnt-1):
//   O_on[t] = S q_t + sum_{j in chunk, j<=t} v_j (k_j . q_t)      online read after
//                                                                the update [MC-ja §3 eq. 4b-5]
//   r_on[t] = <u_t, (ksum + sum_{j<=t} k_j)> / (t - t0 + 1)        online pool score
//                                                                [MC-ja §3.1 eq. 10]
//   S += sum_j v_j k_j^T,  ksum += sum_j k_j
// At the end S is the segment's cached state and ksum / len its key mean.
// With a piece table (FwdArgs::seg_pieces) one CTA takes one piece of piece_len
// tokens: it starts from zero, so for the second and later pieces of a segment
// O_on and r_on miss the part of the state and key sum before the piece, which
// seg_fix_simt adds after seg_prefix_simt has formed those prefixes.
// Thread layout: tx = tid % 16, ty = tid / 16; a thread owns state entries
// (ty + 16 i, tx + 16 j) and output entries (token ty + 16 p, dim tx + 16 r).
// ---------------------------------------------------------------------------
template <typename T, int D, int TC>
__global__ void __launch_bounds__(kThreads) seg_scan_simt(FwdArgs a)
{
    constexpr int P = D + 1;   // padded row stride (conflict-free column walks)
    constexpr int TP = TC + 1;
    constexpr int RB = D / 16; // state rows/cols per thread, value dims per thread
    constexpr int TPT = TC / 16;
    extern __shared__ float sm[];
    float *Qs = sm;
    float *Ks = Qs + TC * P;
    float *Vs = Ks + TC * P;
    float *Us = Vs + TC * P;
    float *Ss = Us + TC * P;  // D x P, the state before the current chunk
    float *As = Ss + D * P;   // TC x TP, masked q.k
    float *Bs = As + TC * TP; // TC x TP, masked u.k
    float *ksum = Bs + TC * TP;

    const bool split = a.seg_pieces != nullptr;
    const int unit = split ? a.npieces : a.N;
    const int bh = blockIdx.x / unit;
    const int pi = blockIdx.x % unit;  // the piece (split) or the segment
    const int seg = split ? a.piece_seg[pi] : pi;
    const int ts = seg_begin(a, seg), te = seg_end(a, seg);  // the segment
    const int pidx = split ? pi - a.seg_pieces[seg] : 0;
    const int t0 = split ? ts + pidx * a.piece_len : ts;    // this CTA's tokens [t0, t1)
    const int t1 = split ? min(t0 + a.piece_len, te) : te;
    const bool whole = !split || a.seg_pieces[seg + 1] - a.seg_pieces[seg] == 1;
    const size_t base = (size_t)bh * a.L * D;
    const T *q = static_cast<const T *>(a.q) + base;
    const T *k = static_cast<const T *>(a.k) + base;
    const T *v = static_cast<const T *>(a.v) + base;
    const T *u = a.u ? static_cast<const T *>(a.u) + base : nullptr;
    float *O_on = a.O_on + base;
    float *r_on = a.r_on + (size_t)bh * a.L;

    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    float S[RB][RB];
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int j = 0; j < RB; ++j) S[i][j] = 0.f;
    for (int e = tid; e < D * P; e += kThreads) Ss[e] = 0.f;
    for (int e = tid; e < D; e += kThreads) ksum[e] = 0.f;

    for (int c0 = t0; c0 < t1; c0 += TC) {
        const int cnt = min(TC, t1 - c0);
        __syncthreads();
        for (int e = tid; e < TC * D; e += kThreads) {
            const int r = e / D, c = e % D;
            const bool ok = r < cnt;
            const size_t g = (size_t)(c0 + r) * D + c;
            Qs[r * P + c] = ok ? to_f(q[g]) : 0.f;
            Ks[r * P + c] = ok ? to_f(k[g]) : 0.f;
            Vs[r * P + c] = ok ? to_f(v[g]) : 0.f;
            Us[r * P + c] = (ok && u) ? to_f(u[g]) : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < TC * TC; e += kThreads) {
            const int t = e / TC, j = e % TC;
            float acc = 0.f, accu = 0.f;
            if (j <= t && t < cnt) {
                for (int c = 0; c < D; ++c) {
                    acc = fmaf(Qs[t * P + c], Ks[j * P + c], acc);
                    accu = fmaf(Us[t * P + c], Ks[j * P + c], accu);
                }
            }
            As[t * TP + j] = acc;
            Bs[t * TP + j] = accu;
        }
        __syncthreads();
        {
            float o[TPT][RB];
#pragma unroll
            for (int p = 0; p < TPT; ++p)
#pragma unroll
                for (int r = 0; r < RB; ++r) o[p][r] = 0.f;
            for (int c = 0; c < D; ++c) {
                float qv[TPT];
#pragma unroll
                for (int p = 0; p < TPT; ++p) qv[p] = Qs[(ty + 16 * p) * P + c];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const float s = Ss[(tx + 16 * r) * P + c];
#pragma unroll
                    for (int p = 0; p < TPT; ++p) o[p][r] = fmaf(qv[p], s, o[p][r]);
                }
            }
            for (int j = 0; j < TC; ++j) {
                float av[TPT];
#pragma unroll
                for (int p = 0; p < TPT; ++p) av[p] = As[(ty + 16 * p) * TP + j];
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const float vv = Vs[j * P + tx + 16 * r];
#pragma unroll
                    for (int p = 0; p < TPT; ++p) o[p][r] = fmaf(av[p], vv, o[p][r]);
                }
            }
#pragma unroll
            for (int p = 0; p < TPT; ++p) {
                const int t = ty + 16 * p;
                if (t < cnt) {
#pragma unroll
                    for (int r = 0; r < RB; ++r) O_on[(size_t)(c0 + t) * D + tx + 16 * r] = o[p][r];
                }
            }
        }
        if (u != nullptr && tid < cnt) {
            const int t = tid;
            float acc = 0.f;
            for (int c = 0; c < D; ++c) acc = fmaf(Us[t * P + c], ksum[c], acc);
            for (int j = 0; j <= t; ++j) acc += Bs[t * TP + j];
            r_on[c0 + t] = acc / (float)(c0 + t - ts + 1);
        }
        __syncthreads();  // Ss and ksum are read above and rewritten below
        for (int j = 0; j < cnt; ++j) {
            float vv[RB], kk[RB];
#pragma unroll
            for (int i = 0; i < RB; ++i) vv[i] = Vs[j * P + ty + 16 * i];
#pragma unroll
            for (int i = 0; i < RB; ++i) kk[i] = Ks[j * P + tx + 16 * i];
#pragma unroll
            for (int i = 0; i < RB; ++i)
#pragma unroll
                for (int jj = 0; jj < RB; ++jj) S[i][jj] = fmaf(vv[i], kk[jj], S[i][jj]);
        }
#pragma unroll
        for (int i = 0; i < RB; ++i)
#pragma unroll
            for (int jj = 0; jj < RB; ++jj) Ss[(ty + 16 * i) * P + tx + 16 * jj] = S[i][jj];
        if (tid < D) {
            float s = ksum[tid];
            for (int j = 0; j < cnt; ++j) s += Ks[j * P + tid];
            ksum[tid] = s;
        }
    }
    __syncthreads();
    float *st = whole ? a.states + ((size_t)bh * a.N + seg) * D * D : a.piece_state + ((size_t)bh * a.npieces + pi) * D * D;
#pragma unroll
    for (int i = 0; i < RB; ++i)
#pragma unroll
        for (int jj = 0; jj < RB; ++jj) st[(size_t)(ty + 16 * i) * D + tx + 16 * jj] = S[i][jj];
    if (tid < D) {
        if (whole) a.kbar[((size_t)bh * a.N + seg) * D + tid] = ksum[tid] / (float)(t1 - t0);
        else a.piece_ksum[((size_t)bh * a.npieces + pi) * D + tid] = ksum[tid];
    }
}

// ---------------------------------------------------------------------------
// seg_prefix_simt: for every segment of more than one piece, a thread per state
// entry (and per key column) walks the pieces in order, replacing each piece's own
// sum by the sum of the pieces before it, and writes the total as the segment's
// cached state (and key mean).  Grid: (bh, segment) x ceil((D*D + D) / 256).
// ---------------------------------------------------------------------------
template <int D>
__global__ void __launch_bounds__(kThreads) seg_prefix_simt(FwdArgs a)
{
    const int bh = blockIdx.x / a.N, seg = blockIdx.x % a.N;
    const int p0 = a.seg_pieces[seg], p1 = a.seg_pieces[seg + 1];
    if (p1 - p0 < 2) return;
    const int e = blockIdx.y * kThreads + threadIdx.x;
    if (e >= D * D + D) return;
    const bool key = e >= D * D;
    float *x = key ? a.piece_ksum + ((size_t)bh * a.npieces + p0) * D + (e - D * D)
                   : a.piece_state + ((size_t)bh * a.npieces + p0) * D * D + e;
    const size_t stride = key ? D : (size_t)D * D;
    float s = 0.f;
    for (int p = p0; p < p1; ++p, x += stride) {
        const float own = *x;
        *x = s;
        s += own;
    }
    if (key) a.kbar[((size_t)bh * a.N + seg) * D + (e - D * D)] = s / (float)(seg_end(a, seg) - seg_begin(a, seg));
    else a.states[((size_t)bh * a.N + seg) * D * D + e] = s;
}

// ---------------------------------------------------------------------------
// seg_fix_simt: one CTA per (bh, piece) after the first of its segment: adds the
// state before the piece to the online reads, O_on[t] += S_pre q_t, and the keys
// before it to the online scores, r_on[t] += <u_t, ksum_pre> / (t - ts + 1).
// S_pre sits in shared memory; tokens go in tiles of 64 (the scan's thread layout).
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) seg_fix_simt(FwdArgs a)
{
    constexpr int P = D + 1;
    constexpr int RB = D / 16;
    constexpr int TF = 64;
    constexpr int TPT = TF / 16;
    extern __shared__ float sm[];
    float *Ss = sm;           // D x P
    float *Qs = Ss + D * P;   // TF x P
    float *kp = Qs + TF * P;  // D
    const int bh = blockIdx.x / a.npieces, pi = blockIdx.x % a.npieces;
    const int seg = a.piece_seg[pi];
    const int pidx = pi - a.seg_pieces[seg];
    if (pidx == 0) return;
    const int ts = seg_begin(a, seg);
    const int t0 = ts + pidx * a.piece_len, t1 = min(t0 + a.piece_len, seg_end(a, seg));
    const size_t base = (size_t)bh * a.L * D;
    const T *q = static_cast<const T *>(a.q) + base;
    const T *u = a.u ? static_cast<const T *>(a.u) + base : nullptr;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const float *sp = a.piece_state + ((size_t)bh * a.npieces + pi) * D * D;
    for (int e = tid; e < D * D; e += kThreads) Ss[(e / D) * P + e % D] = sp[e];
    for (int e = tid; e < D; e += kThreads) kp[e] = a.piece_ksum[((size_t)bh * a.npieces + pi) * D + e];
    for (int c0 = t0; c0 < t1; c0 += TF) {
        const int cnt = min(TF, t1 - c0);
        __syncthreads();
        for (int e = tid; e < TF * D; e += kThreads) {
            const int r = e / D, c = e % D;
            Qs[r * P + c] = r < cnt ? to_f(q[(size_t)(c0 + r) * D + c]) : 0.f;
        }
        __syncthreads();
        float o[TPT][RB];
#pragma unroll
        for (int p = 0; p < TPT; ++p)
#pragma unroll
            for (int r = 0; r < RB; ++r) o[p][r] = 0.f;
        for (int c = 0; c < D; ++c) {
            float qv[TPT];
#pragma unroll
            for (int p = 0; p < TPT; ++p) qv[p] = Qs[(ty + 16 * p) * P + c];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const float s = Ss[(tx + 16 * r) * P + c];
#pragma unroll
                for (int p = 0; p < TPT; ++p) o[p][r] = fmaf(qv[p], s, o[p][r]);
            }
        }
        float *O_on = a.O_on + base;
#pragma unroll
        for (int p = 0; p < TPT; ++p) {
            const int t = ty + 16 * p;
            if (t < cnt) {
#pragma unroll
                for (int r = 0; r < RB; ++r) O_on[(size_t)(c0 + t) * D + tx + 16 * r] += o[p][r];
            }
        }
        if (u != nullptr && tid < cnt) {
            const int t = tid;
            float acc = 0.f;
            for (int c = 0; c < D; ++c) acc = fmaf(to_f(u[(size_t)(c0 + t) * D + c]), kp[c], acc);
            a.r_on[(size_t)bh * a.L + c0 + t] += acc / (float)(c0 + t - ts + 1);
        }
    }
}

// Key means alone (for the stand-alone router): the same sequential fp32 sum
// over the segment's tokens as seg_scan, so the means are bit-identical.
template <typename T, int D>
__global__ void __launch_bounds__(D) kbar_simt(FwdArgs a)
{
    const int seg = blockIdx.x % a.N;
    const int bh = blockIdx.x / a.N;
    const int t0 = seg_begin(a, seg), t1 = seg_end(a, seg);
    const T *k = static_cast<const T *>(a.k) + (size_t)bh * a.L * D;
    float s = 0.f;
    for (int t = t0; t < t1; ++t) s += to_f(k[(size_t)t * D + threadIdx.x]);
    a.kbar[((size_t)bh * a.N + seg) * D + threadIdx.x] = s / (float)(t1 - t0);
}

// ---------------------------------------------------------------------------
// readout: one CTA per (bh, segment n, tile of TR tokens), heavy segments first.
//   GRM / Soup: g_t = softmax over {<u_t,kbar_i>}_{i<n} and r_on[t]   [MC-ja §3.1 eq. 9-10]
//   SSC:        the top-k cached scores plus r_on[t], softmax over those [MC-sum §3.4]
//   Residual:   g = 1                                                 [MC-ja §3.1 eq. 7]
//   Mean:       g = 1 / (n + 1), the post-training form (no router)
//   y_t = g_{t,n} O_on[t] + sum_{i<n} g_{t,i} M^(i) q_t
// Soup is computed as GRM: for a linear memory the parameter average read at q_t
// is the gated sum of the reads ([MC-sum §3.3]).
// ---------------------------------------------------------------------------
constexpr int kTR = 64;

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) readout_simt(FwdArgs a)
{
    constexpr int P = D + 1;
    constexpr int KC = D < 32 ? D : 32;
    constexpr int KP = KC + 1;
    constexpr int RB = D / 16;
    constexpr int TPT = kTR / 16;
    extern __shared__ float sm[];
    float *Qs = sm;             // kTR x P
    float *Us = Qs + kTR * P;   // kTR x P
    float *Ms = Us + kTR * P;   // D x KP, a column block of one cached state
    float *g = Ms + D * KP;     // 2 x kTR, gates of the current segment (double-buffered)
    float *m_t = g + 2 * kTR;   // softmax max
    float *z_t = m_t + kTR;     // softmax sum
    float *gon = z_t + kTR;     // online gate
    float *selv = gon + kTR;    // kTR x kMaxTopk (SSC: gate of each selected segment); this and the
                                // rest exist for SSC only (the launch sizes shared memory by mode)
    int *seli = reinterpret_cast<int *>(selv + kTR * kMaxTopk);  // kTR x kMaxTopk
    int *cur = seli + kTR * kMaxTopk;
    int *nsel = cur + kTR;

    const int tps = (a.C + kTR - 1) / kTR;
    const int per_seg = a.BH * tps;
    const int seg = a.N - 1 - (int)(blockIdx.x / per_seg);
    const int rem = blockIdx.x % per_seg;
    const int bh = rem / tps, tile = rem % tps;
    const int t0 = seg_begin(a, seg);
    const int tb = t0 + tile * kTR;
    const int te = min(tb + kTR, seg_end(a, seg));
    if (tb >= te) return;
    const int cnt = te - tb;
    const int n = seg;  // cached segments 0..n-1
    const int mode = a.mode;
    const bool gated = mode_uses_u(mode);
    const float wmean = mode == MC_MEAN ? 1.f / (float)(n + 1) : 1.f;  // Residual / Mean weight

    const size_t base = (size_t)bh * a.L * D;
    const T *q = static_cast<const T *>(a.q) + base;
    const T *u = gated ? static_cast<const T *>(a.u) + base : nullptr;
    const float *kbar = a.kbar + (size_t)bh * a.N * D;
    const float *states = a.states + (size_t)bh * a.N * D * D;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;

    for (int e = tid; e < kTR * D; e += kThreads) {
        const int r = e / D, c = e % D;
        const bool ok = r < cnt;
        const size_t gi = (size_t)(tb + r) * D + c;
        Qs[r * P + c] = ok ? to_f(q[gi]) : 0.f;
        Us[r * P + c] = (ok && gated) ? to_f(u[gi]) : 0.f;
    }
    __syncthreads();

    // Per-token gate normalisation.
    if (tid < kTR) {
        const int t = tid;
        float go = wmean;
        if (t < cnt && gated) {
            const float ron = a.r_on[(size_t)bh * a.L + tb + t];
            const float *ur = Us + t * P;
            if (mode == MC_SSC) {
                float *vals = selv + t * kMaxTopk;
                int *idxs = seli + t * kMaxTopk;
                int count = 0;
                const int kk = min(a.topk, kMaxTopk);
                if (kk > 0)
                    for (int i = 0; i < n; ++i) topk_insert(vals, idxs, count, kk, gate_score(ur, kbar + (size_t)i * D, D), i);
                float m = ron;
                for (int c = 0; c < count; ++c) m = fmaxf(m, vals[c]);
                float z = expf(ron - m);
                for (int c = 0; c < count; ++c) z += expf(vals[c] - m);
                for (int c = 0; c < count; ++c) vals[c] = expf(vals[c] - m) / z;
                go = expf(ron - m) / z;
                for (int x = 1; x < count; ++x) {  // order the selection by segment index
                    const int ix = idxs[x];
                    const float vx = vals[x];
                    int y = x - 1;
                    while (y >= 0 && idxs[y] > ix) {
                        idxs[y + 1] = idxs[y];
                        vals[y + 1] = vals[y];
                        --y;
                    }
                    idxs[y + 1] = ix;
                    vals[y + 1] = vx;
                }
                nsel[t] = count;
                cur[t] = 0;
            } else {
                float m = ron, z = 1.f;  // streaming softmax over r_on and the cached scores
                for (int i = 0; i < n; ++i) {
                    const float r = gate_score(ur, kbar + (size_t)i * D, D);
                    if (r > m) {
                        z = z * expf(m - r) + 1.f;
                        m = r;
                    } else {
                        z += expf(r - m);
                    }
                }
                m_t[t] = m;
                z_t[t] = z;
                go = expf(ron - m) / z;
            }
        } else if (mode == MC_SSC) {
            nsel[t] = 0;
            cur[t] = 0;
        }
        gon[t] = go;
    }
    __syncthreads();

    float y[TPT][RB];
#pragma unroll
    for (int p = 0; p < TPT; ++p)
#pragma unroll
        for (int r = 0; r < RB; ++r) y[p][r] = 0.f;

    for (int i = 0; i < n; ++i) {
        float *gb = g + (i & 1) * kTR;
        float gi = 0.f;
        if (tid < kTR) {
            const int t = tid;
            if (t < cnt) {
                if (!gated) {
                    gi = wmean;
                } else if (mode == MC_SSC) {
                    const int c = cur[t];
                    if (c < nsel[t] && seli[t * kMaxTopk + c] == i) {
                        gi = selv[t * kMaxTopk + c];
                        cur[t] = c + 1;
                    }
                } else {
                    const float r = gate_score(Us + t * P, kbar + (size_t)i * D, D);
                    gi = expf(r - m_t[t]) / z_t[t];
                }
            }
            gb[t] = gi;
        }
        if (!__syncthreads_or(gi != 0.f)) continue;  // no token of the tile reads segment i
        float z[TPT][RB];
#pragma unroll
        for (int p = 0; p < TPT; ++p)
#pragma unroll
            for (int r = 0; r < RB; ++r) z[p][r] = 0.f;
        const float *Mi = states + (size_t)i * D * D;
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
#pragma unroll
        for (int p = 0; p < TPT; ++p) {
            const float gp = gb[ty + 16 * p];
#pragma unroll
            for (int r = 0; r < RB; ++r) y[p][r] = fmaf(gp, z[p][r], y[p][r]);
        }
    }

    T *yo = static_cast<T *>(a.y) + base;
    const float *O_on = a.O_on + base;
#pragma unroll
    for (int p = 0; p < TPT; ++p) {
        const int t = ty + 16 * p;
        if (t < cnt) {
            const float go = gon[t];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const size_t gi = (size_t)(tb + t) * D + tx + 16 * r;
                yo[gi] = from_f<T>(fmaf(go, O_on[gi], y[p][r]));
            }
        }
    }
}

// Stand-alone SSC router: the readout's selection, written out in rank order.
template <typename T, int D>
__global__ void __launch_bounds__(kTR) ssc_select_simt(FwdArgs a)
{
    constexpr int P = D + 1;
    extern __shared__ float sm[];
    float *Us = sm;                      // kTR x P
    float *vals_all = Us + kTR * P;      // kTR x kMaxTopk
    int *idx_all = reinterpret_cast<int *>(vals_all + kTR * kMaxTopk);
    const int tps = (a.C + kTR - 1) / kTR;
    const int per_bh = a.N * tps;
    const int bh = blockIdx.x / per_bh;
    const int rem = blockIdx.x % per_bh;
    const int seg = rem / tps, tile = rem % tps;
    const int t0 = seg_begin(a, seg);
    const int tb = t0 + tile * kTR;
    const int te = min(tb + kTR, seg_end(a, seg));
    if (tb >= te) return;
    const int cnt = te - tb;
    const size_t base = (size_t)bh * a.L * D;
    const T *u = static_cast<const T *>(a.u) + base;
    for (int e = threadIdx.x; e < kTR * D; e += kTR) {
        const int r = e / D, c = e % D;
        Us[r * P + c] = r < cnt ? to_f(u[(size_t)(tb + r) * D + c]) : 0.f;
    }
    __syncthreads();
    const int t = threadIdx.x;
    if (t >= cnt) return;
    float *vals = vals_all + t * kMaxTopk;
    int *idxs = idx_all + t * kMaxTopk;
    int count = 0;
    const float *kbar = a.kbar + (size_t)bh * a.N * D;
    for (int i = 0; i < seg; ++i) topk_insert(vals, idxs, count, a.topk, gate_score(Us + t * P, kbar + (size_t)i * D, D), i);
    int32_t *out = a.sel_out + ((size_t)bh * a.L + tb + t) * a.topk;
    for (int c = 0; c < a.topk; ++c) out[c] = c < count ? idxs[c] : -1;
}

template <typename F>
cudaError_t set_smem(F *kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

template <typename T, int D>
cudaError_t seg_scan_impl(const Problem &p, const FwdArgs &a, cudaStream_t s)
{
    constexpr int TC = D >= 128 ? 16 : 64;  // d = 128: two CTAs per SM (102 KB of shared memory each)
    constexpr int P = D + 1, TP = TC + 1;
    const size_t smem = sizeof(float) * (4 * TC * P + D * P + 2 * TC * TP + D);
    auto kern = seg_scan_simt<T, D, TC>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    if (!a.seg_pieces) {
        kern<<<(unsigned)((long long)p.BH * p.N), kThreads, smem, s>>>(a);
        return cudaGetLastError();
    }
    // long segments in pieces: every piece at once, then the prefixes over each segment's pieces
    kern<<<(unsigned)((long long)p.BH * a.npieces), kThreads, smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (!a.piece_state) return cudaSuccess;  // one piece per segment: nothing to carry between pieces
    seg_prefix_simt<D><<<dim3((unsigned)((long long)p.BH * p.N), (unsigned)((D * D + D + kThreads - 1) / kThreads)),
                         kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    constexpr size_t fsmem = sizeof(float) * (D * P + 64 * P + D);
    auto fix = seg_fix_simt<T, D>;
    if ((e = set_smem(fix, fsmem)) != cudaSuccess) return e;
    fix<<<(unsigned)((long long)p.BH * a.npieces), kThreads, fsmem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t readout_impl(const Problem &p, const FwdArgs &a, cudaStream_t s)
{
    constexpr int P = D + 1;
    constexpr int KC = D < 32 ? D : 32;
    // the SSC tables come last and only SSC gets them (two CTAs per SM at d = 128 otherwise)
    const bool ssc = p.mode == MC_SSC;
    const size_t smem = sizeof(float) * (2 * kTR * P + D * (KC + 1) + 5 * kTR) +
                        (ssc ? sizeof(float) * kTR * kMaxTopk + sizeof(int) * (kTR * kMaxTopk + 2 * kTR) : 0);
    auto kern = readout_simt<T, D>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const long long tps = (p.C + kTR - 1) / kTR;
    const long long blocks = (long long)p.BH * p.N * tps;
    kern<<<(unsigned)blocks, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t kbar_impl(const Problem &p, const FwdArgs &a, cudaStream_t s)
{
    kbar_simt<T, D><<<(unsigned)((long long)p.BH * p.N), D, 0, s>>>(a);
    return cudaGetLastError();
}

template <typename T, int D>
cudaError_t select_impl(const Problem &p, const FwdArgs &a, cudaStream_t s)
{
    constexpr int P = D + 1;
    const size_t smem = sizeof(float) * (kTR * P + kTR * kMaxTopk) + sizeof(int) * kTR * kMaxTopk;
    auto kern = ssc_select_simt<T, D>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const long long tps = (p.C + kTR - 1) / kTR;
    kern<<<(unsigned)((long long)p.BH * p.N * tps), kTR, smem, s>>>(a);
    return cudaGetLastError();
}

#define MC_DISPATCH(FN, p, a, s)                                                  \
    do {                                                                          \
        switch ((p).d) {                                                          \
        case 16: return (p).bf16 ? FN<__nv_bfloat16, 16>(p, a, s) : FN<float, 16>(p, a, s);   \
        case 32: return (p).bf16 ? FN<__nv_bfloat16, 32>(p, a, s) : FN<float, 32>(p, a, s);   \
        case 64: return (p).bf16 ? FN<__nv_bfloat16, 64>(p, a, s) : FN<float, 64>(p, a, s);   \
        case 128: return (p).bf16 ? FN<__nv_bfloat16, 128>(p, a, s) : FN<float, 128>(p, a, s); \
        default: return cudaErrorInvalidValue;                                    \
        }                                                                         \
    } while (0)

}  // namespace

cudaError_t launch_seg_scan_simt(const Problem &p, const FwdArgs &a, cudaStream_t s) { MC_DISPATCH(seg_scan_impl, p, a, s); }
cudaError_t launch_readout_simt(const Problem &p, const FwdArgs &a, cudaStream_t s) { MC_DISPATCH(readout_impl, p, a, s); }
cudaError_t launch_kbar_simt(const Problem &p, const FwdArgs &a, cudaStream_t s) { MC_DISPATCH(kbar_impl, p, a, s); }
cudaError_t launch_ssc_select_simt(const Problem &p, const FwdArgs &a, cudaStream_t s) { MC_DISPATCH(select_impl, p, a, s); }

}  // namespace mc
