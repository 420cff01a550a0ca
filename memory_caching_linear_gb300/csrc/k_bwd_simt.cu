// k_bwd_simt.cu -- CUDA-core (FFMA) kernels of the Memory Caching backward pass
// over a linear memory: the gradients dq, dk, dv, du of <y, dy>.
//
// Pages cited:
//   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (news.neo-ai.one/ja/article/2519)
//   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
//            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
//
// The forward ([MC-ja §3 eq. 4b-5, §3.1 eq. 7-10; MC-sum §3.3-3.4]) reads, for
// token t of segment n, the memories i <= n (cached M^(i) for i < n, the online
// M_t for i = n) with gates g_{t,i}:  y_t = sum_i g_{t,i} M_i q_t.  Its gradient:
//   dg_{t,i}  = dy_t . M_i q_t,   delta_t = sum_i g_{t,i} dg_{t,i}
//   dr_{t,i}  = g_{t,i} (dg_{t,i} - delta_t)           (softmax gates; the SSC
//               selection is piecewise constant and passes nothing)
//   du_t      = sum_{i<n} dr_{t,i} kbar_i + dr_{t,n} p_t  (scores <u_t, kbar_i>, <u_t, p_t>)
//   dkbar_i   = sum_t dr_{t,i} u_t,  p_t = mean of the segment's keys up to t
//   dq_t      = sum_i g_{t,i} M_i^T dy_t
//   G_i       = sum_{t : n(t) > i} g_{t,i} dy_t q_t^T      (gradient of the cached M^(i))
//   dv_j      = E_j k_j,  dk_j = E_j^T v_j + dkbar_n / |n| + sum_{t >= j in n} dr_{t,n} u_t / cnt_t
//   with E_j  = G_n + sum_{t >= j in segment n} g_{t,n} dy_t q_t^T for token j of segment n.
// Residual (g = 1) and Mean (g = 1 / (n + 1)) have constant gates and du = 0.
//
// After the forward's segment scan has been re-run twice (once for the cached
// states, key means, online scores and O_on = M_t q_t; once on (dy, v, k) for
// X_on = M_t^T dy_t), on the FFMA path:
//   bwd_gates_simt  per (b,h, segment, 64-token tile): gates, dg against every cached
//                   state, dq, du, dkbar (atomics) and the per-token softmax data;
//   bwd_G_simt      per (b,h, cached segment i): G_i over every later token;
//   bwd_scan_simt   per (b,h, segment): walks the segment backwards with E, writes dk, dv.
// On the shapes of the tensor-core path the gates, the memories' reads (dg and all of
// dq), G and dk / dv run on the tensor cores (k_bwd_tc.cu, and the gates mode of the
// router kernel in k_tc.cu), and the gate work on whole shared-memory tables:
// bwd_route_simt (delta, dr, du, the online gates and pooled-key weights for dk / dv)
// and bwd_dkbar_simt (the key-mean gradient from dr).
#include <type_traits>

#include "mc_internal.cuh"

namespace mc {
namespace {

constexpr int kThreads = 256;
constexpr int kTB = 64;  // tokens per gate tile
constexpr int kTab = 64; // cached segments whose scores a gate tile keeps in shared memory
constexpr int kTG = 32;  // tokens per step of the G accumulation

template <typename F>
cudaError_t set_smem(F *kern, size_t bytes)
{
    return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
}

__device__ __forceinline__ bool gated_mode(int mode) { return mode == MC_GRM || mode == MC_SOUP || mode == MC_SSC; }

// Constant gate of the Residual / Mean aggregations for a token of segment n.
__device__ __forceinline__ float const_gate(int mode, int n) { return mode == MC_MEAN ? 1.f / (float)(n + 1) : 1.f; }

// ---------------------------------------------------------------------------
// bwd_gates_simt: one CTA per (bh, segment n, tile of kTB tokens), heavy segments
// first.  Thread layout as the forward readout: tx = tid % 16, ty = tid / 16; a
// thread owns tokens ty + 16 p and dimensions tx + 16 r.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_gates_simt(BwdArgs a)
{
    constexpr int P = D + 1;
    constexpr int KC = D < 32 ? D : 32;
    constexpr int KP = KC + 1;
    constexpr int RB = D / 16;
    constexpr int RK = KC / 16;
    constexpr int TPT = kTB / 16;
    extern __shared__ float sm[];
    float *Qs = sm;              // kTB x P
    float *Ys = Qs + kTB * P;    // kTB x P  dy
    float *Us = Ys + kTB * P;    // kTB x P
    float *Ks = Us + kTB * P;    // kTB x P
    float *Ms = Ks + kTB * P;    // D x KP, a key block of one cached state
    float *kb = Ms + D * KP;     // D: kbar_i
    float *kpre = kb + D;        // D: keys of the segment before the tile
    float *gb = kpre + D;        // kTB: gate of the current memory
    float *cb = gb + kTB;        // kTB: gate x dgate of the current memory
    float *m_t = cb + kTB;       // kTB: softmax max
    float *z_t = m_t + kTB;      // kTB: softmax sum
    float *gon = z_t + kTB;      // kTB: online gate
    float *dl = gon + kTB;       // kTB: delta = sum_i g dg
    float *selv = dl + kTB;      // kTB x kMaxTopk (SSC)
    int *seli = reinterpret_cast<int *>(selv + kTB * kMaxTopk);
    int *cur = seli + kTB * kMaxTopk;
    int *nsel = cur + kTB;
    float *sct = reinterpret_cast<float *>(nsel + kTB);  // kTB x kTab: <u_t, kbar_i>

    const int tps = (a.C + kTB - 1) / kTB;
    const int per_seg = a.BH * tps;
    const int n = a.N - 1 - (int)(blockIdx.x / per_seg);
    const int rem = blockIdx.x % per_seg;
    const int bh = rem / tps, tile = rem % tps;
    const int t0 = n * a.C;
    const int tb = t0 + tile * kTB;
    const int te = min(min(tb + kTB, t0 + a.C), a.L);
    if (tb >= te) return;
    const int cnt = te - tb;
    const int mode = a.mode;
    const bool gated = gated_mode(mode);
    const size_t base = (size_t)bh * a.L * D;
    const T *q = static_cast<const T *>(a.q) + base, *k = static_cast<const T *>(a.k) + base;
    const T *dy = static_cast<const T *>(a.dy) + base;
    const T *u = gated ? static_cast<const T *>(a.u) + base : nullptr;
    const float *kbar = a.kbar + (size_t)bh * a.N * D;
    const float *states = a.states + (size_t)bh * a.N * D * D;
    float *dkbar = a.dkbar + (size_t)bh * a.N * D;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;

    for (int e = tid; e < kTB * D; e += kThreads) {
        const int r = e / D, c = e % D;
        const bool ok = r < cnt;
        const size_t gi = (size_t)(tb + r) * D + c;
        Qs[r * P + c] = ok ? to_f(q[gi]) : 0.f;
        Ys[r * P + c] = ok ? to_f(dy[gi]) : 0.f;
        Us[r * P + c] = (ok && gated) ? to_f(u[gi]) : 0.f;
        Ks[r * P + c] = (ok && gated) ? to_f(k[gi]) : 0.f;
    }
    // keys of this segment before the tile (the online memory's pooled key, for du): every
    // thread sums a column over a strided share of the tokens, four loads in flight
    const bool need_kpre = gated;
    if (need_kpre && tid < D) kpre[tid] = 0.f;
    __syncthreads();
    if (need_kpre) {
        constexpr int parts = kThreads / D;
        const int col = tid % D, part = tid / D;
        float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
        int j = t0 + part;
        for (; j + 3 * parts < tb; j += 4 * parts) {
            s0 += to_f(k[(size_t)j * D + col]);
            s1 += to_f(k[(size_t)(j + parts) * D + col]);
            s2 += to_f(k[(size_t)(j + 2 * parts) * D + col]);
            s3 += to_f(k[(size_t)(j + 3 * parts) * D + col]);
        }
        for (; j < tb; j += parts) s0 += to_f(k[(size_t)j * D + col]);
        atomicAdd(&kpre[col], (s0 + s1) + (s2 + s3));
    }
    __syncthreads();
    // the router scores of the tile against every cached segment, all threads at once (the same
    // arithmetic as gate_score everywhere else, so every pass ranks identically)
    const bool use_tab = gated && n <= kTab;
    if (use_tab) {
        for (int e = tid; e < kTB * n; e += kThreads) {  // a warp: 32 tokens, one segment (its kbar row broadcast)
            const int i = e / kTB, t = e % kTB;
            sct[t * kTab + i] = t < cnt ? gate_score(Us + t * P, kbar + (size_t)i * D, D) : 0.f;
        }
        __syncthreads();
    }
    auto score = [&](int t, int i) -> float {
        return use_tab ? sct[t * kTab + i] : gate_score(Us + t * P, kbar + (size_t)i * D, D);
    };

    // Gates, as in the forward readout.
    if (tid < kTB) {
        const int t = tid;
        float go = const_gate(mode, n), m = 0.f, z = 1.f;
        if (t < cnt && gated) {
            const float ron = a.r_on[(size_t)bh * a.L + tb + t];
            if (mode == MC_SSC) {
                float *vals = selv + t * kMaxTopk;
                int *idxs = seli + t * kMaxTopk;
                int count = 0;
                const int kk = min(a.topk, kMaxTopk);
                if (kk > 0)
                    for (int i = 0; i < n; ++i) topk_insert(vals, idxs, count, kk, score(t, i), i);
                m = ron;
                for (int c = 0; c < count; ++c) m = fmaxf(m, vals[c]);
                z = expf(ron - m);
                for (int c = 0; c < count; ++c) z += expf(vals[c] - m);
                for (int c = 0; c < count; ++c) vals[c] = expf(vals[c] - m) / z;
                go = expf(ron - m) / z;
                for (int x = 1; x < count; ++x) {  // segment order
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
                int32_t *so = a.sel_idx + ((size_t)bh * a.L + tb + t) * a.topk;
                float *sg = a.sel_g + ((size_t)bh * a.L + tb + t) * a.topk;
                for (int c = 0; c < a.topk; ++c) {
                    so[c] = c < count ? idxs[c] : -1;
                    sg[c] = c < count ? vals[c] : 0.f;
                }
            } else {
                m = ron;  // streaming softmax over r_on and the cached scores
                z = 1.f;
                for (int i = 0; i < n; ++i) {
                    const float r = score(t, i);
                    if (r > m) {
                        z = z * expf(m - r) + 1.f;
                        m = r;
                    } else {
                        z += expf(r - m);
                    }
                }
                go = expf(ron - m) / z;
            }
        } else if (mode == MC_SSC) {
            nsel[t] = 0;
        }
        if (mode == MC_SSC) cur[t] = 0;
        m_t[t] = m;
        z_t[t] = z;
        gon[t] = t < cnt ? go : 0.f;
        dl[t] = 0.f;
    }
    __syncthreads();

    // gate of cached memory i for token t (tid < kTB); advances the SSC cursor
    auto gate_of = [&](int t, int i) -> float {
        if (t >= cnt) return 0.f;
        if (!gated) return const_gate(mode, n);
        if (mode == MC_SSC) {
            const int c = cur[t];
            if (c < nsel[t] && seli[t * kMaxTopk + c] == i) {
                cur[t] = c + 1;
                return selv[t * kMaxTopk + c];
            }
            return 0.f;
        }
        return expf(score(t, i) - m_t[t]) / z_t[t];
    };

    float dq[TPT][RB], dua[TPT][RB], gk[TPT][RB];
#pragma unroll
    for (int p = 0; p < TPT; ++p)
#pragma unroll
        for (int r = 0; r < RB; ++r) dq[p][r] = dua[p][r] = gk[p][r] = 0.f;

    for (int i = 0; i < n; ++i) {
        float gi = 0.f;
        if (tid < kTB) {
            gi = gate_of(tid, i);
            gb[tid] = gi;
        }
        if (gated && tid < D) kb[tid] = kbar[(size_t)i * D + tid];
        if (!__syncthreads_or(gi != 0.f)) continue;  // no token of the tile reads segment i
        float dgv[TPT];  // dg_{t,i} = dy_t . (M^(i) q_t), complete in every lane of the token's group
        {
            const float *Mi = states + (size_t)i * D * D;
            float z1[TPT][RB];  // (M^(i) q_t) at value dims tx + 16 r
#pragma unroll
            for (int p = 0; p < TPT; ++p)
#pragma unroll
                for (int r = 0; r < RB; ++r) z1[p][r] = 0.f;
#pragma unroll
            for (int kc = 0; kc < D; kc += KC) {  // unrolled: dq is indexed by the block
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
                        for (int p = 0; p < TPT; ++p) z1[p][r] = fmaf(qv[p], mv, z1[p][r]);
                    }
                }
                // (M^(i)^T dy_t) at the block's key dims kc + tx + 16 r2
                float z2[TPT][RK];
#pragma unroll
                for (int p = 0; p < TPT; ++p)
#pragma unroll
                    for (int r2 = 0; r2 < RK; ++r2) z2[p][r2] = 0.f;
#pragma unroll 4
                for (int vr = 0; vr < D; ++vr) {
                    float yv[TPT];
#pragma unroll
                    for (int p = 0; p < TPT; ++p) yv[p] = Ys[(ty + 16 * p) * P + vr];
#pragma unroll
                    for (int r2 = 0; r2 < RK; ++r2) {
                        const float mv = Ms[vr * KP + tx + 16 * r2];
#pragma unroll
                        for (int p = 0; p < TPT; ++p) z2[p][r2] = fmaf(yv[p], mv, z2[p][r2]);
                    }
                }
#pragma unroll
                for (int p = 0; p < TPT; ++p) {
                    const float g = gb[ty + 16 * p];
#pragma unroll
                    for (int r2 = 0; r2 < RK; ++r2) dq[p][kc / 16 + r2] = fmaf(g, z2[p][r2], dq[p][kc / 16 + r2]);
                }
                __syncthreads();
            }
            // partial over this thread's dims, then the 16 lanes of the token
#pragma unroll
            for (int p = 0; p < TPT; ++p) {
                const int t = ty + 16 * p;
                float part = 0.f;
#pragma unroll
                for (int r = 0; r < RB; ++r) part = fmaf(Ys[t * P + tx + 16 * r], z1[p][r], part);
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                dgv[p] = part;
            }
        }
#pragma unroll
        for (int p = 0; p < TPT; ++p) {
            const int t = ty + 16 * p;
            const float c = gb[t] * dgv[p];  // g dg
            if (gated) {
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    dua[p][r] = fmaf(c, kb[tx + 16 * r], dua[p][r]);
                    gk[p][r] = fmaf(gb[t], kb[tx + 16 * r], gk[p][r]);
                }
            }
            if (tx == 0) cb[t] = c;
        }
        __syncthreads();
        if (tid < kTB) dl[tid] += cb[tid];
        if (gated && tid < D) {  // dkbar_i += sum_t g dg u_t (the -g delta u_t part follows once delta is known)
            float s = 0.f;
            for (int t = 0; t < cnt; ++t) s = fmaf(cb[t], Us[t * P + tid], s);
            if (s != 0.f) atomicAdd(dkbar + (size_t)i * D + tid, s);
        }
        __syncthreads();
    }

    // the online memory: dg_on = dy_t . O_on[t], dq += g_on M_t^T dy_t
    const float *Oon = a.O_on + base, *Xon = a.X_on + base;
    float dgon[TPT];
#pragma unroll
    for (int p = 0; p < TPT; ++p) {
        const int t = ty + 16 * p;
        float part = 0.f;
        if (t < cnt) {
            const float g = gon[t];
#pragma unroll
            for (int r = 0; r < RB; ++r) {
                const size_t gi = (size_t)(tb + t) * D + tx + 16 * r;
                part = fmaf(Ys[t * P + tx + 16 * r], Oon[gi], part);
                dq[p][r] = fmaf(g, Xon[gi], dq[p][r]);
            }
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
        dgon[p] = part;
    }
    // delta_t = sum over the cached memories (dl) + the online one; every lane of a token's group computes it
    float delta[TPT];
#pragma unroll
    for (int p = 0; p < TPT; ++p) {
        const int t = ty + 16 * p;
        delta[p] = dl[t] + gon[t] * dgon[p];
    }

    T *dqo = static_cast<T *>(a.dq) + base;
    T *duo = gated ? static_cast<T *>(a.du) + base : nullptr;
    float *tok = a.tok + ((size_t)bh * a.L + tb) * kBwdTokWords;
#pragma unroll
    for (int p = 0; p < TPT; ++p) {
        const int t = ty + 16 * p;
        if (t >= cnt) continue;
        const float dron = gon[t] * (dgon[p] - delta[p]);  // dr of the online memory
        const float inv_cnt = 1.f / (float)(tb + t - t0 + 1);
#pragma unroll
        for (int r = 0; r < RB; ++r) {
            const int c = tx + 16 * r;
            const size_t gi = (size_t)(tb + t) * D + c;
            dqo[gi] = from_f<T>(dq[p][r]);
            if (gated) {
                float ps = kpre[c];  // pooled keys of the segment up to t
                for (int j = 0; j <= t; ++j) ps += Ks[j * P + c];
                duo[gi] = from_f<T>(dua[p][r] - delta[p] * gk[p][r] + dron * ps * inv_cnt);
            }
        }
        if (tx == 0) {
            float *w = tok + (size_t)t * kBwdTokWords;
            w[0] = m_t[t];
            w[1] = z_t[t];
            w[2] = gon[t];
            w[3] = delta[p];
            w[4] = gated ? dron * inv_cnt : 0.f;
            dl[t] = delta[p];
        }
    }
    __syncthreads();

    // dkbar_i -= sum_t g_{t,i} delta_t u_t
    if (gated) {
        if (mode == MC_SSC && tid < kTB) cur[tid] = 0;
        __syncthreads();
        for (int i = 0; i < n; ++i) {
            float gi = 0.f;
            if (tid < kTB) {
                gi = gate_of(tid, i);
                gb[tid] = gi * dl[tid];
            }
            if (!__syncthreads_or(gi != 0.f)) continue;
            if (tid < D) {
                float s = 0.f;
                for (int t = 0; t < cnt; ++t) s = fmaf(gb[t], Us[t * P + tid], s);
                if (s != 0.f) atomicAdd(dkbar + (size_t)i * D + tid, -s);
            }
            __syncthreads();
        }
    }
}

// ---------------------------------------------------------------------------
// bwd_route_simt: the gate work of the tensor-core backward, one CTA per (bh,
// segment n, tile of kTB tokens), heavy segments first.  It reads the gates g_{t,i}
// (routed aggregations: the tensor-core gates pass wrote them with the online gate in
// token word 2; Residual 1; Mean 1 / (n + 1)) and, from the tensor cores, dg_{t,i},
// dg_on and dq, and computes per token
//   delta_t = sum_i g dg + g_on dg_on,  dr_{t,i} = g (dg - delta) -> dr,
//   du_t = sum_i dr_{t,i} kbar_i + dr_on p_t   (p_t = mean of the segment's keys up to t),
//   dq_t in the output type, and for dk / dv the online gate and w = dr_on / cnt_t.
// The gate and dr tables sit in shared memory as [i][t]; for du a warp owns kTB / 8
// tokens and a lane D / 32 dimensions (a register tile over every cached segment).
// ---------------------------------------------------------------------------
template <int CPL, typename T>
__device__ __forceinline__ void load_cols(const T *p, float (&x)[CPL])
{
    if constexpr (std::is_same<T, float>::value && CPL == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else if constexpr (std::is_same<T, __nv_bfloat16>::value && CPL == 4) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.x));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&v.y));
        x[0] = a.x; x[1] = a.y; x[2] = b.x; x[3] = b.y;
    } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) x[c] = to_f(p[c]);
    }
}

template <int CPL, typename T>
__device__ __forceinline__ void store_cols(T *p, const float (&x)[CPL])
{
    if constexpr (std::is_same<T, float>::value && CPL == 4) {
        *reinterpret_cast<float4 *>(p) = make_float4(x[0], x[1], x[2], x[3]);
    } else if constexpr (std::is_same<T, __nv_bfloat16>::value && CPL == 4) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(x[0], x[1]), b = __floats2bfloat162_rn(x[2], x[3]);
        uint2 v;
        v.x = *reinterpret_cast<const uint32_t *>(&a);
        v.y = *reinterpret_cast<const uint32_t *>(&b);
        *reinterpret_cast<uint2 *>(p) = v;
    } else {
#pragma unroll
        for (int c = 0; c < CPL; ++c) p[c] = from_f<T>(x[c]);
    }
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 3) bwd_route_simt(BwdArgs a)
{
    constexpr int CPL = D >= 32 ? D / 32 : 1;  // dimensions per lane
    constexpr int NW = kThreads / 32;
    constexpr int TPW = kTB / NW;              // tokens per warp
    constexpr int PARTS = kThreads / kTB;      // threads per token in the delta sum
    static_assert(TPW == 8 && PARTS * kTB == kThreads, "tile shape");
    __shared__ __align__(16) float gt[kTab * kTB];  // [i][t]: gates
    __shared__ __align__(16) float dt[kTab * kTB];  // [i][t]: dg, then dr
    __shared__ float tot[NW][D];                    // each warp's key sums over its tokens
    __shared__ float red[PARTS][kTB];
    __shared__ float gon[kTB], dgo[kTB], dl[kTB];

    const int tps = (a.C + kTB - 1) / kTB;
    const int per_seg = a.BH * tps;
    const int n = a.N - 1 - (int)(blockIdx.x / per_seg);
    const int rem = blockIdx.x % per_seg;
    const int bh = rem / tps, tile = rem % tps;
    const int t0 = n * a.C;
    const int tb = t0 + tile * kTB;
    const int te = min(min(tb + kTB, t0 + a.C), a.L);
    if (tb >= te) return;
    const int cnt = te - tb;
    const bool gated = gated_mode(a.mode);
    const float gconst = const_gate(a.mode, n);
    const size_t base = (size_t)bh * a.L * D;
    const size_t seg_base = (size_t)bh * a.N * a.L + tb;  // [N][L] tables of this head, at the tile
    const size_t tok0 = (size_t)bh * a.L + tb;            // the tile's first token within the [BH][L] tables
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c0 = CPL * lane;
    const bool lane_on = c0 < D;
    const int tw = warp * TPW;  // the warp's first token of the tile

    constexpr int kV = kTB / 4;  // 16-byte groups of 4 tokens per table row (rows start 64-token aligned)
#pragma unroll 4
    for (int e = tid; e < kV * n; e += kThreads) {  // unrolled: several rows' loads in flight per thread
        const int i = e / kV, t = 4 * (e % kV);
        const size_t gi = seg_base + (size_t)i * a.L + t;
        float4 g4 = make_float4(0.f, 0.f, 0.f, 0.f), d4 = g4;
        if (t + 3 < cnt) {
            g4 = gated ? *reinterpret_cast<const float4 *>(a.gam + gi) : make_float4(gconst, gconst, gconst, gconst);
            d4 = *reinterpret_cast<const float4 *>(a.dg_in + gi);
            if (a.dg_in2) {
                const float4 e4 = *reinterpret_cast<const float4 *>(a.dg_in2 + gi);
                d4.x += e4.x; d4.y += e4.y; d4.z += e4.z; d4.w += e4.w;
            }
        } else {
            float gs[4], ds[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool in = t + k < cnt;
                gs[k] = in ? (gated ? a.gam[gi + k] : gconst) : 0.f;
                ds[k] = in ? a.dg_in[gi + k] + (a.dg_in2 ? a.dg_in2[gi + k] : 0.f) : 0.f;
            }
            g4 = make_float4(gs[0], gs[1], gs[2], gs[3]);
            d4 = make_float4(ds[0], ds[1], ds[2], ds[3]);
        }
        *reinterpret_cast<float4 *>(gt + i * kTB + t) = g4;
        *reinterpret_cast<float4 *>(dt + i * kTB + t) = d4;
    }
    if (tid < kTB) {
        const int t = tid;
        gon[t] = t < cnt ? (gated ? a.tok[(tok0 + t) * kBwdTokWords + 2] : gconst) : 0.f;
        dgo[t] = t < cnt ? a.dgon_in[tok0 + t] + (a.dgon_in2 ? a.dgon_in2[tok0 + t] : 0.f) : 0.f;
    }
    // the key sums of each warp's tokens (the pooled key of the online memory)
    if (gated) {
        const T *k = static_cast<const T *>(a.k) + base;
        float s[CPL];
#pragma unroll
        for (int c = 0; c < CPL; ++c) s[c] = 0.f;
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
            float x[CPL];
#pragma unroll
            for (int c = 0; c < CPL; ++c) x[c] = 0.f;
            if (lane_on && tw + j < cnt) load_cols<CPL>(k + (size_t)(tb + tw + j) * D + c0, x);
#pragma unroll
            for (int c = 0; c < CPL; ++c) s[c] += x[c];
        }
        if (lane_on)
#pragma unroll
            for (int c = 0; c < CPL; ++c) tot[warp][c0 + c] = s[c];
    }
    __syncthreads();
    {  // delta_t: kTB tokens x PARTS strided shares of the segments
        const int t = tid % kTB, part = tid / kTB;
        float s = 0.f;
        for (int i = part; i < n; i += PARTS) s = fmaf(gt[i * kTB + t], dt[i * kTB + t], s);
        red[part][t] = s;
    }
    __syncthreads();
    if (tid < kTB) {
        const int t = tid;
        float s = gon[t] * dgo[t];
#pragma unroll
        for (int part = 0; part < PARTS; ++part) s += red[part][t];
        dl[t] = s;
    }
    __syncthreads();
    // dr = g (dg - delta), in place, and out for the key-mean gradient (4 tokens per thread and step)
#pragma unroll 4
    for (int e = tid; e < kV * n; e += kThreads) {
        const int i = e / kV, t = 4 * (e % kV);
        const float4 g4 = *reinterpret_cast<const float4 *>(gt + i * kTB + t);
        const float4 d4 = *reinterpret_cast<const float4 *>(dt + i * kTB + t);
        const float4 r4 = make_float4(g4.x * (d4.x - dl[t]), g4.y * (d4.y - dl[t + 1]), g4.z * (d4.z - dl[t + 2]),
                                      g4.w * (d4.w - dl[t + 3]));
        *reinterpret_cast<float4 *>(dt + i * kTB + t) = r4;
        if (gated && a.dr_hi) {  // hi = RN(dr), lo = RN(dr - hi): two bf16 terms, 16 bits of dr
            const size_t o = ((size_t)bh * a.Np + i) * a.L + tb + t;
            const float rs[4] = {r4.x, r4.y, r4.z, r4.w};
            __nv_bfloat16 hi[4], lo[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                hi[k] = __float2bfloat16_rn(rs[k]);
                lo[k] = __float2bfloat16_rn(rs[k] - __bfloat162float(hi[k]));
            }
            if (t + 3 < cnt) {
                *reinterpret_cast<uint2 *>(a.dr_hi + o) = *reinterpret_cast<const uint2 *>(hi);
                *reinterpret_cast<uint2 *>(a.dr_lo + o) = *reinterpret_cast<const uint2 *>(lo);
            } else {
                for (int k = 0; k < 4 && t + k < cnt; ++k) {
                    a.dr_hi[o + k] = hi[k];
                    a.dr_lo[o + k] = lo[k];
                }
            }
        } else if (gated && a.dr) {
            float *out = a.dr + seg_base + (size_t)i * a.L + t;
            if (t + 3 < cnt) {
                *reinterpret_cast<float4 *>(out) = r4;
            } else {
                const float rs[4] = {r4.x, r4.y, r4.z, r4.w};
                for (int k = 0; k < 4 && t + k < cnt; ++k) out[k] = rs[k];
            }
        }
    }
    if (gated && a.dr_hi) {  // zero rows n .. up to the next multiple of 16 (the key-mean MMA reads them)
        const int nz = min((n + 15) & ~15, a.Np) - n;
        for (int e = tid; e < nz * kTB; e += kThreads) {
            const int i = n + e / kTB, t = e % kTB;
            if (t < cnt) {
                const size_t o = ((size_t)bh * a.Np + i) * a.L + tb + t;
                a.dr_hi[o] = __float2bfloat16_rn(0.f);
                a.dr_lo[o] = __float2bfloat16_rn(0.f);
            }
        }
    }
    __syncthreads();

    if (lane_on && a.dq_in) {
        T *dqo = static_cast<T *>(a.dq) + base;
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
            const int t = tw + j;
            if (t < cnt) {
                float x[CPL];
                load_cols<CPL>(a.dq_in + (tok0 + t) * D + c0, x);
                store_cols<CPL>(dqo + (size_t)(tb + t) * D + c0, x);
            }
        }
    }
    if (gated && lane_on) {
        float acc[TPW][CPL];
#pragma unroll
        for (int j = 0; j < TPW; ++j)
#pragma unroll
            for (int c = 0; c < CPL; ++c) acc[j][c] = 0.f;
        const float *kb = a.kbar + (size_t)bh * a.N * D + c0;
        for (int i = 0; i < n; ++i) {
            float kv[CPL];
            load_cols<CPL>(kb + (size_t)i * D, kv);
            const float4 r0 = *reinterpret_cast<const float4 *>(dt + i * kTB + tw);
            const float4 r1 = *reinterpret_cast<const float4 *>(dt + i * kTB + tw + 4);
            const float dr[TPW] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
            for (int j = 0; j < TPW; ++j)
#pragma unroll
                for (int c = 0; c < CPL; ++c) acc[j][c] = fmaf(dr[j], kv[c], acc[j][c]);
        }
        // the keys of the segment before the warp's tokens, then through each token
        float off[CPL];
        load_cols<CPL>(a.kpre_tiles + (((size_t)bh * a.N + n) * tps + tile) * D + c0, off);
        for (int w = 0; w < warp; ++w)
#pragma unroll
            for (int c = 0; c < CPL; ++c) off[c] += tot[w][c0 + c];
        T *duo = static_cast<T *>(a.du) + base;
        const T *k = static_cast<const T *>(a.k) + base;
#pragma unroll
        for (int j = 0; j < TPW; ++j) {
            const int t = tw + j;
            if (t < cnt) {
                float x[CPL];
                load_cols<CPL>(k + (size_t)(tb + t) * D + c0, x);  // the running key sum, again (cached)
                const float dron = gon[t] * (dgo[t] - dl[t]);
                const float inv_cnt = 1.f / (float)(tb + t - t0 + 1);
#pragma unroll
                for (int c = 0; c < CPL; ++c) {
                    off[c] += x[c];
                    x[c] = fmaf(dron * off[c], inv_cnt, acc[j][c]);
                }
                store_cols<CPL>(duo + (size_t)(tb + t) * D + c0, x);
            }
        }
    }
    if (tid < cnt) {  // for dk and dv: the online gate and the pooled-key weight
        const int t = tid;
        a.kv_gw[tok0 + t] = gon[t];
        a.kv_gw[(size_t)a.BH * a.L + tok0 + t] = gated ? gon[t] * (dgo[t] - dl[t]) / (float)(tb + t - t0 + 1) : 0.f;
    }
}

// ---------------------------------------------------------------------------
// bwd_dkbar_simt: the key-mean gradients from the score gradients,
// dkbar_i = sum_{t : n(t) > i} dr_{t,i} u_t, on the shapes of the tensor-core path
// (N <= 64, seg_len and L multiples of kDkSub, so each kDkSub-token sub-chunk lies in
// one segment).  One CTA per (bh, kDkChunk tokens), the last chunks (the most cached
// segments scored) first: every token's u is read once and
// feeds every cached segment it scored; a thread keeps one dimension's sums for all
// segments over a strided share of each sub-chunk, four tokens per step.  The
// sub-chunks' dr rows are staged in shared memory by asynchronous copies, two
// buffers deep; the CTA adds its sums to dkbar (zeroed first).
// ---------------------------------------------------------------------------
constexpr int kDkChunk = 1024;
constexpr int kDkSub = 128;
constexpr size_t kDkSmem = 2 * sizeof(float) * kTab * kDkSub;

__device__ __forceinline__ void cp_async16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_one() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_dkbar_simt(BwdArgs a, int chunks)
{
    constexpr int parts = kThreads / D;
    constexpr int TG = 4;  // tokens per step: one 16-byte row of dr per segment
    extern __shared__ __align__(16) float sdr[];  // [2][kTab][kDkSub]
    const int ch = chunks - 1 - (int)blockIdx.x / a.BH, bh = (int)blockIdx.x % a.BH;  // the most scores first
    const int t_lo = ch * kDkChunk, t_hi = min(t_lo + kDkChunk, a.L);
    const int nsub = (t_hi - t_lo) / kDkSub;
    const int col = threadIdx.x % D, part = threadIdx.x / D;
    const int nmax = min(a.N - 1, (t_hi - 1) / a.C);  // cached segments any token of the chunk scored
    const T *u = static_cast<const T *>(a.u) + (size_t)bh * a.L * D + col;
    const float *dr = a.dr + (size_t)bh * a.N * a.L;
    // sub-chunk s into buffer s % 2: the rows of the segments its tokens scored
    auto stage = [&](int s) {
        const int t0 = t_lo + s * kDkSub;
        const int ns = min(t0 / a.C, kTab);
        float *dst = sdr + (s & 1) * kTab * kDkSub;
        for (int e = threadIdx.x; e < ns * (kDkSub / 4); e += kThreads) {
            const int i = e / (kDkSub / 4), q = e % (kDkSub / 4);
            cp_async16(dst + i * kDkSub + 4 * q, dr + (size_t)i * a.L + t0 + 4 * q);
        }
        cp_async_commit();
    };
    float acc[kTab];
#pragma unroll
    for (int i = 0; i < kTab; ++i) acc[i] = 0.f;
    stage(0);
    if (nsub > 1) stage(1);
    else cp_async_commit();
    for (int s = 0; s < nsub; ++s) {
        cp_async_wait_one();  // every group but the newest: sub-chunk s is in
        __syncthreads();
        const int t0 = t_lo + s * kDkSub;
        const int ns = min(t0 / a.C, kTab);
        const float *buf = sdr + (s & 1) * kTab * kDkSub;
        float un[TG];
#pragma unroll
        for (int j = 0; j < TG; ++j) un[j] = to_f(u[(size_t)(t0 + part * TG + j) * D]);
        for (int t = part * TG; t < kDkSub; t += parts * TG) {
            float uv[TG];
#pragma unroll
            for (int j = 0; j < TG; ++j) uv[j] = un[j];
            if (t + parts * TG < kDkSub)
#pragma unroll
                for (int j = 0; j < TG; ++j) un[j] = to_f(u[(size_t)(t0 + t + parts * TG + j) * D]);
#pragma unroll
            for (int ib = 0; ib < kTab / 8; ++ib) {
                if (8 * ib >= ns) break;
#pragma unroll
                for (int ii = 0; ii < 8; ++ii) {
                    const int i = 8 * ib + ii;
                    if (i < ns) {
                        const float4 r = *reinterpret_cast<const float4 *>(buf + i * kDkSub + t);
                        acc[i] = fmaf(r.x, uv[0], fmaf(r.y, uv[1], fmaf(r.z, uv[2], fmaf(r.w, uv[3], acc[i]))));
                    }
                }
            }
        }
        __syncthreads();  // buffer s % 2 is free again
        if (s + 2 < nsub) stage(s + 2);
        else cp_async_commit();
    }
    float *dk = a.dkbar + (size_t)bh * a.N * D + col;
#pragma unroll
    for (int i = 0; i < kTab; ++i)
        if (i < nmax && acc[i] != 0.f) atomicAdd(dk + (size_t)i * D, acc[i]);
}

// ---------------------------------------------------------------------------
// bwd_G_simt: one CTA per (bh, cached segment i < N-1), i = 0 (the most later
// tokens) first.  G_i = sum_{t >= (i+1) C} g_{t,i} dy_t q_t^T; a thread owns the
// entries (ty + 16 a, tx + 16 b).  The gate is recomputed the way bwd_gates_simt
// computed it (same score arithmetic, its softmax max and sum) or read from the
// SSC selection.
// ---------------------------------------------------------------------------
template <typename T, int D>
__global__ void __launch_bounds__(kThreads) bwd_G_simt(BwdArgs a)
{
    constexpr int P = D + 1;
    constexpr int RB = D / 16;
    extern __shared__ float sm[];
    float *Ys = sm;            // kTG x P  (g dy)
    float *Qs = Ys + kTG * P;  // kTG x P
    float *Us = Qs + kTG * P;  // kTG x P
    float *gb = Us + kTG * P;  // kTG

    const int i = (int)blockIdx.x / a.BH, bh = (int)blockIdx.x % a.BH;
    const int mode = a.mode;
    const bool gated = gated_mode(mode);
    const size_t base = (size_t)bh * a.L * D;
    const T *q = static_cast<const T *>(a.q) + base, *dy = static_cast<const T *>(a.dy) + base;
    const T *u = gated ? static_cast<const T *>(a.u) + base : nullptr;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;
    const float *kbi = a.kbar + ((size_t)bh * a.N + i) * D;  // global: gate_score reads it through the read-only path

    float G[RB][RB];
#pragma unroll
    for (int x = 0; x < RB; ++x)
#pragma unroll
        for (int y = 0; y < RB; ++y) G[x][y] = 0.f;

    for (int c0 = (i + 1) * a.C; c0 < a.L; c0 += kTG) {
        const int cnt = min(kTG, a.L - c0);
        __syncthreads();
        for (int e = tid; e < kTG * D; e += kThreads) {
            const int r = e / D, c = e % D;
            const bool ok = r < cnt;
            const size_t gi = (size_t)(c0 + r) * D + c;
            Ys[r * P + c] = ok ? to_f(dy[gi]) : 0.f;
            Qs[r * P + c] = ok ? to_f(q[gi]) : 0.f;
            if (mode != MC_SSC && gated) Us[r * P + c] = ok ? to_f(u[gi]) : 0.f;
        }
        __syncthreads();
        if (tid < kTG) {
            const int t = c0 + tid;
            float g = 0.f;
            if (tid < cnt) {
                const float *tw = a.tok + ((size_t)bh * a.L + t) * kBwdTokWords;
                if (!gated) {
                    g = const_gate(mode, t / a.C);
                } else if (mode == MC_SSC) {
                    const int32_t *si = a.sel_idx + ((size_t)bh * a.L + t) * a.topk;
                    const float *sg = a.sel_g + ((size_t)bh * a.L + t) * a.topk;
                    for (int c = 0; c < a.topk; ++c)
                        if (si[c] == i) g = sg[c];
                } else {
                    g = expf(gate_score(Us + tid * P, kbi, D) - tw[0]) / tw[1];
                }
            }
            gb[tid] = g;
        }
        __syncthreads();
        for (int t = 0; t < cnt; ++t) {
            const float g = gb[t];
            if (g == 0.f) continue;  // uniform across the CTA
            float yv[RB], qv[RB];
#pragma unroll
            for (int x = 0; x < RB; ++x) yv[x] = g * Ys[t * P + ty + 16 * x];
#pragma unroll
            for (int y = 0; y < RB; ++y) qv[y] = Qs[t * P + tx + 16 * y];
#pragma unroll
            for (int x = 0; x < RB; ++x)
#pragma unroll
                for (int y = 0; y < RB; ++y) G[x][y] = fmaf(yv[x], qv[y], G[x][y]);
        }
    }
    float *Go = a.G + ((size_t)bh * a.N + i) * D * D;
#pragma unroll
    for (int x = 0; x < RB; ++x)
#pragma unroll
        for (int y = 0; y < RB; ++y) Go[(size_t)(ty + 16 * x) * D + tx + 16 * y] = G[x][y];
}

// ---------------------------------------------------------------------------
// bwd_scan_simt: one CTA per (bh, segment n).  Walks the segment's chunks of TC
// tokens from the last to the first with E = G_n + sum_{t in later chunks} g_on dy_t q_t^T
// (a thread owns E entries (ty + 16 i, tx + 16 j)) and the running sum of the pooled
// key gradient of later tokens.  For token j of a chunk (t over the chunk, t >= j):
//   dv_j = E k_j + sum_t g_on[t] (q_t . k_j) dy_t
//   dk_j = E^T v_j + sum_t g_on[t] (dy_t . v_j) q_t + dkbar_n / |n| + psum + sum_t w_t u_t
// ---------------------------------------------------------------------------
template <typename T, int D, int TC>
__global__ void __launch_bounds__(kThreads) bwd_scan_simt(BwdArgs a)
{
    constexpr int P = D + 1;
    constexpr int TP = TC + 1;
    constexpr int RB = D / 16;
    constexpr int TPT = TC / 16;
    extern __shared__ float sm[];
    float *Qs = sm;
    float *Ks = Qs + TC * P;
    float *Vs = Ks + TC * P;
    float *Ys = Vs + TC * P;   // g_on dy
    float *Uw = Ys + TC * P;   // w u
    float *Es = Uw + TC * P;   // D x P
    float *As = Es + D * P;    // TC x TP: [j][t] = k_j . q_t, t >= j
    float *Bs = As + TC * TP;  // TC x TP: [j][t] = v_j . (g dy)_t, t >= j
    float *rho = Bs + TC * TP; // D: dkbar_n / |n| + pooled-key gradient of later chunks

    const int n = (int)blockIdx.x % a.N, bh = (int)blockIdx.x / a.N;
    const int t0 = n * a.C, t1 = min(t0 + a.C, a.L);
    const int mode = a.mode;
    const bool gated = gated_mode(mode);
    const size_t base = (size_t)bh * a.L * D;
    const T *q = static_cast<const T *>(a.q) + base, *k = static_cast<const T *>(a.k) + base;
    const T *v = static_cast<const T *>(a.v) + base, *dy = static_cast<const T *>(a.dy) + base;
    const T *u = gated ? static_cast<const T *>(a.u) + base : nullptr;
    T *dko = static_cast<T *>(a.dk) + base, *dvo = static_cast<T *>(a.dv) + base;
    const float *tok = a.tok + (size_t)bh * a.L * kBwdTokWords;
    const int tid = threadIdx.x, tx = tid % 16, ty = tid / 16;

    float E[RB][RB];
    const float *Gn = n < a.N - 1 ? a.G + ((size_t)bh * a.N + n) * D * D : nullptr;
#pragma unroll
    for (int x = 0; x < RB; ++x)
#pragma unroll
        for (int y = 0; y < RB; ++y) {
            const int r = ty + 16 * x, c = tx + 16 * y;
            E[x][y] = Gn ? Gn[(size_t)r * D + c] : 0.f;
            Es[r * P + c] = E[x][y];
        }
    if (tid < D) rho[tid] = gated ? a.dkbar[((size_t)bh * a.N + n) * D + tid] / (float)(t1 - t0) : 0.f;

    const int nch = (t1 - t0 + TC - 1) / TC;
    for (int ch = nch - 1; ch >= 0; --ch) {
        const int c0 = t0 + ch * TC;
        const int cnt = min(TC, t1 - c0);
        __syncthreads();
        for (int e = tid; e < TC * D; e += kThreads) {
            const int r = e / D, c = e % D;
            const bool ok = r < cnt;
            const size_t g = (size_t)(c0 + r) * D + c;
            const float *tw = tok + (size_t)(c0 + r) * kBwdTokWords;
            Qs[r * P + c] = ok ? to_f(q[g]) : 0.f;
            Ks[r * P + c] = ok ? to_f(k[g]) : 0.f;
            Vs[r * P + c] = ok ? to_f(v[g]) : 0.f;
            Ys[r * P + c] = ok ? tw[2] * to_f(dy[g]) : 0.f;
            Uw[r * P + c] = (ok && gated) ? tw[4] * to_f(u[g]) : 0.f;
        }
        __syncthreads();
        for (int e = tid; e < TC * TC; e += kThreads) {
            const int j = e / TC, t = e % TC;
            float acc = 0.f, accb = 0.f;
            if (t >= j && t < cnt) {
                for (int c = 0; c < D; ++c) {
                    acc = fmaf(Ks[j * P + c], Qs[t * P + c], acc);
                    accb = fmaf(Vs[j * P + c], Ys[t * P + c], accb);
                }
            }
            As[j * TP + t] = acc;
            Bs[j * TP + t] = accb;
        }
        __syncthreads();
        {
            float dv[TPT][RB], dk[TPT][RB];
#pragma unroll
            for (int p = 0; p < TPT; ++p)
#pragma unroll
                for (int r = 0; r < RB; ++r) dv[p][r] = dk[p][r] = 0.f;
            for (int c = 0; c < D; ++c) {
                float kv[TPT], vv[TPT];
#pragma unroll
                for (int p = 0; p < TPT; ++p) {
                    kv[p] = Ks[(ty + 16 * p) * P + c];
                    vv[p] = Vs[(ty + 16 * p) * P + c];
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const float er = Es[(tx + 16 * r) * P + c];  // E[value dim tx + 16 r][key dim c]
                    const float ec = Es[c * P + tx + 16 * r];    // E[value dim c][key dim tx + 16 r]
#pragma unroll
                    for (int p = 0; p < TPT; ++p) {
                        dv[p][r] = fmaf(er, kv[p], dv[p][r]);
                        dk[p][r] = fmaf(ec, vv[p], dk[p][r]);
                    }
                }
            }
            for (int t = 0; t < cnt; ++t) {
                float av[TPT], bv[TPT];
#pragma unroll
                for (int p = 0; p < TPT; ++p) {
                    av[p] = As[(ty + 16 * p) * TP + t];
                    bv[p] = Bs[(ty + 16 * p) * TP + t];
                }
#pragma unroll
                for (int r = 0; r < RB; ++r) {
                    const float yv = Ys[t * P + tx + 16 * r], qv = Qs[t * P + tx + 16 * r];
                    const float uw = Uw[t * P + tx + 16 * r];
#pragma unroll
                    for (int p = 0; p < TPT; ++p) {
                        dv[p][r] = fmaf(av[p], yv, dv[p][r]);
                        dk[p][r] = fmaf(bv[p], qv, dk[p][r]);
                        if (t >= ty + 16 * p) dk[p][r] += uw;  // pooled keys of the tokens t >= j
                    }
                }
            }
#pragma unroll
            for (int p = 0; p < TPT; ++p) {
                const int j = ty + 16 * p;
                if (j < cnt) {
#pragma unroll
                    for (int r = 0; r < RB; ++r) {
                        const size_t g = (size_t)(c0 + j) * D + tx + 16 * r;
                        dvo[g] = from_f<T>(dv[p][r]);
                        dko[g] = from_f<T>(dk[p][r] + rho[tx + 16 * r]);
                    }
                }
            }
        }
        __syncthreads();  // Es and rho are read above and rewritten below
        for (int t = 0; t < cnt; ++t) {
            float yv[RB], qv[RB];
#pragma unroll
            for (int x = 0; x < RB; ++x) yv[x] = Ys[t * P + ty + 16 * x];
#pragma unroll
            for (int y = 0; y < RB; ++y) qv[y] = Qs[t * P + tx + 16 * y];
#pragma unroll
            for (int x = 0; x < RB; ++x)
#pragma unroll
                for (int y = 0; y < RB; ++y) E[x][y] = fmaf(yv[x], qv[y], E[x][y]);
        }
#pragma unroll
        for (int x = 0; x < RB; ++x)
#pragma unroll
            for (int y = 0; y < RB; ++y) Es[(ty + 16 * x) * P + tx + 16 * y] = E[x][y];
        if (tid < D) {
            float s = rho[tid];
            for (int t = 0; t < cnt; ++t) s += Uw[t * P + tid];
            rho[tid] = s;
        }
    }
}

template <typename T, int D>
cudaError_t gates_impl(const Problem &p, const BwdArgs &a, cudaStream_t s)
{
    constexpr int P = D + 1;
    constexpr int KC = D < 32 ? D : 32;
    const size_t smem = sizeof(float) * (4 * kTB * P + D * (KC + 1) + 2 * D + 6 * kTB + kTB * kMaxTopk + kTB * kTab) +
                        sizeof(int) * (kTB * kMaxTopk + 2 * kTB);
    auto kern = bwd_gates_simt<T, D>;
    cudaError_t e = set_smem(kern, smem);
    if (e != cudaSuccess) return e;
    const long long tps = (p.C + kTB - 1) / kTB;
    kern<<<(unsigned)((long long)p.BH * p.N * tps), kThreads, smem, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_after_kernel(s, "bwd_gates_simt");
    return cudaSuccess;
}

template <typename T, int D>
cudaError_t backward_impl(const Problem &p, const BwdArgs &a, cudaStream_t s)
{
    constexpr int P = D + 1;
    cudaError_t e = gates_impl<T, D>(p, a, s);
    if (e != cudaSuccess) return e;
    if (p.N > 1) {
        const size_t smem = sizeof(float) * (3 * kTG * P + kTG);
        auto kern = bwd_G_simt<T, D>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        kern<<<(unsigned)((long long)p.BH * (p.N - 1)), kThreads, smem, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "bwd_G_simt");
    }
    {
        constexpr int TC = D >= 128 ? 32 : 64;
        constexpr int TP = TC + 1;
        const size_t smem = sizeof(float) * (5 * TC * P + D * P + 2 * TC * TP + D);
        auto kern = bwd_scan_simt<T, D, TC>;
        if ((e = set_smem(kern, smem)) != cudaSuccess) return e;
        kern<<<(unsigned)((long long)p.BH * p.N), kThreads, smem, s>>>(a);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "bwd_scan_simt");
    }
    return cudaSuccess;
}

#define MC_BWD_DISPATCH(FN, p, a, s)                                                                 \
    do {                                                                                           \
        switch ((p).d) {                                                                           \
        case 16: return (p).bf16 ? FN<__nv_bfloat16, 16>(p, a, s) : FN<float, 16>(p, a, s);   \
        case 32: return (p).bf16 ? FN<__nv_bfloat16, 32>(p, a, s) : FN<float, 32>(p, a, s);   \
        case 64: return (p).bf16 ? FN<__nv_bfloat16, 64>(p, a, s) : FN<float, 64>(p, a, s);   \
        case 128: return (p).bf16 ? FN<__nv_bfloat16, 128>(p, a, s) : FN<float, 128>(p, a, s); \
        default: return cudaErrorInvalidValue;                                                     \
        }                                                                                          \
    } while (0)

template <typename T, int D>
cudaError_t route_impl(const Problem &p, const BwdArgs &a, cudaStream_t s)
{
    cudaError_t e;
    const long long tps = (p.C + kTB - 1) / kTB;
    bwd_route_simt<T, D><<<(unsigned)((long long)p.BH * p.N * tps), kThreads, 0, s>>>(a);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    profile_after_kernel(s, "bwd_route_simt");
    if (a.dr_hi && p.N > 1) {  // the key-mean gradient on the tensor cores
        if ((e = launch_bwd_dkbar_tc(p, a.u, a.dr_hi, a.dr_lo, a.Np, a.dkbar, s)) != cudaSuccess) return e;
        profile_after_kernel(s, "bwd_dkbar_tc");
    } else if (a.dr && p.N > 1) {
        const int chunks = (p.L + kDkChunk - 1) / kDkChunk;
        if ((e = set_smem(bwd_dkbar_simt<T, D>, kDkSmem)) != cudaSuccess) return e;
        bwd_dkbar_simt<T, D><<<(unsigned)((long long)p.BH * chunks), kThreads, kDkSmem, s>>>(a, chunks);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        profile_after_kernel(s, "bwd_dkbar_simt");
    }
    return cudaSuccess;
}

// The tensor-core path after the cached pass: the gate work, G and dk / dv on the tensor cores.
template <typename T, int D>
cudaError_t backward_tc_impl(const Problem &p, const BwdArgs &a, cudaStream_t s)
{
    cudaError_t e = route_impl<T, D>(p, a, s);
    if (e != cudaSuccess) return e;
    uint8_t *Gimg = reinterpret_cast<uint8_t *>(a.G);
    if (p.N > 1) {
        if ((e = launch_bwd_G_tc(p, a.dy, a.q, a.gam, Gimg, s)) != cudaSuccess) return e;
        profile_after_kernel(s, "bwd_G_tc");
    }
    if ((e = launch_bwd_kv_tc(p, a.q, a.k, a.v, a.u, a.dy, Gimg, a.kv_gw, a.dkbar, a.dk, a.dv, s)) != cudaSuccess) return e;
    profile_after_kernel(s, "bwd_kv_tc");
    return cudaSuccess;
}

cudaError_t launch_bwd_kernels(const Problem &p, const BwdArgs &a, cudaStream_t s) { MC_BWD_DISPATCH(backward_impl, p, a, s); }
cudaError_t launch_bwd_tc_rest(const Problem &p, const BwdArgs &a, cudaStream_t s) { MC_BWD_DISPATCH(backward_tc_impl, p, a, s); }

size_t pad256(size_t x) { return (x + 255) & ~(size_t)255; }

}  // namespace

// Scratch of one backward call.  FFMA path, in this order: states, G (N d^2 floats
// per head each), kbar, dkbar (N d), r_on (L), O_on, X_on (L d), per-token words
// (L x 5), SSC selection indices and gates (L x topk each).  Tensor-core path: states,
// G, kbar, dkbar, per-token words, the gates of the cached segments (routed: L x N),
// the keys before each 64-token tile (routed), the online gates and pooled-key
// weights (2 L), the forward state kernel's images and r_on, and the cached pass's
// outputs.
size_t backward_scratch_bytes(const Problem &p)
{
    const size_t BH = p.BH, N = p.N, L = p.L, d = p.d;
    const size_t gbytes = bwd_tc_supported(p) ? (size_t)32768 * BH * N : 4 * BH * N * d * d;  // G: images or fp32
    const size_t common = pad256(4 * BH * N * d * d) + pad256(gbytes) + 2 * pad256(4 * BH * N * d) +
                          pad256(4 * BH * L * kBwdTokWords);
    if (bwd_tc_supported(p)) {
        const size_t gam = mode_uses_u(p.mode) ? N : 0;
        const size_t kpre = mode_uses_u(p.mode) ? N * ((p.C + kTB - 1) / kTB) * d : 0;
        const size_t drp = mode_uses_u(p.mode) ? 2 * pad256(2 * BH * ((N + 15) & ~(size_t)15) * L) : 0;
        return common + pad256(4 * BH * L * gam) + pad256(4 * BH * kpre) + pad256(8 * BH * L) +
               pad256(tc_state_scratch_bytes(p)) + pad256(bwd_cached_scratch_bytes(p)) + drp;
    }
    const size_t sel = p.mode == MC_SSC ? (size_t)p.topk : 0;
    return common + pad256(4 * BH * L) + 2 * pad256(4 * BH * L * d) + 2 * pad256(4 * BH * L * sel);
}

cudaError_t launch_backward_simt(const Problem &p, const void *q, const void *k, const void *v, const void *u,
                                 const void *dy, void *dq, void *dk, void *dv, void *du, void *scratch,
                                 cudaStream_t s)
{
    const size_t BH = p.BH, N = p.N, L = p.L, d = p.d;
    char *b = static_cast<char *>(scratch);
    auto take = [&](size_t bytes) {
        char *r = b;
        b += pad256(bytes);
        return r;
    };
    const bool gated = p.mode == MC_GRM || p.mode == MC_SOUP || p.mode == MC_SSC;
    const bool tc = bwd_tc_supported(p);
    float *states = reinterpret_cast<float *>(take(4 * BH * N * d * d));
    float *G = reinterpret_cast<float *>(take(tc ? (size_t)32768 * BH * N : 4 * BH * N * d * d));
    float *kbar = reinterpret_cast<float *>(take(4 * BH * N * d));
    float *dkbar = reinterpret_cast<float *>(take(4 * BH * N * d));
    float *tok = reinterpret_cast<float *>(take(4 * BH * L * kBwdTokWords));

    BwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.u = gated ? u : nullptr; a.dy = dy;
    a.dq = dq; a.dk = dk; a.dv = dv; a.du = gated ? du : nullptr;
    a.states = states; a.kbar = kbar;
    a.G = G; a.dkbar = dkbar; a.tok = tok;
    a.BH = p.BH; a.L = p.L; a.C = p.C; a.N = p.N; a.mode = p.mode; a.topk = p.topk;
    FwdArgs f{};
    f.q = q; f.k = k; f.v = v; f.u = gated ? u : nullptr;
    f.states = states; f.kbar = kbar;
    f.BH = p.BH; f.L = p.L; f.C = p.C; f.N = p.N; f.mode = p.mode; f.topk = p.topk;
    cudaError_t e;
    profile_call_start(s);

    if (tc) {
        // Tensor-core path: the forward's state kernel (state, prefix-state and key-mean images,
        // r_on), the key means, the gates (routed, tensor cores), every memory's read on the tensor
        // cores (dg, the online dg, dq), the gate work on whole tables, the key-mean gradient, G
        // and dk / dv on the tensor cores.
        float *gam = gated ? reinterpret_cast<float *>(take(4 * BH * L * N)) : nullptr;
        a.kpre_tiles = gated ? reinterpret_cast<float *>(take(4 * BH * N * ((p.C + kTB - 1) / kTB) * d)) : nullptr;
        a.kv_gw = reinterpret_cast<float *>(take(8 * BH * L));
        f.kpre_tiles = a.kpre_tiles;  // the state kernel writes the key means and the tile key prefixes
        void *state_scratch = take(tc_state_scratch_bytes(p));
        void *cached_scratch = take(bwd_cached_scratch_bytes(p));
        TcImages img{};
        if ((e = launch_state_tc(p, f, state_scratch, &img, s)) != cudaSuccess) return e;
        profile_after_kernel(s, "seg_state_tc");
        if ((e = cudaMemsetAsync(dkbar, 0, 4 * BH * N * d, s)) != cudaSuccess) return e;
        a.r_on = img.r_on;
        a.gam = gam;
        if (gated) {  // the gates on the tensor cores, from the state kernel's key-mean images and r_on
            if ((e = launch_bwd_gates_tc(p, u, img, gam, tok, s)) != cudaSuccess) return e;
            profile_after_kernel(s, "gate_tiles_tc");
        }
        float *dg = nullptr, *dgon = nullptr;
        if ((e = launch_bwd_cached_tc(p, q, k, v, dy, img, gam, tok, dq, cached_scratch, &dg, &dgon, s)) != cudaSuccess)
            return e;
        profile_after_kernel(s, "bwd_cached_tc");
        a.dg_in = dg;
        a.dgon_in = dgon;
        a.dg_in2 = dg + BH * N * L;  // the cached pass's second column half
        a.dgon_in2 = dgon + BH * L;
        a.dq_in = nullptr;  // dq is written whole by the cached pass
        a.dr = nullptr;
        if (gated) {  // the score gradients as the key-mean MMA's bf16 hi / lo planes
            a.Np = (int)((N + 15) & ~(size_t)15);
            a.dr_hi = reinterpret_cast<__nv_bfloat16 *>(take(2 * BH * a.Np * L));
            a.dr_lo = reinterpret_cast<__nv_bfloat16 *>(take(2 * BH * a.Np * L));
        }
        return launch_bwd_tc_rest(p, a, s);
    }

    // FFMA path
    const size_t sel = p.mode == MC_SSC ? (size_t)p.topk : 0;
    float *r_on = reinterpret_cast<float *>(take(4 * BH * L));
    float *O_on = reinterpret_cast<float *>(take(4 * BH * L * d));
    float *X_on = reinterpret_cast<float *>(take(4 * BH * L * d));
    int32_t *sel_idx = reinterpret_cast<int32_t *>(take(4 * BH * L * sel));
    float *sel_g = reinterpret_cast<float *>(take(4 * BH * L * sel));
    // The forward's segment scan: cached states, key means, online scores, M_t q_t.
    f.O_on = O_on;
    f.r_on = r_on;
    if ((e = launch_seg_scan_simt(p, f, s)) != cudaSuccess) return e;
    profile_after_kernel(s, "seg_scan_simt");
    // The same scan on (dy, v, k) gives M_t^T dy_t = sum_{j <= t} k_j (v_j . dy_t); its state and
    // key-mean outputs land in G and dkbar, which are rewritten below.
    FwdArgs x = f;
    x.q = dy; x.k = v; x.v = k; x.u = nullptr;
    x.states = G; x.O_on = X_on; x.kbar = dkbar;
    if ((e = launch_seg_scan_simt(p, x, s)) != cudaSuccess) return e;
    profile_after_kernel(s, "seg_scan_simt");
    if ((e = cudaMemsetAsync(dkbar, 0, 4 * BH * N * d, s)) != cudaSuccess) return e;
    a.r_on = r_on; a.O_on = O_on; a.X_on = X_on;
    a.sel_idx = sel_idx; a.sel_g = sel_g;
    return launch_bwd_kernels(p, a, s);
}

}  // namespace mc
