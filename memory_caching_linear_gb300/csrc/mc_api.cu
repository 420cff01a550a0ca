// mc_api.cu -- the C ABI declared in include/mc.h: argument checks, stream-ordered
// scratch, and the choice of kernels for a shape.
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <array>
#include <atomic>
#include <mutex>
#include <vector>

#include "mc_internal.cuh"

namespace mc {

namespace {
// Scratch comes from a library-owned stream-ordered pool per device that keeps
// freed blocks cached (release threshold = all), so repeated calls -- including
// calls that synchronise, like mc_forward_host -- do not re-map device memory.
// mc_trim_scratch() returns the cached memory to the driver.
std::mutex g_pool_mu;
cudaMemPool_t g_pools[64];

cudaMemPool_t scratch_pool()
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_pool_mu);
    if (!g_pools[dev]) {
        cudaMemPoolProps props{};
        props.allocType = cudaMemAllocationTypePinned;
        props.location.type = cudaMemLocationTypeDevice;
        props.location.id = dev;
        cudaMemPool_t pool = nullptr;
        if (cudaMemPoolCreate(&pool, &props) != cudaSuccess) {
            cudaGetLastError();
            return nullptr;
        }
        uint64_t keep = UINT64_MAX;
        cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &keep);
        g_pools[dev] = pool;
    }
    return g_pools[dev];
}
}  // namespace

cudaError_t scratch_alloc(void **p, size_t bytes, cudaStream_t s)
{
    cudaMemPool_t pool = scratch_pool();
    if (!pool) return cudaMallocAsync(p, bytes, s);
    return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

namespace {
struct ProfileState {
    void *const *events = nullptr;
    int capacity = 0;
    int count = 0;
    const char *stage[4096];  // stage[j]: kernel between event j and j+1
};
ProfileState g_prof;
}  // namespace

void profile_call_start(cudaStream_t s)
{
    if (!g_prof.events || g_prof.count >= g_prof.capacity) return;
    if (g_prof.count > 0 && g_prof.count - 1 < 4096) g_prof.stage[g_prof.count - 1] = nullptr;
    cudaEventRecord(static_cast<cudaEvent_t>(g_prof.events[g_prof.count]), s);
    ++g_prof.count;
}

void profile_after_kernel(cudaStream_t s, const char *name)
{
    if (!g_prof.events || g_prof.count >= g_prof.capacity) return;
    if (g_prof.count - 1 < 4096) g_prof.stage[g_prof.count - 1] = name;
    cudaEventRecord(static_cast<cudaEvent_t>(g_prof.events[g_prof.count]), s);
    ++g_prof.count;
}

namespace {

std::atomic<int> g_readout_form{MC_READOUT_AUTO};

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int check_device()
{
    // The library is built for sm_103a only; refuse anything else up front.
    static int cached[64];  // 0 unknown, 1 ok, 2 not ok
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MC_ERR_CUDA;
    if (dev >= 0 && dev < 64 && cached[dev]) return cached[dev] == 1 ? MC_OK : MC_ERR_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return MC_ERR_CUDA;
    const bool ok = major == 10 && minor == 3;
    if (dev >= 0 && dev < 64) cached[dev] = ok ? 1 : 2;
    return ok ? MC_OK : MC_ERR_DEVICE;
}

int check_shape(int B, int H, int L, int d, int seg_len)
{
    if (B < 1 || H < 1 || L < 1 || seg_len < 1) return MC_ERR_SHAPE;
    if (d != 16 && d != 32 && d != 64 && d != 128) return MC_ERR_SHAPE;
    const long long BH = (long long)B * H;
    const long long N = ((long long)L + seg_len - 1) / seg_len;
    if (BH > (1ll << 24)) return MC_ERR_SHAPE;
    // every element count used for indexing fits in 62 bits and the grids fit in 2^31 blocks
    if (BH * L * d > (1ll << 40) || BH * N * d * d > (1ll << 40)) return MC_ERR_SHAPE;
    if (BH * N * ((seg_len + 63) / 64) >= (1ll << 31)) return MC_ERR_SHAPE;
    return MC_OK;
}

size_t round_up(size_t x) { return (x + 255) & ~(size_t)255; }

struct ScratchPlan {
    size_t off_states, off_O, off_r, off_kbar, total;
};

ScratchPlan plan_scratch(const Problem &p, bool need_states)
{
    ScratchPlan s{};
    size_t off = 0;
    s.off_states = off;
    if (need_states) off += round_up(sizeof(float) * (size_t)p.BH * p.N * p.d * p.d);
    s.off_O = off;
    off += round_up(sizeof(float) * (size_t)p.BH * p.L * p.d);
    s.off_r = off;
    off += round_up(sizeof(float) * (size_t)p.BH * p.L);
    s.off_kbar = off;
    off += round_up(sizeof(float) * (size_t)p.BH * p.N * p.d);
    s.total = off;
    return s;
}

int forward_common(const void *q, const void *k, const void *v, const void *u, int B, int H, int L, int d,
                   int seg_len, int agg_mode, int topk, void *y, float *states, bool bf16, cudaStream_t stream,
                   const float *alpha = nullptr, const float *beta = nullptr, const float *lam = nullptr,
                   bool swla = false)
{
    int st = check_shape(B, H, L, d, seg_len);
    if (st != MC_OK) return st;
    if (agg_mode < MC_RESIDUAL || agg_mode > MC_MEAN) return MC_ERR_MODE;
    if (!q || !k || !v || !y) return MC_ERR_NULL;
    if (mode_uses_u(agg_mode) && !u) return MC_ERR_NULL;
    if (swla && (!alpha || !beta || !lam)) return MC_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y) || (u && !aligned16(u)) ||
        (states && !aligned16(states)) || (swla && (!aligned16(alpha) || !aligned16(beta) || !aligned16(lam))))
        return MC_ERR_ALIGN;
    Problem p{};
    p.B = B; p.H = H; p.L = L; p.d = d; p.C = seg_len;
    p.N = (L + seg_len - 1) / seg_len;
    p.BH = B * H;
    p.bf16 = bf16;
    p.mode = agg_mode;
    p.topk = agg_mode == MC_SSC ? topk : 0;
    if (agg_mode == MC_SSC) {
        if (topk < 0) return MC_ERR_TOPK;
        // topk >= N-1 selects every cached segment for every token: that is GRM exactly.
        if (topk >= p.N - 1) p.mode = MC_GRM;
        else if (topk > kMaxTopk) return MC_ERR_TOPK;
    }
    if (swla && !tc_fused_gates(p)) return MC_ERR_SHAPE;  // the SWLA update runs on the tensor-core path only
    st = check_device();
    if (st != MC_OK) return st;

    const bool factorised = g_readout_form.load() == MC_READOUT_FACTORISED && !swla && gen_supported(p);
    if (tc_supported(p) && !factorised) {
        const size_t b_states = states ? 0 : round_up(sizeof(float) * (size_t)p.BH * p.N * d * d);
        void *scratch = nullptr;
        if (scratch_alloc(&scratch, b_states + tc_scratch_bytes(p), stream) != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_ALLOC;
        }
        FwdArgs a{};
        a.q = q; a.k = k; a.v = v;
        a.u = mode_uses_u(p.mode) ? u : nullptr;
        a.y = y;
        a.states = states ? states : static_cast<float *>(scratch);
        a.alpha = swla ? alpha : nullptr;
        a.beta = swla ? beta : nullptr;
        a.lam = swla ? lam : nullptr;
        a.BH = p.BH; a.L = L; a.C = seg_len; a.N = p.N; a.mode = p.mode; a.topk = p.topk;
        cudaError_t e = launch_forward_tc(p, a, static_cast<char *>(scratch) + b_states, stream);
        cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e != cudaSuccess || ef != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_CUDA;
        }
        return MC_OK;
    }

    if (gen_supported(p)) {  // any seg_len a multiple of 16: the factorised readout on the tensor cores
        void *scratch = nullptr;
        const size_t bytes = gen_scratch_bytes(p);
        if (bytes && scratch_alloc(&scratch, bytes, stream) != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_ALLOC;
        }
        FwdArgs a{};
        a.q = q; a.k = k; a.v = v;
        a.u = mode_uses_u(p.mode) ? u : nullptr;
        a.y = y;
        a.states = states;  // NULL: the states are not needed by this path and not formed
        a.BH = p.BH; a.L = L; a.C = seg_len; a.N = p.N; a.mode = p.mode; a.topk = p.topk;
        cudaError_t e = launch_forward_gen(p, a, scratch, stream);
        cudaError_t ef = scratch ? cudaFreeAsync(scratch, stream) : cudaSuccess;
        if (e != cudaSuccess || ef != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_CUDA;
        }
        return MC_OK;
    }

    const ScratchPlan plan = plan_scratch(p, states == nullptr);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, plan.total, stream) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    char *base = static_cast<char *>(scratch);
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.u = mode_uses_u(p.mode) ? u : nullptr;
    a.y = y;
    a.states = states ? states : reinterpret_cast<float *>(base + plan.off_states);
    a.O_on = reinterpret_cast<float *>(base + plan.off_O);
    a.r_on = reinterpret_cast<float *>(base + plan.off_r);
    a.kbar = reinterpret_cast<float *>(base + plan.off_kbar);
    a.BH = p.BH; a.L = L; a.C = seg_len; a.N = p.N; a.mode = p.mode; a.topk = p.topk;

    profile_call_start(stream);
    cudaError_t e = launch_seg_scan_simt(p, a, stream);
    profile_after_kernel(stream, "seg_scan_simt");
    if (e == cudaSuccess) {
        e = launch_readout_simt(p, a, stream);
        profile_after_kernel(stream, "readout_simt");
    }
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

// The forward over given boundaries (host seg_off) whose first nbig segments are whole
// 128-token chunks and whose remaining segments lie in the last L % 128 tokens: the
// state-form tensor-core kernels for the first, the CUDA-core scan and readout for the tail.
int forward_segments_tc(const Problem &p, const void *q, const void *k, const void *v, const void *u,
                        const int32_t *seg_off, int nbig, void *y, float *states, cudaStream_t stream)
{
    const int N = p.N, L = p.L, d = p.d;
    const int ntail = N - nbig;
    const int NC = seg_off[nbig] / 128;  // 128-token chunks of the tensor-core segments
    int tail_max = 0;
    for (int n = nbig; n < N; ++n) tail_max = std::max(tail_max, seg_off[n + 1] - seg_off[n]);
    // one int32 table: boundaries [N + 1], first chunks [nbig], readout tiles [2 NC] (segment,
    // chunk, the segments with more cached states first), then for the tail scan the first
    // piece of every segment [N + 1] and the segment of every piece [ntail]
    std::vector<int32_t> tab(seg_off, seg_off + N + 1);
    const size_t o_cbase = tab.size();
    for (int n = 0; n < nbig; ++n) tab.push_back(seg_off[n] / 128);
    if (tab.size() % 2) tab.push_back(0);  // int2 alignment
    const size_t o_tiles = tab.size();
    for (int n = nbig - 1; n >= 0; --n)
        for (int c = 0; c < (seg_off[n + 1] - seg_off[n]) / 128; ++c) {
            tab.push_back(n);
            tab.push_back(c);
        }
    const size_t o_pieces = tab.size();
    for (int n = 0; n <= N; ++n) tab.push_back(n <= nbig ? 0 : n - nbig);
    const size_t o_pseg = tab.size();
    for (int j = 0; j < ntail; ++j) tab.push_back(nbig + j);
    // The state walk's units: pieces of kStatePiece chunks (a segment's last piece shorter), so that no
    // CTA walks a long segment alone; the pieces before a segment's last get their own states from a
    // first pass (slots), and every piece starts from the sum of the ones before it.  Int4 rows
    // (segment, first chunk, chunks, aux), the longest first.
    constexpr int kStatePiece = 16;
    std::vector<std::array<int32_t, 4>> u1, u2;
    int nslots = 0;
    for (int n = 0; n < nbig; ++n) {
        const int nch = (seg_off[n + 1] - seg_off[n]) / 128;
        const int pl = std::max(kStatePiece, (nch + 255) / 256);  // at most 256 pieces (8-bit count)
        const int np = (nch + pl - 1) / pl;
        for (int q = 0; q < np; ++q) {
            const int len = std::min(pl, nch - q * pl);
            if (q + 1 < np) u1.push_back({n, q * pl, len, nslots + q});
            u2.push_back({n, q * pl, len, (nslots << 8) | q});
        }
        nslots += np - 1;
    }
    std::stable_sort(u2.begin(), u2.end(), [](const auto &x, const auto &y) { return x[2] > y[2]; });
    while (tab.size() % 4) tab.push_back(0);  // int4 alignment
    const size_t o_u1 = tab.size();
    for (const auto &x : u1) tab.insert(tab.end(), x.begin(), x.end());
    const size_t o_u2 = tab.size();
    for (const auto &x : u2) tab.insert(tab.end(), x.begin(), x.end());

    const size_t BH = p.BH;
    const size_t b_tab = round_up(sizeof(int32_t) * tab.size());
    const size_t b_states = states ? 0 : round_up(sizeof(float) * BH * N * d * d);
    const size_t b_kbar = round_up(sizeof(float) * BH * N * d);
    const size_t b_O = ntail ? round_up(sizeof(float) * BH * L * d) : 0;
    const size_t b_r = ntail ? round_up(sizeof(float) * BH * L) : 0;
    const int t_tail = seg_off[nbig];  // the tail's first token
    const size_t b_acc = ntail ? round_up(tail_scratch_bytes(p, t_tail)) : 0;
    const size_t b_tc = tc_segments_scratch_bytes(p, NC, nslots);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, b_tab + b_states + b_kbar + b_O + b_r + b_acc + b_tc, stream) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    char *base = static_cast<char *>(scratch);
    int32_t *dtab = reinterpret_cast<int32_t *>(base);
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.u = mode_uses_u(p.mode) ? u : nullptr;
    a.y = y;
    a.states = states ? states : reinterpret_cast<float *>(base + b_tab);
    a.kbar = reinterpret_cast<float *>(base + b_tab + b_states);
    a.O_on = ntail ? reinterpret_cast<float *>(base + b_tab + b_states + b_kbar) : nullptr;
    a.r_on = ntail ? reinterpret_cast<float *>(base + b_tab + b_states + b_kbar + b_O) : nullptr;
    void *tail_scratch = base + b_tab + b_states + b_kbar + b_O + b_r;
    void *tc_scratch = base + b_tab + b_states + b_kbar + b_O + b_r + b_acc;
    TcSegTables tb{};
    tb.off = dtab;
    tb.cbase = dtab + o_cbase;
    tb.tiles = reinterpret_cast<const int2 *>(dtab + o_tiles);
    tb.Nseg = nbig;
    tb.NC = NC;
    tb.units1 = reinterpret_cast<const int4 *>(dtab + o_u1);
    tb.units2 = reinterpret_cast<const int4 *>(dtab + o_u2);
    tb.n1 = (int)u1.size();
    tb.n2 = (int)u2.size();
    tb.nslots = nslots;
    cudaError_t e = cudaMemcpyAsync(dtab, tab.data(), sizeof(int32_t) * tab.size(), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) {
        profile_call_start(stream);
        e = launch_state_tc_segments(p, a, tb, tc_scratch, stream);
    }
    if (e == cudaSuccess && ntail) {  // the tail's segments on the CUDA cores, one piece each
        FwdArgs t = a;
        t.seg_off = dtab;
        t.seg_pieces = dtab + o_pieces;
        t.piece_seg = dtab + o_pseg;
        t.npieces = ntail;
        t.piece_len = 128;
        t.BH = p.BH; t.L = L; t.C = tail_max; t.N = N; t.mode = p.mode; t.topk = p.topk;
        Problem pt = p;
        pt.C = tail_max;
        e = launch_seg_scan_simt(pt, t, stream);
        profile_after_kernel(stream, "seg_scan_simt");
    }
    if (e == cudaSuccess) e = launch_readout_tc_segments(p, a, tb, tc_scratch, stream);
    if (e == cudaSuccess && ntail) {  // the tail's tokens read every earlier state
        FwdArgs t = a;
        t.seg_off = dtab;
        t.BH = p.BH; t.L = L; t.C = tail_max; t.N = N; t.mode = p.mode; t.topk = p.topk;
        e = launch_tail_readout(p, t, t_tail, tail_scratch, stream);
        profile_after_kernel(stream, "tail_readout_simt");
    }
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

// The forward over given segment boundaries (FFMA kernels; seg_off is host memory).
int forward_segments(const void *q, const void *k, const void *v, const void *u, int B, int H, int L, int d,
                     const int32_t *seg_off, int nseg, int agg_mode, int topk, void *y, float *states, bool bf16,
                     cudaStream_t stream)
{
    if (!seg_off) return MC_ERR_NULL;
    if (nseg < 1 || nseg > L || seg_off[0] != 0 || seg_off[nseg] != L) return MC_ERR_SHAPE;
    int maxlen = 0;
    for (int n = 0; n < nseg; ++n) {
        if (seg_off[n + 1] <= seg_off[n]) return MC_ERR_SHAPE;
        maxlen = seg_off[n + 1] - seg_off[n] > maxlen ? seg_off[n + 1] - seg_off[n] : maxlen;
    }
    int st = check_shape(B, H, L, d, maxlen);
    if (st != MC_OK) return st;
    if ((long long)B * H * nseg * ((maxlen + 63) / 64) >= (1ll << 31) || (long long)B * H * nseg * d * d > (1ll << 40))
        return MC_ERR_SHAPE;
    if (agg_mode < MC_RESIDUAL || agg_mode > MC_MEAN) return MC_ERR_MODE;
    if (!q || !k || !v || !y) return MC_ERR_NULL;
    if (mode_uses_u(agg_mode) && !u) return MC_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(y) || (u && !aligned16(u)) ||
        (states && !aligned16(states)))
        return MC_ERR_ALIGN;
    Problem p{};
    p.B = B; p.H = H; p.L = L; p.d = d; p.C = maxlen;
    p.N = nseg;
    p.BH = B * H;
    p.bf16 = bf16;
    p.mode = agg_mode;
    p.topk = agg_mode == MC_SSC ? topk : 0;
    if (agg_mode == MC_SSC) {
        if (topk < 0) return MC_ERR_TOPK;
        if (topk >= p.N - 1) p.mode = MC_GRM;
        else if (topk > kMaxTopk) return MC_ERR_TOPK;
    }
    st = check_device();
    if (st != MC_OK) return st;
    // Tensor cores for the leading segments that are whole 128-token chunks (start and
    // length multiples of 128) when the rest -- a tail of shorter segments -- fits in the
    // last L % 128 tokens (the logarithmic segmentation of Log-Linear++ is of this kind).
    int nbig = 0;
    while (nbig < nseg && seg_off[nbig] % 128 == 0 && (seg_off[nbig + 1] - seg_off[nbig]) % 128 == 0) ++nbig;
    if (bf16 && (d == 64 || d == 128) && p.N <= 64 && nbig >= 1 && L - seg_off[nbig] < 128 &&
        (p.mode != MC_SSC || p.topk <= 16))
        return forward_segments_tc(p, q, k, v, u, seg_off, nbig, y, states, stream);
    // Segments longer than kPieceLen tokens are scanned in pieces (all at once, then a
    // prefix over each segment's pieces): boundaries, then the first piece of every
    // segment, then the segment of every piece, in one host table.
    std::vector<int32_t> table(seg_off, seg_off + nseg + 1);
    int npieces = 0;
    if (maxlen > kPieceLen) {
        table.resize((size_t)2 * (nseg + 1));
        for (int n = 0; n < nseg; ++n) {
            table[(size_t)nseg + 1 + n] = npieces;
            npieces += (seg_off[n + 1] - seg_off[n] + kPieceLen - 1) / kPieceLen;
        }
        table[(size_t)2 * nseg + 1] = npieces;
        for (int n = 0; n < nseg; ++n)
            for (int i = table[(size_t)nseg + 1 + n]; i < table[(size_t)nseg + 2 + n]; ++i) table.push_back(n);
    }
    const ScratchPlan plan = plan_scratch(p, states == nullptr);
    const size_t off_bytes = round_up(sizeof(int32_t) * table.size());
    const size_t piece_bytes = round_up(sizeof(float) * (size_t)p.BH * npieces * d * d) +
                               round_up(sizeof(float) * (size_t)p.BH * npieces * d);
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, plan.total + off_bytes + piece_bytes, stream) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    char *base = static_cast<char *>(scratch);
    int32_t *doff = reinterpret_cast<int32_t *>(base + plan.total);
    FwdArgs a{};
    if (npieces > 0) {
        a.seg_pieces = doff + nseg + 1;
        a.piece_seg = doff + 2 * (nseg + 1);
        a.npieces = npieces;
        a.piece_len = kPieceLen;
        a.piece_state = reinterpret_cast<float *>(base + plan.total + off_bytes);
        a.piece_ksum = reinterpret_cast<float *>(base + plan.total + off_bytes +
                                                 round_up(sizeof(float) * (size_t)p.BH * npieces * d * d));
    }
    a.q = q; a.k = k; a.v = v;
    a.u = mode_uses_u(p.mode) ? u : nullptr;
    a.y = y;
    a.states = states ? states : reinterpret_cast<float *>(base + plan.off_states);
    a.O_on = reinterpret_cast<float *>(base + plan.off_O);
    a.r_on = reinterpret_cast<float *>(base + plan.off_r);
    a.kbar = reinterpret_cast<float *>(base + plan.off_kbar);
    a.seg_off = doff;
    a.BH = p.BH; a.L = L; a.C = maxlen; a.N = p.N; a.mode = p.mode; a.topk = p.topk;
    cudaError_t e = cudaMemcpyAsync(doff, table.data(), sizeof(int32_t) * table.size(), cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess) {
        profile_call_start(stream);
        e = launch_seg_scan_simt(p, a, stream);
        profile_after_kernel(stream, "seg_scan_simt");
    }
    if (e == cudaSuccess) {
        e = launch_readout_simt(p, a, stream);
        profile_after_kernel(stream, "readout_simt");
    }
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

int backward_common(const void *q, const void *k, const void *v, const void *u, const void *dy, int B, int H, int L,
                    int d, int seg_len, int agg_mode, int topk, void *dq, void *dk, void *dv, void *du, bool bf16,
                    cudaStream_t stream)
{
    int st = check_shape(B, H, L, d, seg_len);
    if (st != MC_OK) return st;
    if (agg_mode < MC_RESIDUAL || agg_mode > MC_MEAN) return MC_ERR_MODE;
    const bool uses_u = mode_uses_u(agg_mode);
    if (!q || !k || !v || !dy || !dq || !dk || !dv) return MC_ERR_NULL;
    if (uses_u && (!u || !du)) return MC_ERR_NULL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(dy) || !aligned16(dq) || !aligned16(dk) ||
        !aligned16(dv) || (u && !aligned16(u)) || (du && !aligned16(du)))
        return MC_ERR_ALIGN;
    Problem p{};
    p.B = B; p.H = H; p.L = L; p.d = d; p.C = seg_len;
    p.N = (L + seg_len - 1) / seg_len;
    p.BH = B * H;
    p.bf16 = bf16;
    p.mode = agg_mode == MC_SOUP ? MC_GRM : agg_mode;  // the same function for a linear memory
    p.topk = agg_mode == MC_SSC ? topk : 0;
    if (agg_mode == MC_SSC) {
        if (topk < 0) return MC_ERR_TOPK;
        if (topk >= p.N - 1) p.mode = MC_GRM;
        else if (topk > kMaxTopk) return MC_ERR_TOPK;
    }
    if (p.mode != MC_SSC) p.topk = 0;
    st = check_device();
    if (st != MC_OK) return st;
    void *scratch = nullptr;
    if (scratch_alloc(&scratch, backward_scratch_bytes(p), stream) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    cudaError_t e = cudaSuccess;
    if (!uses_u && du) e = cudaMemsetAsync(du, 0, (size_t)p.BH * L * d * (bf16 ? 2 : 4), stream);
    if (e == cudaSuccess) e = launch_backward_simt(p, q, k, v, uses_u ? u : nullptr, dy, dq, dk, dv, du, scratch, stream);
    cudaError_t ef = cudaFreeAsync(scratch, stream);
    if (e != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

}  // namespace
}  // namespace mc

extern "C" {

int mc_forward_segments(const void *q, const void *k, const void *v, const void *u, int B, int H, int L, int d,
                        const int32_t *seg_off, int nseg, int agg_mode, int topk, void *y, float *states, int is_bf16,
                        mc_stream_t stream)
{
    return mc::forward_segments(q, k, v, u, B, H, L, d, seg_off, nseg, agg_mode, topk, y, states, is_bf16 != 0,
                                reinterpret_cast<cudaStream_t>(stream));
}

int mc_log_segments(int L, int32_t *seg_off, int cap)
{
    if (L < 1) return MC_ERR_SHAPE;
    if (!seg_off) return MC_ERR_NULL;
    int nseg = 0;
    for (int bit = 30; bit >= 0; --bit) nseg += (L >> bit) & 1;
    if (cap < nseg + 1) return MC_ERR_SHAPE;
    int n = 0;
    seg_off[0] = 0;
    for (int bit = 30; bit >= 0; --bit)
        if ((L >> bit) & 1) {
            seg_off[n + 1] = seg_off[n] + (1 << bit);
            ++n;
        }
    return nseg;
}

int mc_backward(const void *q, const void *k, const void *v, const void *u, const void *dy, int B, int H, int L,
                int d, int seg_len, int agg_mode, int topk, void *dq, void *dk, void *dv, void *du, mc_stream_t stream)
{
    return mc::backward_common(q, k, v, u, dy, B, H, L, d, seg_len, agg_mode, topk, dq, dk, dv, du, true,
                               reinterpret_cast<cudaStream_t>(stream));
}

int mc_backward_f32(const float *q, const float *k, const float *v, const float *u, const float *dy, int B, int H,
                    int L, int d, int seg_len, int agg_mode, int topk, float *dq, float *dk, float *dv, float *du,
                    mc_stream_t stream)
{
    return mc::backward_common(q, k, v, u, dy, B, H, L, d, seg_len, agg_mode, topk, dq, dk, dv, du, false,
                               reinterpret_cast<cudaStream_t>(stream));
}

int mc_forward(const void *q, const void *k, const void *v, const void *u, int B, int H, int L, int d, int seg_len,
               int agg_mode, int topk, void *y, float *states, mc_stream_t stream)
{
    return mc::forward_common(q, k, v, u, B, H, L, d, seg_len, agg_mode, topk, y, states, true,
                              reinterpret_cast<cudaStream_t>(stream));
}

int mc_forward_f32(const float *q, const float *k, const float *v, const float *u, int B, int H, int L, int d,
                   int seg_len, int agg_mode, int topk, float *y, float *states, mc_stream_t stream)
{
    return mc::forward_common(q, k, v, u, B, H, L, d, seg_len, agg_mode, topk, y, states, false,
                              reinterpret_cast<cudaStream_t>(stream));
}

int mc_forward_swla(const void *q, const void *k, const void *v, const void *u, const float *alpha,
                    const float *beta, const float *lam, int B, int H, int L, int d, int seg_len, int agg_mode,
                    int topk, void *y, float *states, mc_stream_t stream)
{
    return mc::forward_common(q, k, v, u, B, H, L, d, seg_len, agg_mode, topk, y, states, true,
                              reinterpret_cast<cudaStream_t>(stream), alpha, beta, lam, true);
}

int mc_decode_step(const void *q, const void *k, const void *v, const void *u, int B, int H, int d, int seg_len,
                   int agg_mode, int topk, int t, float *states, float *kbar, float *online, float *ksum, int n_max,
                   void *y, int is_bf16, mc_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int st = mc::check_shape(B, H, 1, d, seg_len);
    if (st != MC_OK) return st;
    if (t < 0 || n_max < 1 || n_max > mc::kDecMaxN - 1 || t / seg_len >= n_max) return MC_ERR_SHAPE;
    if (agg_mode < MC_RESIDUAL || agg_mode > MC_MEAN) return MC_ERR_MODE;
    if (agg_mode == MC_SSC && topk < 0) return MC_ERR_TOPK;
    if (!q || !k || !v || !y || !states || !kbar || !online || !ksum) return MC_ERR_NULL;
    if (mc::mode_uses_u(agg_mode) && !u) return MC_ERR_NULL;
    if (!mc::aligned16(q) || !mc::aligned16(k) || !mc::aligned16(v) || !mc::aligned16(y) || (u && !mc::aligned16(u)) ||
        !mc::aligned16(states) || !mc::aligned16(kbar) || !mc::aligned16(online) || !mc::aligned16(ksum))
        return MC_ERR_ALIGN;
    st = mc::check_device();
    if (st != MC_OK) return st;
    mc::DecodeArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.u = mc::mode_uses_u(agg_mode) ? u : nullptr;
    a.y = y;
    a.states = states; a.kbar = kbar; a.online = online; a.ksum = ksum;
    a.BH = B * H; a.d = d; a.C = seg_len; a.mode = agg_mode == MC_SOUP ? MC_GRM : agg_mode;
    a.topk = agg_mode == MC_SSC ? topk : 0;
    a.t = t; a.nmax = n_max; a.bf16 = is_bf16 != 0;
    void *gates = nullptr;
    if (mc::scratch_alloc(&gates, sizeof(float) * (size_t)a.BH * mc::kDecGateWords, stream) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    a.gates = static_cast<float *>(gates);
    cudaError_t e = mc::launch_decode_step(a, stream);
    cudaError_t ef = cudaFreeAsync(gates, stream);
    if (e != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

int mc_ssc_select(const void *k, const void *u, int B, int H, int L, int d, int seg_len, int topk, int32_t *idx,
                  int is_bf16, mc_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int st = mc::check_shape(B, H, L, d, seg_len);
    if (st != MC_OK) return st;
    if (!k || !u || !idx) return MC_ERR_NULL;
    if (topk < 1 || topk > mc::kMaxTopk) return MC_ERR_TOPK;
    if (!mc::aligned16(k) || !mc::aligned16(u) || !mc::aligned16(idx)) return MC_ERR_ALIGN;
    st = mc::check_device();
    if (st != MC_OK) return st;
    mc::Problem p{};
    p.B = B; p.H = H; p.L = L; p.d = d; p.C = seg_len;
    p.N = (L + seg_len - 1) / seg_len;
    p.BH = B * H;
    p.bf16 = is_bf16 != 0;
    p.mode = MC_SSC;
    p.topk = topk;
    if (mc::tc_fused_gates(p)) {  // the tensor-core forward's own router, bit for bit
        void *scratch = nullptr;
        if (mc::scratch_alloc(&scratch, mc::tc_select_scratch_bytes(p), stream) != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_ALLOC;
        }
        mc::FwdArgs a{};
        a.k = k; a.u = u; a.sel_out = idx;
        cudaError_t e = mc::launch_ssc_select_tc(p, a, scratch, stream);
        cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e != cudaSuccess || ef != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_CUDA;
        }
        return MC_OK;
    }
    if (mc::gen_supported(p)) {  // the general path's own router, bit for bit
        void *scratch = nullptr;
        if (mc::scratch_alloc(&scratch, mc::gen_select_scratch_bytes(p), stream) != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_ALLOC;
        }
        mc::FwdArgs a{};
        a.k = k; a.u = u; a.sel_out = idx;
        cudaError_t e = mc::launch_ssc_select_gen(p, a, scratch, stream);
        cudaError_t ef = cudaFreeAsync(scratch, stream);
        if (e != cudaSuccess || ef != cudaSuccess) {
            cudaGetLastError();
            return MC_ERR_CUDA;
        }
        return MC_OK;
    }
    float *kbar = nullptr;
    if (mc::scratch_alloc(reinterpret_cast<void **>(&kbar), sizeof(float) * (size_t)p.BH * p.N * d, stream) !=
        cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    mc::FwdArgs a{};
    a.k = k; a.u = u; a.kbar = kbar; a.sel_out = idx;
    a.BH = p.BH; a.L = L; a.C = seg_len; a.N = p.N; a.mode = MC_SSC; a.topk = topk;
    cudaError_t e = mc::launch_kbar_simt(p, a, stream);
    if (e == cudaSuccess) e = mc::launch_ssc_select_simt(p, a, stream);
    cudaError_t ef = cudaFreeAsync(kbar, stream);
    if (e != cudaSuccess || ef != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

int mc_forward_host(const void *q, const void *k, const void *v, const void *u, int B, int H, int L, int d,
                    int seg_len, int agg_mode, int topk, void *y, float *states, int is_bf16, mc_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    int st = mc::check_shape(B, H, L, d, seg_len);
    if (st != MC_OK) return st;
    if (agg_mode < MC_RESIDUAL || agg_mode > MC_MEAN) return MC_ERR_MODE;
    if (!q || !k || !v || !y) return MC_ERR_NULL;
    if (mc::mode_uses_u(agg_mode) && !u) return MC_ERR_NULL;
    st = mc::check_device();
    if (st != MC_OK) return st;
    const size_t elt = is_bf16 ? 2 : 4;
    const size_t n_in = (size_t)B * H * L * d;
    const size_t N = ((size_t)L + seg_len - 1) / seg_len;
    const size_t bytes_in = mc::round_up(n_in * elt);
    const size_t bytes_states = states ? mc::round_up(sizeof(float) * (size_t)B * H * N * d * d) : 0;
    const int nin = u && mc::mode_uses_u(agg_mode) ? 4 : 3;
    void *dmem = nullptr;
    if (mc::scratch_alloc(&dmem, bytes_in * (nin + 1) + bytes_states, stream) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_ALLOC;
    }
    char *p = static_cast<char *>(dmem);
    char *dq = p, *dk = p + bytes_in, *dv = p + 2 * bytes_in;
    char *du = nin == 4 ? p + 3 * bytes_in : nullptr;
    char *dy = p + nin * bytes_in;
    float *ds = states ? reinterpret_cast<float *>(p + (nin + 1) * bytes_in) : nullptr;
    // The (b, h) problems are independent, so the copies are pipelined against the
    // forward over groups of heads: inputs of group c go up on `up` while group c-1
    // runs on `stream` and y of group c-2 comes down on `down`.
    const size_t BH = (size_t)B * H;
    const int groups = BH >= 8 ? 8 : (int)BH;
    const size_t per = (BH + groups - 1) / groups;  // heads per group
    const size_t head_in = (size_t)L * d * elt, head_st = N * (size_t)d * d;
    cudaStream_t up = nullptr, down = nullptr;
    cudaEvent_t ev[2 * 8 + 3] = {};
    const int nev = 2 * groups + 3;
    cudaError_t e = cudaStreamCreateWithFlags(&up, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&down, cudaStreamNonBlocking);
    for (int i = 0; i < nev && e == cudaSuccess; ++i) e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
    cudaEvent_t ev_alloc = ev[2 * groups], ev_up = ev[2 * groups + 1], ev_down = ev[2 * groups + 2];
    int rc = MC_OK;
    if (e == cudaSuccess) e = cudaEventRecord(ev_alloc, stream);  // the device buffers exist from here on
    if (e == cudaSuccess) e = cudaStreamWaitEvent(up, ev_alloc, 0);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(down, ev_alloc, 0);
    for (int c = 0; c < groups && e == cudaSuccess && rc == MC_OK; ++c) {
        const size_t h0 = c * per;
        if (h0 >= BH) break;
        const size_t hc = BH - h0 < per ? BH - h0 : per;
        const size_t off = h0 * head_in, bytes = hc * head_in;
        const char *hq = static_cast<const char *>(q), *hk = static_cast<const char *>(k),
                   *hv = static_cast<const char *>(v), *hu = static_cast<const char *>(u);
        e = cudaMemcpyAsync(dq + off, hq + off, bytes, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dk + off, hk + off, bytes, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaMemcpyAsync(dv + off, hv + off, bytes, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess && du) e = cudaMemcpyAsync(du + off, hu + off, bytes, cudaMemcpyHostToDevice, up);
        if (e == cudaSuccess) e = cudaEventRecord(ev[2 * c], up);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev[2 * c], 0);
        if (e != cudaSuccess) break;
        float *dsc = ds ? ds + h0 * head_st : nullptr;
        rc = is_bf16 ? mc_forward(dq + off, dk + off, dv + off, du ? du + off : nullptr, 1, (int)hc, L, d, seg_len,
                                  agg_mode, topk, dy + off, dsc, stream_)
                     : mc_forward_f32(reinterpret_cast<const float *>(dq + off), reinterpret_cast<const float *>(dk + off),
                                      reinterpret_cast<const float *>(dv + off),
                                      du ? reinterpret_cast<const float *>(du + off) : nullptr, 1, (int)hc, L, d,
                                      seg_len, agg_mode, topk, reinterpret_cast<float *>(dy + off), dsc, stream_);
        if (rc != MC_OK) break;
        e = cudaEventRecord(ev[2 * c + 1], stream);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(down, ev[2 * c + 1], 0);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(static_cast<char *>(y) + off, dy + off, bytes, cudaMemcpyDeviceToHost, down);
        if (e == cudaSuccess && states)
            e = cudaMemcpyAsync(states + h0 * head_st, dsc, sizeof(float) * hc * head_st, cudaMemcpyDeviceToHost, down);
    }
    // everything on `up` and `down` is ordered before the free on `stream`
    cudaError_t ew = cudaSuccess;
    if (up && ev_up && (ew = cudaEventRecord(ev_up, up)) == cudaSuccess) ew = cudaStreamWaitEvent(stream, ev_up, 0);
    if (down && ev_down && ew == cudaSuccess && (ew = cudaEventRecord(ev_down, down)) == cudaSuccess)
        ew = cudaStreamWaitEvent(stream, ev_down, 0);
    if (ew != cudaSuccess) {  // cannot order the free after the copies: wait for them here
        if (up) cudaStreamSynchronize(up);
        if (down) cudaStreamSynchronize(down);
    }
    cudaError_t ef = cudaFreeAsync(dmem, stream);
    cudaError_t es = cudaStreamSynchronize(stream);
    if (up) cudaStreamSynchronize(up);
    if (down) cudaStreamSynchronize(down);
    for (int i = 0; i < nev; ++i)
        if (ev[i]) cudaEventDestroy(ev[i]);
    if (up) cudaStreamDestroy(up);
    if (down) cudaStreamDestroy(down);
    if (rc != MC_OK) return rc;
    if (e != cudaSuccess || ef != cudaSuccess || es != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

int mc_set_readout_form(int form)
{
    if (form != MC_READOUT_AUTO && form != MC_READOUT_FACTORISED) return MC_ERR_MODE;
    return mc::g_readout_form.exchange(form);
}

int mc_trim_scratch(void)
{
    std::lock_guard<std::mutex> lock(mc::g_pool_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    if (mc::g_pools[dev] && cudaMemPoolTrimTo(mc::g_pools[dev], 0) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}

int mc_check_device(mc_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    int was = 0, was_bwd = 0, was_gen = 0, was64 = 0;
    if (mc::take_device_abort(&was) != cudaSuccess || mc::take_bwd_abort(&was_bwd) != cudaSuccess ||
        mc::take_gen_abort(&was_gen) != cudaSuccess || mc::take_tc64_abort(&was64) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return was || was_bwd || was_gen || was64 ? MC_ERR_DEVICE_TIMEOUT : MC_OK;
}

int mc_profile_begin(void *const *events, int capacity)
{
    if (!events || capacity < 1) return MC_ERR_NULL;
    mc::g_prof.events = events;
    mc::g_prof.capacity = capacity;
    mc::g_prof.count = 0;
    for (int j = 0; j < 4096; ++j) mc::g_prof.stage[j] = nullptr;
    return MC_OK;
}

int mc_profile_end(void)
{
    const int n = mc::g_prof.count;
    mc::g_prof.events = nullptr;
    mc::g_prof.capacity = 0;
    return n;
}

const char *mc_profile_stage(int j)
{
    if (j < 0 || j >= 4096) return nullptr;
    return mc::g_prof.stage[j];
}

const char *mc_status_string(int status)
{
    switch (status) {
    case MC_OK: return "ok";
    case MC_ERR_NULL: return "a required pointer is NULL";
    case MC_ERR_SHAPE: return "unsupported shape (B,H,L,seg_len >= 1; d in {16,32,64,128}; sizes within limits)";
    case MC_ERR_MODE: return "agg_mode must be MC_RESIDUAL, MC_GRM, MC_SOUP, MC_SSC or MC_MEAN";
    case MC_ERR_TOPK: return "SSC topk out of range (0..64, or >= N-1 for all segments)";
    case MC_ERR_ALLOC: return "stream-ordered scratch allocation failed";
    case MC_ERR_CUDA: return "a CUDA call or kernel launch failed";
    case MC_ERR_DEVICE_TIMEOUT: return "a bounded device-side wait timed out";
    case MC_ERR_ALIGN: return "every pointer must be 16-byte aligned";
    case MC_ERR_DEVICE: return "the current device is not a compute capability 10.3 (sm_103a) GPU";
    case MC_ERR_SCRATCH: return "problem too large for mc_forward_noalloc's 64 MiB static scratch (use mc_forward)";
    default: return "unknown status";
    }
}

}  // extern "C"
