// mc_noalloc.cu -- mc_forward_noalloc: the bf16 forward (the FFMA segment-scan
// and readout kernels) with its scratch in one fixed, library-owned device
// buffer instead of the stream-ordered allocator.
//
// Who needs it: callers that may not allocate device memory once they are
// running.  An inference-engine plugin is typically handed its streams and
// buffers by the host framework, which owns all device memory and forbids
// allocation inside its execute call; a latency-critical serving loop cannot
// accept an allocator call (or an out-of-memory failure) in the middle of a
// request; a process that reserved nearly all device memory up front has none
// left for a pool.  For them the scratch lives in a file-scope __device__
// array of kNoAllocScratchBytes (64 MiB) that every GPU which loads this
// library holds until the process exits.  The caller still provides q, k, v, u,
// y and (optionally) states.
#include "mc_internal.cuh"

namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;

// Host code must not use this name as an address: on the host it is only a
// stand-in for the symbol.  Its device address is looked up, with the device
// current, on each call below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's device address for the current device.  Looked up on every call
// (a symbol lookup, no allocation) rather than cached, so that a device reset or
// a rebuilt primary context between calls never leaves a stale address behind.
// The first lookup on a device may load the library's device code there.
int scratch_for_current_device(void **out)
{
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    *out = p;
    return MC_OK;
}

size_t pad256(size_t x) { return (x + 255) & ~(size_t)255; }
bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" int mc_forward_noalloc(const void *q, const void *k, const void *v, const void *u, int B, int H, int L,
                                  int d, int seg_len, int agg_mode, int topk, void *y, float *states,
                                  mc_stream_t stream_)
{
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
    if (B < 1 || H < 1 || L < 1 || seg_len < 1 || (d != 16 && d != 32 && d != 64 && d != 128)) return MC_ERR_SHAPE;
    const long long BH = (long long)B * H;
    const long long N = ((long long)L + seg_len - 1) / seg_len;
    if (BH > (1ll << 24) || BH * L * d > (1ll << 40) || BH * N * d * d > (1ll << 40) ||
        BH * N * ((seg_len + 63) / 64) >= (1ll << 31))
        return MC_ERR_SHAPE;
    if (agg_mode < MC_RESIDUAL || agg_mode > MC_MEAN) return MC_ERR_MODE;
    if (!q || !k || !v || !y) return MC_ERR_NULL;
    if (mc::mode_uses_u(agg_mode) && !u) return MC_ERR_NULL;
    if (!al16(q) || !al16(k) || !al16(v) || !al16(y) || (u && !al16(u)) || (states && !al16(states)))
        return MC_ERR_ALIGN;

    mc::Problem p{};
    p.B = B; p.H = H; p.L = L; p.d = d; p.C = seg_len;
    p.N = (int)N;
    p.BH = (int)BH;
    p.bf16 = true;
    p.mode = agg_mode;
    p.topk = agg_mode == MC_SSC ? topk : 0;
    if (agg_mode == MC_SSC) {
        if (topk < 0) return MC_ERR_TOPK;
        if (topk >= p.N - 1) p.mode = MC_GRM;  // every cached segment selected: GRM exactly
        else if (topk > mc::kMaxTopk) return MC_ERR_TOPK;
    }

    // Scratch layout inside the static array (each piece 256-byte aligned).
    const size_t b_states = states ? 0 : pad256(sizeof(float) * (size_t)BH * N * d * d);
    const size_t b_O = pad256(sizeof(float) * (size_t)BH * L * d);
    const size_t b_r = pad256(sizeof(float) * (size_t)BH * L);
    const size_t b_kbar = pad256(sizeof(float) * (size_t)BH * N * d);
    if (b_states + b_O + b_r + b_kbar > kNoAllocScratchBytes) return MC_ERR_SCRATCH;

    int major = 0, minor = 0, dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return MC_ERR_DEVICE;

    void *scratch = nullptr;
    const int st = scratch_for_current_device(&scratch);
    if (st != MC_OK) return st;
    char *base = static_cast<char *>(scratch);

    // Every scratch element is written by the segment scan before the readout
    // reads it, so nothing left by an earlier call needs clearing.
    mc::FwdArgs a{};
    a.q = q; a.k = k; a.v = v;
    a.u = mc::mode_uses_u(p.mode) ? u : nullptr;
    a.y = y;
    a.states = states ? states : reinterpret_cast<float *>(base);
    a.O_on = reinterpret_cast<float *>(base + b_states);
    a.r_on = reinterpret_cast<float *>(base + b_states + b_O);
    a.kbar = reinterpret_cast<float *>(base + b_states + b_O + b_r);
    a.BH = p.BH; a.L = L; a.C = seg_len; a.N = p.N; a.mode = p.mode; a.topk = p.topk;

    cudaError_t e = mc::launch_seg_scan_simt(p, a, stream);
    if (e == cudaSuccess) e = mc::launch_readout_simt(p, a, stream);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return MC_ERR_CUDA;
    }
    return MC_OK;
}
