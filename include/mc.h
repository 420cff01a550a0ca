/*
 * mc.h -- C ABI of the Memory Caching (MC) forward pass over a linear
 * matrix-valued memory, for one NVIDIA GB300 (sm_103a).
 *
 * The method (pages cited by title, section and equation):
 *   [MC-ja]  "メモリキャッシング：メモリ容量が増大する RNN" (Memory Caching:
 *            RNNs with growing memory; news.neo-ai.one/ja/article/2519)
 *   [MC-sum] "给 RNN 装上“会增长的记忆”：解读 Google 的 Memory Caching"
 *            (gitcode.csdn.net/6a26b456662f9a54cb7b57bd.html)
 *
 * Per (batch b, head h) the length-L sequence is cut into N = ceil(L/seg_len)
 * segments of seg_len tokens (the last one may be shorter).  Each segment is
 * compressed from a zero memory with M <- M + v_t k_t^T ([MC-ja §3 eq. 4b]) and
 * its final d x d state is cached.  Token t of segment s reads the online memory
 * M_t^(s) (after its own update) and every cached memory at q_t, and combines
 * them with one of five aggregations:
 *   MC_RESIDUAL  y_t = M_t^(s) q_t + sum_{i<s} M^(i) q_t                [MC-ja §3.1 eq. 7]
 *   MC_GRM       y_t = g_{t,s} M_t^(s) q_t + sum_{i<s} g_{t,i} M^(i) q_t,
 *                g_t = softmax_i <u_t, mean of segment i's keys>, the current
 *                segment pooled over its keys up to t                  [MC-ja §3.1 eq. 9-10]
 *   MC_SOUP      y_t = (g_{t,s} M_t^(s) + sum_{i<s} g_{t,i} M^(i)) q_t  [MC-sum §3.3]
 *                (equal to GRM for a linear memory, and computed as GRM)
 *   MC_SSC       R_t = the topk largest <u_t, pool_i>, i<s (fp32 scores, equal
 *                scores to the lower i); softmax over R_t and the online score;
 *                y_t = g_{t,s} M_t^(s) q_t + sum_{i in R_t} g_{t,i} M^(i) q_t   [MC-sum §3.4]
 *   MC_MEAN      y_t = (M_t^(s) q_t + sum_{i<s} M^(i) q_t) / (s + 1): memory caching
 *                added after training, an average over the memories with no
 *                learned weights (u is not read and may be NULL) [MC-ja, variants
 *                appendix after eq. 35, "memory caching as post-training"]; equal to
 *                GRM with u = 0
 * There is no 1/Z normaliser and no softmax temperature.
 *
 * Conventions for every entry point:
 *   - Tensors are dense and row-major: q, k, v, u, y are [B][H][L][d];
 *     states are [B][H][N][d][d] with states[..][n][a][c] = sum v[a] k[c]
 *     over segment n (row = value dimension, column = key dimension).
 *   - Pointers are DEVICE pointers (except mc_forward_host), allocated and owned
 *     by the caller; the library keeps no reference after the call returns.
 *     Every pointer must be 16-byte aligned.
 *   - Work is enqueued on `stream` (any stream, NULL = the legacy default
 *     stream) and the call returns without synchronising.  Scratch is taken from
 *     a library-owned stream-ordered memory pool of the current device and freed
 *     on the same stream; the pool keeps freed blocks for later calls until
 *     mc_trim_scratch().  Calls on different streams are independent.
 *   - d must be 16, 32, 64 or 128.  B, H, L, seg_len >= 1.
 *   - The kernels are chosen per shape.  bf16 inputs with d = 64 or 128 run on the
 *     tensor cores: the cached readout in the state form (every cached state read
 *     once per 128-token tile, a C x d by d x (N d) product) when seg_len is a
 *     multiple of 128, L a multiple of seg_len and N <= 64; otherwise, when seg_len
 *     is a multiple of 16 (N <= 512 for the routed aggregations), in the factorised
 *     form y_t = sum_{j <= t} g_{t, seg(j)} v_j (k_j . q_t), which costs 4 d t per
 *     token instead of 2 d^2 (N - 1) and so wins for segments shorter than d / 2
 *     ([MC-sum §2.2]: the read is O(N) per token).  Everything else (fp32 inputs,
 *     d = 16 or 32, other segment lengths) runs on CUDA-core kernels.
 *   - Return value: MC_OK (0) or a negative MC_ERR_* code (shape is checked
 *     first, then the mode, then pointers).  On an argument
 *     error nothing is enqueued.  On MC_ERR_CUDA the contents of y and states
 *     are undefined; work already enqueued finishes on the stream.
 */
#ifndef MC_H_
#define MC_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t / CUstream, declared here so C callers need no CUDA headers. */
typedef struct CUstream_st *mc_stream_t;

typedef enum {
    MC_RESIDUAL = 0,
    MC_GRM = 1,
    MC_SOUP = 2,
    MC_SSC = 3,
    MC_MEAN = 4
} mc_agg_mode;

enum {
    MC_OK = 0,
    MC_ERR_NULL = -1,           /* a required pointer is NULL */
    MC_ERR_SHAPE = -2,          /* B,H,L,seg_len < 1, d not in {16,32,64,128}, or sizes overflow */
    MC_ERR_MODE = -3,           /* agg_mode not one of mc_agg_mode */
    MC_ERR_TOPK = -4,           /* SSC with topk < 0, or 64 < topk < N-1 */
    MC_ERR_ALLOC = -5,          /* stream-ordered scratch allocation failed */
    MC_ERR_CUDA = -6,           /* a CUDA runtime call or kernel launch failed */
    MC_ERR_DEVICE_TIMEOUT = -7, /* a bounded device-side wait gave up */
    MC_ERR_ALIGN = -8,          /* a pointer is not 16-byte aligned */
    MC_ERR_DEVICE = -9,         /* the current device is not a compute-capability 10.3 GPU */
    MC_ERR_SCRATCH = -10        /* mc_forward_noalloc: the problem needs more than its 64 MiB static scratch */
};

/*
 * mc_forward -- MC forward, bf16 inputs and output, fp32 state and accumulation.
 *   q, k, v, u : bf16 [B][H][L][d], read only.  u may be NULL for MC_RESIDUAL and MC_MEAN.
 *   seg_len    : constant segment length C; N = ceil(L / C).
 *   agg_mode   : an mc_agg_mode value.
 *   topk       : cached segments each token selects (MC_SSC only; ignored otherwise).
 *                0 keeps only the online memory; topk >= N-1 selects every cached one.
 *   y          : bf16 [B][H][L][d], written.
 *   states     : fp32 [B][H][N][d][d], written with every segment's final state
 *                (the cache, [MC-ja §3 after eq. 4b]); may be NULL, then the
 *                states live in scratch only.
 *   stream     : CUDA stream to enqueue on.
 */
int mc_forward(const void *q, const void *k, const void *v, const void *u,
               int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
               void *y, float *states, mc_stream_t stream);

/* mc_forward_f32 -- identical contract with fp32 q, k, v, u and y (fp32 arithmetic throughout). */
int mc_forward_f32(const float *q, const float *k, const float *v, const float *u,
                   int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
                   float *y, float *states, mc_stream_t stream);

/*
 * mc_forward_swla -- memory caching over sliding-window linear attention with a
 * window of c = 2 ([MC-ja §3.1 eq. 28-29]): inside a segment the memory follows
 *     M_t = alpha_t M_{t-1} + beta_t v_{t-1} k_{t-1}^T + lambda_t v_t k_t^T
 * from an empty memory at the segment's first token (whose beta term, which would
 * reach into the previous segment, is absent); the cached states, gates and
 * aggregation are those of mc_forward.  GRM and Soup coincide for this linear
 * memory.
 *   alpha, beta, lam : fp32 [B][H][L], device, 16-byte aligned; alpha is a decay
 *                      in (0, 1] (values are floored at 1e-30 before their log).
 *   Other arguments as mc_forward (bf16).
 *   Runs on the tensor-core path only: d in {64, 128}, seg_len a multiple of 128,
 *   L a multiple of seg_len, N <= 64, SSC with topk <= 16 (or >= N-1); other
 *   shapes return MC_ERR_SHAPE.  A NULL scalar array returns MC_ERR_NULL.
 */
int mc_forward_swla(const void *q, const void *k, const void *v, const void *u,
                    const float *alpha, const float *beta, const float *lam,
                    int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
                    void *y, float *states, mc_stream_t stream);

/*
 * mc_forward_segments -- the forward with given segment boundaries instead of a
 * constant segment length: segment n is tokens [seg_off[n], seg_off[n+1]), the
 * same for every (b, h).  With the logarithmic segmentation of mc_log_segments and
 * MC_GRM this is the Log-Linear++ variant ([MC-ja] variants appendix; [MC-sum]
 * §4.2: segments of power-of-two lengths, N <= log2 L + 1).
 *   seg_off : HOST int32 [nseg + 1], 0 = seg_off[0] < seg_off[1] < ... < seg_off[nseg] = L;
 *             read during the call only.
 *   states  : fp32 [B][H][nseg][d][d] or NULL.
 *   is_bf16 : q, k, v, u, y are bf16 if non-zero, fp32 otherwise.
 *   Other arguments as mc_forward.  MC_ERR_SHAPE for boundaries that do not rise
 *   strictly from 0 to L.
 *   Kernels: with bf16 inputs, d in {64, 128}, nseg <= 64 (SSC: topk <= 16), when the
 *   leading segments start and end on multiples of 128 tokens and the remaining
 *   segments lie in the last L mod 128 tokens (the logarithmic segmentation is of this
 *   kind), the leading segments run on the tensor cores (the state form over tables
 *   of offsets; segments longer than 2048 tokens in pieces whose own states are
 *   formed first) and the short tail on the CUDA cores; every other case runs on the
 *   CUDA-core kernels.  The tensor-core path reads bf16 operand images of the states,
 *   as mc_forward does.
 */
int mc_forward_segments(const void *q, const void *k, const void *v, const void *u,
                        int B, int H, int L, int d, const int32_t *seg_off, int nseg,
                        int agg_mode, int topk, void *y, float *states, int is_bf16, mc_stream_t stream);

/*
 * mc_log_segments -- the logarithmic segmentation of a length-L sequence ([MC-sum]
 * §4.2): one segment per set bit of L, that power of two long, the longest first
 * (37 -> 32, 4, 1).  Writes the boundaries [0, ..., L] to seg_off (host, cap
 * entries) and returns the number of segments, or MC_ERR_SHAPE (L < 1, or cap too
 * small) / MC_ERR_NULL.  Host only; touches no device.
 */
int mc_log_segments(int L, int32_t *seg_off, int cap);

/*
 * mc_backward -- gradients of the forward over the plain linear memory (the
 * update M <- M + v k^T): for an upstream gradient dy of y, the gradients of
 * <y, dy> with respect to q, k, v and u.  They follow the forward's steps by the
 * chain rule: the gates' softmax ([MC-ja §3.1 eq. 9-10]), the pooled keys of the
 * scores, the reads of the online and cached memories ([MC-ja §3 eq. 4b-5]) and,
 * through the cached states M^(i) = sum v k^T, every token of a cached segment.
 * The SSC selection ([MC-sum §3.4]) is piecewise constant and passes no
 * gradient; Soup takes GRM's (the same function for a linear memory).
 *   q, k, v, u, dy : bf16 [B][H][L][d], read only (u may be NULL for MC_RESIDUAL
 *                    and MC_MEAN).
 *   dq, dk, dv, du : bf16 [B][H][L][d], written (fp32 accumulation).  du may be
 *                    NULL for MC_RESIDUAL and MC_MEAN (it is zero there); if
 *                    given it is zeroed.
 *   Other arguments and errors as mc_forward.  The call recomputes the forward's
 *   segment states in scratch (about (2 N d^2 + 2 L d + 6 L) floats per (b, h)).
 */
int mc_backward(const void *q, const void *k, const void *v, const void *u, const void *dy,
                int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
                void *dq, void *dk, void *dv, void *du, mc_stream_t stream);

/* mc_backward_f32 -- identical contract with fp32 inputs and gradients. */
int mc_backward_f32(const float *q, const float *k, const float *v, const float *u, const float *dy,
                    int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
                    float *dq, float *dk, float *dv, float *du, mc_stream_t stream);

/*
 * mc_decode_step -- one recurrent decoding step: the token at position t of each
 * of the B*H sequences (all at the same position) updates and reads the memory
 * caches, exactly as mc_forward treats token t ([MC-ja §3 eq. 4b-5, §3.1 eq.
 * 7-10]; Soup is read as GRM, identical for this linear memory).  Run for
 * t = 0, 1, 2, ... from caches whose contents are ignored at t = 0, it
 * reproduces mc_forward's y token by token and leaves every completed
 * segment's state in `states`.
 *   q, k, v, u : the new token, [B][H][d], bf16 if is_bf16 != 0 else fp32 (u may
 *                be NULL for Residual).  y: [B][H][d], written, same dtype.
 *   t          : the token's position; segment s = t / seg_len.
 *   states     : fp32 [B][H][n_max][d][d], cached segment states M^(i), i < s,
 *                read; at the segment's last token (t % seg_len == seg_len - 1)
 *                M^(s) is written to slot s.
 *   kbar       : fp32 [B][H][n_max][d], cached key means, same rule.
 *   online     : fp32 [B][H][d][d], the current segment's memory (in/out).
 *   ksum       : fp32 [B][H][d], the current segment's key sum (in/out).
 *   n_max      : capacity of the caches in segments, 1..64; t / seg_len < n_max.
 *   SSC ranks fp32 scores <u, kbar_i> (equal scores: lower index first).
 *   Errors as mc_forward; MC_ERR_SHAPE also for t < 0 or a full cache.  The
 *   call is asynchronous on `stream`; it allocates a few bytes of scratch
 *   per head from the library's pool.
 */
int mc_decode_step(const void *q, const void *k, const void *v, const void *u,
                   int B, int H, int d, int seg_len, int agg_mode, int topk, int t,
                   float *states, float *kbar, float *online, float *ksum, int n_max,
                   void *y, int is_bf16, mc_stream_t stream);

/*
 * mc_ssc_select -- the SSC router alone ([MC-sum §3.4]), for inspection and tests.
 *   k, u     : [B][H][L][d], bf16 if is_bf16 != 0 else fp32, device.
 *   idx      : int32 [B][H][L][topk], written: for token t of segment s, the
 *              selected cached segments (indices < s) in rank order -- highest
 *              fp32 score first, equal scores lower index first -- padded with -1
 *              when s < topk.  The selection is the one mc_forward /
 *              mc_forward_f32 use for MC_SSC on the same inputs.
 *   topk     : 1..64.
 */
int mc_ssc_select(const void *k, const void *u, int B, int H, int L, int d, int seg_len,
                  int topk, int32_t *idx, int is_bf16, mc_stream_t stream);

/*
 * mc_forward_host -- mc_forward / mc_forward_f32 on HOST buffers (end-to-end use).
 *   Same arguments, but q, k, v, u, y and states (optional) are host pointers
 *   (pinned memory gives asynchronous copies).  The call copies the inputs to
 *   device memory it allocates on `stream`, runs the forward, copies y (and the
 *   states when non-NULL) back, frees the device memory and synchronises
 *   `stream` before returning.  is_bf16 selects the element type of q,k,v,u,y.
 */
int mc_forward_host(const void *q, const void *k, const void *v, const void *u,
                    int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
                    void *y, float *states, int is_bf16, mc_stream_t stream);

/*
 * mc_forward_noalloc -- mc_forward without any device allocation.  (The paper
 * has no counterpart: this is a deployment variant of the same forward.)
 *   For callers that cannot allocate device memory while they run -- e.g. an
 *   engine plugin whose host framework owns all device memory and forbids
 *   allocation inside its execute call, or a serving loop that must not risk an
 *   allocator call or an out-of-memory error mid-request.  Same arguments,
 *   layouts and results as mc_forward (it runs the CUDA-core kernels); the
 *   caller still provides q, k, v, u, y and, optionally, states.
 *   Scratch comes from one static device array of 64 MiB inside the library,
 *   held by every GPU that loads the library until the process exits.  It must
 *   hold O_on (B*H*L*d fp32), the online scores (B*H*L fp32), the key means
 *   (B*H*N*d fp32) and, when states is NULL, the states (B*H*N*d*d fp32), each
 *   rounded up to 256 bytes; larger problems return MC_ERR_SCRATCH and enqueue
 *   nothing.  The call allocates and frees nothing.
 *   Every call looks up the array's device address on the current device (no
 *   allocation), so a device reset between calls is harmless.  The first call on
 *   a device may load the library's device code there: make that first call
 *   before any stream capture.
 *   All calls share the one array: calls whose work overlaps on the GPU (other
 *   streams, other host threads) race on it and must be serialised by the
 *   caller.  Every scratch element is rewritten before it is read, so nothing
 *   left by an earlier call needs clearing.
 */
int mc_forward_noalloc(const void *q, const void *k, const void *v, const void *u,
                       int B, int H, int L, int d, int seg_len, int agg_mode, int topk,
                       void *y, float *states, mc_stream_t stream);

/*
 * mc_set_readout_form -- how later forward calls in this process choose the form
 *   of the cached readout on the tensor cores (a switch for measurement; the
 *   library does not need it):
 *     MC_READOUT_AUTO        (0) per shape, as described at the top (the default);
 *     MC_READOUT_FACTORISED  (1) the factorised form wherever it applies, also on
 *                                shapes the state form would take.
 *   Both give the same y up to rounding.  Returns the previous setting (>= 0), or
 *   MC_ERR_MODE for an unknown form.  The setting is process-wide; change it only
 *   while no forward call is being made on another thread.
 */
enum { MC_READOUT_AUTO = 0, MC_READOUT_FACTORISED = 1 };
int mc_set_readout_form(int form);

/*
 * mc_trim_scratch -- return the scratch memory cached by the library's pool on
 *   the current device to the driver (blocks still in use by enqueued work are
 *   kept).  Returns MC_OK or MC_ERR_CUDA.
 */
int mc_trim_scratch(void);

/*
 * mc_check_device -- synchronise `stream`, then report whether any tensor-core
 *   kernel of this library gave up on a bounded device-side wait since the last
 *   check (and clear that record).  Every wait inside the kernels is bounded; a
 *   kernel that gives up abandons its tile and exits cleanly, so the context
 *   stays usable but the outputs of that call are undefined.
 *   Returns MC_OK, MC_ERR_DEVICE_TIMEOUT, or MC_ERR_CUDA if the stream reports
 *   an error.
 */
int mc_check_device(mc_stream_t stream);

/*
 * Kernel-boundary timing, for benchmarks and profilers.
 *   mc_profile_begin(events, capacity): `events` is a caller-owned array of
 *     `capacity` cudaEvent_t handles (created by the caller).  From now on every
 *     forward call records, on its own stream, one event before its first
 *     kernel and one after each kernel it launches, filling the array in order;
 *     recording stops silently when the array is full.
 *   mc_profile_end(): stops recording and returns how many events were recorded.
 *   mc_profile_stage(j): name of the kernel that ran between recorded event j
 *     and event j+1 (NULL where j+1 opened a new call, or j is out of range).
 * Process-wide state, not thread-safe; forward calls without an active
 * profile record nothing.  Returns MC_OK / MC_ERR_NULL.
 */
int mc_profile_begin(void *const *events, int capacity);
int mc_profile_end(void);
const char *mc_profile_stage(int j);

/* Human-readable text for a status code (static storage, never NULL). */
const char *mc_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* MC_H_ */
