/*
 * gdn.h - C ABI of the GB300 (sm_103a) gated delta-rule state update library
 * (libgdn_gb300.so).
 *
 * The operation.  For every sequence b and value head vi, with key head
 * hh = vi / (vh / kh) and a row-major [kd][vd] fp32 state S, one token does
 *     alpha = exp(g);  S = alpha * S;
 *     kv = S^T k;  tmp = (v - kv) * beta;  S = S + k tmp^T;
 *     o = S^T q                                  (with the updated S)
 * as defined in "Kestrel_VLLM - 24 · GDN linear attention to GPU"
 * (wsisp.com/helps/119760.html), section 4 (the delta-recurrence kernel) and
 * figure 1 step 5; the register-resident kernel of "Kestrel_VLLM - 27 ·
 * register-resident & fused launch" (juejin.cn/post/7703369445846777871),
 * section 3.1, computes the same thing.  M tokens are M serial updates
 * ("Kestrel_VLLM - 34 · batched M rows", juejin.cn/post/7704936491831377954,
 * section 3.6), and mark / rollback snapshot and restore the state
 * (same article, section 3.7).
 *
 * Conventions shared by every call
 *   - Shapes: kd == vd == 128, vh % kh == 0, B >= 0 (B == 0 is a no-op that
 *     returns GDN_OK).  Anything else returns GDN_ESHAPE.
 *   - Layouts: contiguous row-major fp32 DEVICE arrays
 *         S          [B][vh][kd][vd]
 *         q, k       [B][T][kh][kd]     (T = 1 for gdn_step, M, or T)
 *         v, o       [B][T][vh][vd]
 *         g, beta    [B][T][vh]         (g is the log-domain decay, alpha = exp(g))
 *         ckpt       [M][B][vh][kd][vd]
 *     Every array pointer must be 16-byte aligned (GDN_EALIGN otherwise) and
 *     point to device (or managed) memory of the current device (GDN_EPTR
 *     otherwise).  NULL where a buffer is required gives GDN_EINVAL.
 *     Exception: the token inputs and outputs of gdn_step, gdn_step_m and
 *     gdn_layer_step_m's o may also be page-locked host memory mapped at
 *     the same address on the device (cudaHostAlloc / cudaMallocHost under
 *     unified addressing); the kernel then reads and writes it over the
 *     host link.  On a GB300 a 64 x 48-head decode step writing o to host
 *     memory this way took the same time as with device memory, while
 *     reading q, k, v, g, beta from host memory added ~13 us of latency;
 *     copy the inputs in, write o out directly.  Pageable memory is refused
 *     (GDN_EPTR).
 *   - Ownership: the caller allocates and frees everything.  The library
 *     never allocates device memory and never synchronises; every call only
 *     enqueues work on `stream` and returns.  (The one exception is the
 *     static scratch array of gdn_layer_step_m_noalloc, created with the
 *     library's device code.)
 *   - Aliasing: outputs must not overlap inputs or each other, except where
 *     a call states otherwise (GDN_EALIAS).
 *   - Errors: arguments are validated on the host before anything is
 *     enqueued; on any error nothing is launched.  A failed kernel launch
 *     returns GDN_ECUDA.  Asynchronous faults surface on the stream as
 *     usual CUDA errors.
 *   - Precision: fp32 throughout (expf from CUDA's math library, fused
 *     multiply-adds, fixed reduction trees), except the chunked prefill
 *     modes, whose tensor-core products take bf16 operands (see
 *     gdn_prefill).  Results are deterministic: the same inputs and shape
 *     give the same bits on every call.
 */
#ifndef GDN_GB300_H
#define GDN_GB300_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream.  NULL is the legacy default
 * stream. */
typedef struct CUstream_st *gdn_stream_t;

typedef struct gdn_shape {
    int B;   /* sequences, each with its own vh states                    */
    int kh;  /* key heads (q and k are per key head)                      */
    int vh;  /* value heads; value head vi reads key head vi / (vh / kh)  */
    int kd;  /* key dimension: must be 128                                */
    int vd;  /* value dimension: must be 128                              */
} gdn_shape;

enum {
    GDN_OK = 0,
    GDN_EINVAL = -1, /* NULL pointer or meaningless argument               */
    GDN_ESHAPE = -2, /* shape not supported (kd, vd, vh % kh, negative)    */
    GDN_EALIGN = -3, /* a pointer is not 16-byte aligned                   */
    GDN_ECUDA = -4,  /* a CUDA runtime call or kernel launch failed        */
    GDN_ERANGE = -5, /* M, m, T, chunk or workspace size out of range      */
    GDN_EPTR = -6,   /* a pointer is not device memory of this device      */
    GDN_EALIAS = -7, /* buffers overlap where they must not                */
    GDN_ESCRATCH = -8 /* request larger than the static scratch of
                         gdn_layer_step_m_noalloc                          */
};

/* Largest M / T accepted by one call. */
#define GDN_MAX_TOKENS (1 << 20)

/* Prefill precisions. */
enum {
    GDN_PREC_FP32 = 0,   /* token-serial fp32: bit-identical to T gdn_step   */
    GDN_PREC_BF16X3 = 1, /* chunked, tensor cores, operands split into bf16
                            hi + lo, 3 products per term, fp32 accumulation:
                            relative error ~1e-5                             */
    GDN_PREC_BF16 = 2    /* chunked, tensor cores, operands rounded to bf16,
                            one product per term: relative error ~1e-2       */
};

/*
 * gdn_step - one token for all B * vh heads, state updated in place.
 * The operation is the delta-recurrence kernel of "24 · GDN linear
 * attention to GPU", section 4 (figure 1, step 5): decay, read-out S^T k,
 * delta, rank-1 update and o from the updated state, with its argument set
 * (S, q, k, v, g, beta, o and the head counts), extended by B sequences.
 *   S     [B][vh][kd][vd]  in/out
 *   q, k  [B][kh][kd]      in
 *   v     [B][vh][vd]      in
 *   g     [B][vh]          in, log-domain decay (alpha = exp(g))
 *   beta  [B][vh]          in
 *   o     [B][vh][vd]      out
 * Bit-identical to gdn_step_m with M = 1 and S_out == S_in (it is that
 * call).  Algorithmic HBM traffic: 2 * B*vh*kd*vd*4 bytes of state plus the
 * token inputs and o.
 */
int gdn_step(const gdn_shape *shape, float *S, const float *q, const float *k,
             const float *v, const float *g, const float *beta, float *o,
             gdn_stream_t stream);

/*
 * gdn_step_m - M tokens in one launch; the state is read once, kept on chip
 * across the M serial updates, and written once.  "34 · batched M rows",
 * section 3.6, defines the M tokens of a verify launch as M serial state
 * updates (no chunked scan); the per-token checkpoints serve the rollback of
 * its section 3.7 to any accepted count.
 *   S_in   [B][vh][kd][vd]      in  (state before token 0)
 *   S_out  [B][vh][kd][vd]      out (state after token M-1); may equal S_in
 *                               exactly (in place), no other overlap
 *   ckpt   [M][B][vh][kd][vd]   out, or NULL: ckpt[m] = state after token m
 *   q, k   [B][M][kh][kd]       in
 *   v      [B][M][vh][vd]       in
 *   g,beta [B][M][vh]           in
 *   o      [B][M][vh][vd]       out
 * 1 <= M <= GDN_MAX_TOKENS (GDN_ERANGE otherwise).  Output m is
 * bit-identical to the m-th of M successive gdn_step calls on the same
 * inputs, and ckpt[m] to the state after it.
 * Stream order: a launch of at most 16 tokens without checkpoints whose
 * grid fills the GPU starts as a programmatic dependent of the kernel
 * before it on the stream.  Its CTAs may become resident before that
 * kernel ends, but they read and write no memory until it has completed,
 * so the call sees every earlier write on the stream, as an ordinary launch
 * would.  The same holds for gdn_step, gdn_layer_step_m and
 * gdn_layer_prologue_m.
 */
int gdn_step_m(const gdn_shape *shape, int M, const float *S_in, float *S_out,
               float *ckpt, const float *q, const float *k, const float *v,
               const float *g, const float *beta, float *o,
               gdn_stream_t stream);

/*
 * gdn_mark - snapshot the state: snap = S (B*vh*kd*vd floats, device to
 * device, on `stream`).  snap must not overlap S.  The one-shot
 * device-to-device clone of the recurrent state that "34 · batched M rows",
 * section 3.7, takes before a speculative launch.
 */
int gdn_mark(const gdn_shape *shape, const float *S, float *snap,
             gdn_stream_t stream);

/*
 * gdn_rollback - restore the state after m of the M tokens of a gdn_step_m
 * call ("34 · batched M rows", section 3.7: roll the state back to the
 * accepted prefix; the article restores its one snapshot, and the
 * per-token checkpoints extend that to any m):  m == 0 copies snap (the state before the call, from gdn_mark or the
 * S_in of an out-of-place call) into S;  1 <= m <= M copies ckpt[m-1].
 * snap may be NULL when m > 0; ckpt may be NULL when m == 0.  0 <= m <= M
 * (GDN_ERANGE otherwise).  The copy is bit-exact.  Sources must not overlap
 * S.
 */
int gdn_rollback(const gdn_shape *shape, int M, int m, const float *snap,
                 const float *ckpt, float *S, gdn_stream_t stream);

/*
 * gdn_rollback_seq - per-sequence rollback: sequence b restores the state
 * after m_dev[b] tokens (same rule as gdn_rollback, "34 · batched M rows",
 * section 3.7, applied to each sequence of a batch), where m_dev is an int
 * array [B] in DEVICE memory, so a count produced on the device needs no
 * host round trip.  A value outside 0..M leaves that sequence's S
 * untouched and sets *err_dev (device int, may be NULL) to 1; the host call
 * itself cannot see device values.  Both snap and ckpt are required.
 */
int gdn_rollback_seq(const gdn_shape *shape, int M, const int *m_dev,
                     const float *snap, const float *ckpt, float *S,
                     int *err_dev, gdn_stream_t stream);

/*
 * gdn_prefill_workspace - bytes of device workspace gdn_prefill needs for
 * this shape, T, chunk and precision (0 for GDN_PREC_FP32).  Returns 0 and
 * sets nothing on invalid arguments; gdn_prefill validates again.  The
 * size-query convention of "24 · GDN linear attention to GPU", section 10
 * (ask for the size first, then pass a buffer that is large enough; a
 * buffer that is too small is refused, never truncated into), with the
 * caller owning the workspace as in "34 · batched M rows", section 3.5.
 */
size_t gdn_prefill_workspace(const gdn_shape *shape, int T, int chunk,
                             int precision);

/*
 * gdn_prefill - T tokens for all heads, state in place (in: S_0, out: S_T).
 *   q, k [B][T][kh][kd];  v, o [B][T][vh][vd];  g, beta [B][T][vh].
 * precision GDN_PREC_FP32: the token-serial path, bit-identical to T
 *   successive gdn_step calls; chunk and workspace are ignored (pass 0 /
 *   NULL).
 * GDN_PREC_BF16X3 / GDN_PREC_BF16: the chunk-parallel form with chunk ==
 *   64 (GDN_ERANGE otherwise), its dense products on tcgen05 tensor cores
 *   with fp32 accumulation and the state kept in tensor memory; one CTA
 *   per (sequence, value head) walks the chunks in order.  The chunked form
 *   regroups the token-serial recurrence of "24 · GDN linear attention to
 *   GPU", section 4; the articles themselves never use it ("34 · batched M
 *   rows", section 3.6).  Needs no workspace (gdn_prefill_workspace returns
 *   0; pass NULL, 0).  Results agree with the token-serial definition to
 *   the stated relative error, not bitwise.  The chunked form works with
 *   differences of cumulative sums of g, so every g must be finite there
 *   (a decay that empties the state is any g below about -104, where
 *   exp(g) is 0 in fp32; g = -inf would give NaN).  The token-serial path
 *   also accepts g = -inf.
 * 1 <= T <= GDN_MAX_TOKENS; in the chunked modes also T * vh < 2^31
 * (the tensor copies that move q, k and o address a sequence's rows with
 * strides below 2^40 bytes).  Other values, and other precision values,
 * give GDN_ERANGE.
 */
int gdn_prefill(const gdn_shape *shape, int T, float *S, const float *q,
                const float *k, const float *v, const float *g,
                const float *beta, float *o, int chunk, int precision,
                void *workspace, size_t ws_bytes, gdn_stream_t stream);

/*
 * gdn_prefill_timeouts - (an interface addition with no counterpart in the
 * articles) number of chunked-prefill CTAs, since the library
 * was loaded on the current device, that gave up waiting for a tensor-core
 * operation (each wait is bounded).  Such a CTA writes NaN into its head's
 * whole state and every o row of its head, so the failure shows in the
 * results too.  Synchronises the current device.  Expected to stay 0.
 */
int gdn_prefill_timeouts(unsigned int *count);

/*
 * gdn_wait_timeouts - (an interface addition with no counterpart in the
 * articles) number of bounded waits, since the library was loaded on the
 * current device, that ran out in any kernel: the chunked prefill's
 * tensor-core waits (as gdn_prefill_timeouts) and the multi-token update's
 * waits for its token inputs (gdn_step_m with M > 1 or checkpoints, the
 * fp32 prefill, the layer step; device-resident inputs).  A CTA whose wait
 * runs out writes NaN into every state, checkpoint and o element it had not
 * yet produced, so the failure also shows in the results themselves.
 * Synchronises the current device.  Expected to stay 0.
 */
int gdn_wait_timeouts(unsigned int *count);

/*
 * gdn_layer_prologue_m - the per-token layer core that produces the inputs
 * of the update from raw projections, for M tokens: a depthwise causal
 * convolution of width ck over the raw mixed q|k|v projection with a
 * rolling history of the previous ck-1 inputs (oldest first), SiLU, q and k
 * scaled to unit L2 norm per key head (x / sqrt(|x|^2 + eps)), and the gates
 *     beta = 1 / (1 + exp(-b)),
 *     g    = -exp(A_log) * softplus(a + dt_bias)
 *            (softplus(x) = x above 20, exp(x) below -20,
 *             log1p(exp(x)) otherwise).
 * These are steps 2-4 of figure 1 of "24 · GDN linear attention to GPU"
 * (conv + SiLU and the gates are listed in its section 3; the article names
 * the q/k normalisation without its formula, and the form above is this
 * library's reading).  One streaming kernel: one warp per 128-channel row.
 *   ck       must be 4 (GDN_ESHAPE otherwise); conv_dim = 2*kh*kd + vh*vd
 *   hist_in  [B][ck-1][conv_dim]  in: the previous ck-1 raw inputs
 *   hist_out [B][ck-1][conv_dim]  out: the last ck-1 raw inputs after
 *            token M-1; must not overlap hist_in (use two buffers in turn)
 *   x        [B][M][conv_dim]  raw projections, channels q (kh*kd), then k
 *            (kh*kd), then v (vh*vd)
 *   conv_w   [conv_dim][ck]
 *   a, b     [B][M][vh];   A_log, dt_bias [vh]
 *   eps      >= 0 (GDN_EINVAL otherwise)
 *   q, k     [B][M][kh][kd] out;  v [B][M][vh][vd] out;  g, beta [B][M][vh] out
 *            (exactly the inputs gdn_step_m takes)
 */
int gdn_layer_prologue_m(const gdn_shape *shape, int M, int ck, float eps,
                         const float *hist_in, float *hist_out,
                         const float *x, const float *conv_w, const float *a,
                         const float *b, const float *A_log,
                         const float *dt_bias, float *q, float *k, float *v,
                         float *g, float *beta, gdn_stream_t stream);

/*
 * gdn_layer_workspace - bytes of device workspace gdn_layer_step_m needs to
 * hold the M tokens' q, k, v, g and beta between its two kernels (0 on
 * invalid arguments).  Size query as in "24 · GDN linear attention to GPU",
 * section 10; the caller-owned M-token slab of "34 · batched M rows",
 * section 3.5.
 */
size_t gdn_layer_workspace(const gdn_shape *shape, int M);

/*
 * gdn_layer_step_m - steps 2-5 of figure 1 of "24 · GDN linear attention to
 * GPU" for M tokens: gdn_layer_prologue_m followed by gdn_step_m on the same
 * stream, with the intermediate q, k, v, g, beta in the caller's workspace
 * (at least gdn_layer_workspace() bytes, 16-byte aligned, device memory;
 * GDN_ERANGE if smaller).  Arguments as in those two calls.  Output m and
 * ckpt[m] are bit-identical to the m-th of M successive calls with M = 1
 * that pass the history forward.
 */
int gdn_layer_step_m(const gdn_shape *shape, int M, int ck, float eps,
                     const float *S_in, float *S_out, float *ckpt,
                     const float *hist_in, float *hist_out, const float *x,
                     const float *conv_w, const float *a, const float *b,
                     const float *A_log, const float *dt_bias, float *o,
                     void *workspace, size_t ws_bytes, gdn_stream_t stream);

/*
 * gdn_layer_hist_rollback - the convolution history after m_dev[b] of the
 * M tokens of a gdn_layer_step_m call, for every sequence b ("34 · batched
 * M rows", section 3.7, rolls the convolution history back together with
 * the recurrent state): rows
 * m .. m+ck-2 of the sequence [hist_snap rows, x rows], where hist_snap is
 * that call's hist_in and x its raw inputs (the history stores inputs, so
 * no per-token copy is needed).  m_dev: device int [B]; a value outside
 * 0..M leaves that sequence's hist untouched and sets *err_dev (may be
 * NULL) to 1.  hist must not overlap hist_snap or x.  ck must be 4.
 */
int gdn_layer_hist_rollback(const gdn_shape *shape, int M, int ck,
                            const int *m_dev, const float *hist_snap,
                            const float *x, float *hist, int *err_dev,
                            gdn_stream_t stream);

/*
 * gdn_gated_rmsnorm_m - the gated RMS normalisation of the update's output,
 * per (sequence, token, value head) row of vd channels:
 *     y = w * o / sqrt(mean(o^2) + eps) * silu(z),   silu(z) = z / (1 + exp(-z)).
 * Step 6 of figure 1 of "24 · GDN linear attention to GPU", run there one
 * value head at a time; the article prints no formula, and the form above
 * (weight per channel, SiLU output gate) is this library's reading.
 *   o, z, y  [B][M][vh][vd]  (o as written by gdn_step_m / gdn_layer_step_m;
 *            z the gate projection); y may be o (in place), otherwise y must
 *            not overlap o; y must not overlap z or w
 *   w        [vd], shared by all heads
 *   eps      >= 0 (GDN_EINVAL otherwise);  1 <= M <= GDN_MAX_TOKENS
 * One streaming kernel, one warp per row.
 */
int gdn_gated_rmsnorm_m(const gdn_shape *shape, int M, float eps,
                        const float *o, const float *z, const float *w,
                        float *y, gdn_stream_t stream);

/* Bytes of the static scratch array behind gdn_layer_step_m_noalloc. */
#define GDN_NOALLOC_SCRATCH_BYTES (16u << 20)

/*
 * gdn_layer_step_m_noalloc - gdn_layer_step_m without a workspace argument,
 * for callers that cannot allocate device memory (a host handed only the
 * layer's tensors by a runtime whose allocator it cannot reach, or a decode
 * loop that must not call cudaMalloc, which can synchronise the device and
 * fail under memory pressure, between steps).  The article has no
 * counterpart: this is an interface variant, not a step of the method.
 *
 * The intermediate q, k, v, g and beta go to a file-scope device array of
 * GDN_NOALLOC_SCRATCH_BYTES (16 MiB), which every GPU that loads the
 * library's device code holds until the process exits.  The call allocates
 * nothing: no cudaMalloc, no cudaFree, no allocating library routine.
 *   - Limit: a request whose gdn_layer_workspace() exceeds
 *     GDN_NOALLOC_SCRATCH_BYTES returns GDN_ESCRATCH and launches nothing
 *     (at kh = 16, vh = 48, kd = vd = 128, 41,344 bytes per sequence and
 *     token: B * M > 405).
 *   - Set-up: the first call on a device, with that device current, looks
 *     up the array's device address (cudaGetSymbolAddress) and keeps it;
 *     make that first call before any stream capture begins.  The address
 *     is kept per device and CUDA context: after cudaDeviceReset the next
 *     call on that device repeats the set-up (make it, too, outside any
 *     capture).
 *   - Sharing: all calls on a device share the one array, which keeps the
 *     last call's contents.  Nothing in it needs to start at zero (every
 *     byte read is written first in the same call), so nothing is cleared.
 *     Calls whose work overlaps on the GPU (different streams with no
 *     ordering between them) race on the array: order them on one stream or
 *     with events.
 * Other arguments, results and status codes are those of gdn_layer_step_m,
 * and results are bit-identical to it on the same inputs.  Arguments are
 * checked first, exactly as gdn_layer_step_m checks them, so GDN_ESCRATCH
 * is returned only for a request that is otherwise valid.
 */
int gdn_layer_step_m_noalloc(const gdn_shape *shape, int M, int ck, float eps,
                             const float *S_in, float *S_out, float *ckpt,
                             const float *hist_in, float *hist_out,
                             const float *x, const float *conv_w,
                             const float *a, const float *b,
                             const float *A_log, const float *dt_bias,
                             float *o, gdn_stream_t stream);

/* Static description of a status code (never NULL).  The codes are the
 * refusals of "24 · GDN linear attention to GPU", section 8 (a request the
 * library cannot serve as asked is refused with an error, never served by a
 * silent fallback), and of its section 10 (no truncation). */
const char *gdn_strerror(int status);

/* Library ABI version: major * 10000 + minor * 100 + patch (an interface
 * addition; the articles have no counterpart). */
int gdn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GDN_GB300_H */
