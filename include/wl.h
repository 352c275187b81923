/*
 * wl.h -- C ABI of libwl.so, weightless linear projections on GB300 (sm_103a).
 *
 * A weightless projection never holds its dense weight.  Each weight is the
 * theta bundle of the "Serve and generate with weightless" page (overview):
 * a W0 block shared per band of layers, a per-output-row scale s and a rank-r
 * delta U, V.  Every call rebuilds the projection inside the kernel
 * ("In-kernel reconstruction" page, formula section):
 *
 *     y[t,o] = s[o] * sum_i W0[o,i] x[t,i] + sum_k U[o,k] * sum_i V[i,k] x[t,i]
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layouts (row-major, contiguous, PyTorch Linear convention):
 *    x  [T, in]   bf16          W0 [out, in] bf16        s [out] fp32
 *    U  [out, r]  bf16          V  [in, r]   bf16        y [T, out] bf16 or fp32
 *  Precision: bf16 inputs, fp32 accumulation, fp32 combine, one final
 *    round-to-nearest-even cast to the output type ("In-kernel
 *    reconstruction": the custom-op path accumulates in float32; the GEMM
 *    path does its final combine in float32 before the cast).
 *  Memory: every pointer is device memory owned by the caller.  The library
 *    allocates nothing in these calls.  Outputs must not alias inputs.
 *  Streams: `stream` is a cudaStream_t (NULL = legacy default stream).  Calls
 *    are asynchronous on that stream; results are ready when it is.  The
 *    decode-size launches (wl_linear, wl_qkv_fused, wl_mlp_geglu_fused at
 *    T <= 8) use programmatic dependent launch: they start streaming W0, s,
 *    U and V while the previous kernel on the stream finishes, and read x
 *    (and write y) only after it has completed.  So the weights must not be
 *    written by the kernel launched immediately before the call on the same
 *    stream; weights written by a copy (cudaMemcpy*), on another stream
 *    joined by an event, or by any earlier kernel are fine.
 *  Errors: return codes only; nothing is thrown or aborted across the ABI.
 *    Arguments are checked before anything is launched; on error nothing is
 *    launched and wl_last_error() describes the failure.  A failed launch
 *    returns WL_ERR_CUDA.  Kernel-side bounded waits that give up record
 *    WL_ERR_TIMEOUT in a device status word, read by wl_device_status().
 *  Limits: T >= 1, in >= 8, out >= 1, in % 8 == 0, 0 <= r <= WL_MAX_RANK;
 *    x, W0 and y must be 16-byte aligned (in % 8 == 0 keeps every row of x
 *    and W0 aligned when the base is); U and V may be NULL only if r == 0.
 */
#ifndef WL_H_
#define WL_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    WL_OK = 0,
    WL_ERR_INVALID_ARG = 1, /* bad pointer, size, alignment or rank        */
    WL_ERR_UNSUPPORTED = 2, /* valid arguments this build cannot run       */
    WL_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed        */
    WL_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up          */
    WL_ERR_WORKSPACE = 5,   /* workspace missing, misaligned or too small  */
    WL_ERR_INTERNAL = 6     /* a plan broke an invariant of the library;
                               nothing was launched (a library bug)        */
} wl_status;

typedef enum { WL_OUT_BF16 = 0, WL_OUT_F32 = 1 } wl_out_dtype;

/* One projection's theta bundle: W0 [out, in], s [out], U [out, r], V [in, r]. */
typedef struct {
    const void *W0;
    const float *s;
    const void *U;
    const void *V;
    int64_t out;
} wl_proj;

#define WL_MAX_RANK 128

/*
 * wl_linear -- one weightless projection, y = s*(x W0^T) + (x V) U^T.
 * Source: "In-kernel reconstruction", formula section (per-element form) and
 * "The GEMM path" (the same map as s[None,:]*(x@W0.T) + (x@V)@U.T).
 * x [T,in] bf16, W0 [out,in] bf16, s [out] fp32, U [out,r] bf16, V [in,r] bf16,
 * y [T,out] of type ydt.  Small T (decode) streams W0 once from HBM with the
 * rank-r term and the scale folded into the same launch; large T (prefill)
 * runs the dense contraction on the tensor cores with the low-rank term in
 * the epilogue.  Both give the same result within fp32 accumulation order.
 */
wl_status wl_linear(const void *x, const void *W0, const float *s, const void *U,
                    const void *V, void *y, int64_t T, int64_t in, int64_t out,
                    int64_t r, wl_out_dtype ydt, void *stream);

/*
 * wl_qkv_fused -- the three attention projections that share one input x, in
 * one launch that reads x once ("In-kernel reconstruction", "Q/K/V fusion").
 * Each of q, k, v is a full theta bundle with its own out (in and r shared);
 * yq [T,q.out], yk [T,k.out], yv [T,v.out].  Equal, within accumulation
 * order, to three wl_linear calls.
 */
wl_status wl_qkv_fused(const void *x, wl_proj q, wl_proj k, wl_proj v, void *yq,
                       void *yk, void *yv, int64_t T, int64_t in, int64_t r,
                       wl_out_dtype ydt, void *stream);

/*
 * wl_mlp_workspace_bytes -- bytes of device workspace wl_mlp_geglu_fused
 * needs for these sizes (the intermediate h = gelu(g)*u and the partial sums
 * of the down projection's low-rank input h V_down).  Calls of up to 8 tokens
 * run the HBM-streaming kernels unless no launch plan of theirs fits shared
 * memory for these sizes (then the tensor-core kernels run); the size covers
 * both.  Returns 0 for invalid sizes.
 */
size_t wl_mlp_workspace_bytes(int64_t T, int64_t hidden, int64_t inter, int64_t r,
                              wl_out_dtype ydt);

/*
 * wl_mlp_geglu_fused -- the gated MLP of a weightless layer in one call
 * ("In-kernel reconstruction", custom-op path: gate, up, activation and down
 * fused into one dispatch):
 *     g = wl(x; gate), u = wl(x; up)          [T, inter]
 *     h = gelu_tanh(g) * u                    [T, inter]
 *     y = wl(h; down)                         [T, hidden]   (down.out == hidden)
 * gelu_tanh(v) = 0.5 v (1 + tanh(sqrt(2/pi) (v + 0.044715 v^3))).
 * workspace: caller-owned device memory of at least
 * wl_mlp_workspace_bytes(T, hidden, inter, r, ydt) bytes, 256-byte aligned;
 * its contents need no initialisation.  Calls sharing one workspace must not
 * overlap in time (calls on one stream never do).
 */
wl_status wl_mlp_geglu_fused(const void *x, wl_proj gate, wl_proj up, wl_proj down,
                             void *y, int64_t T, int64_t hidden, int64_t inter,
                             int64_t r, void *workspace, size_t ws_bytes,
                             wl_out_dtype ydt, void *stream);

/*
 * wl_mlp_geglu_fused_noalloc -- the same fused GeGLU MLP as
 * wl_mlp_geglu_fused, for callers that cannot allocate device memory (code
 * that may not call cudaMalloc, such as a host callback, an allocator hook or
 * a process whose device-memory budget is fixed at start-up).  It takes no
 * workspace: it uses a 4 MiB scratch array built into libwl.so, which every
 * GPU that loads the library holds until the process exits.  The documentation
 * pages have no counterpart to this call; it exists for such callers.
 *   - Sizes whose workspace (wl_mlp_workspace_bytes) exceeds 4 MiB are
 *     rejected with WL_ERR_UNSUPPORTED and a message; nothing is launched.
 *   - The first call on a device looks up the scratch address for that device
 *     (make it before any stream capture on that device).
 *   - The scratch keeps whatever the previous call left; nothing in it has to
 *     start at zero.  No call allocates or frees memory.
 *   - All calls share the one scratch array: calls that overlap on the GPU
 *     (different streams, or different host threads) race and give wrong
 *     results.  Serialise them.
 */
wl_status wl_mlp_geglu_fused_noalloc(const void *x, wl_proj gate, wl_proj up, wl_proj down,
                                     void *y, int64_t T, int64_t hidden, int64_t inter,
                                     int64_t r, wl_out_dtype ydt, void *stream);

/*
 * fp32 encoding ("Serve and generate with weightless", "Supported encodings
 * and devices": the architectures default to bfloat16 and also support
 * float32).  The same projection with x, W0, s, U and V all fp32:
 *     y = s*(x W0^T) + (x V) U^T
 * computed with fp32 multiply-adds throughout (no bf16 or tf32 rounding of
 * any operand); y is fp32 or bf16 (ydt).  Layouts as above with 4-byte
 * elements: x [T,in], W0 [out,in], s [out], U [out,r], V [in,r], y [T,out].
 * Limits and errors as wl_linear; pointers 16-byte aligned except s, U, V
 * (4-byte).  Equal, within fp32 accumulation order, to the fp64 product of
 * the fp32 values.
 */
typedef struct {
    const float *W0;
    const float *s;
    const float *U;
    const float *V;
    int64_t out;
} wl_proj_f32;

wl_status wl_linear_f32(const float *x, const float *W0, const float *s, const float *U,
                        const float *V, void *y, int64_t T, int64_t in, int64_t out,
                        int64_t r, wl_out_dtype ydt, void *stream);

/* Q, K, V of one fp32 x in one launch (x read once per token tile). */
wl_status wl_qkv_fused_f32(const float *x, wl_proj_f32 q, wl_proj_f32 k, wl_proj_f32 v,
                           void *yq, void *yk, void *yv, int64_t T, int64_t in, int64_t r,
                           wl_out_dtype ydt, void *stream);

/*
 * wl_materialize -- W_eff = s*W0 + U V^T, formed once (the load-time
 * precompute of "Serve and generate with weightless", "Set the fast path on
 * NVIDIA").  W_eff [out, in] of type dt (fp32 or bf16).  Bit-exact with one
 * fixed fp32 order per element:
 *     d = +0; for k = 0..r-1: d = fma(U[o,k], V[i,k], d)
 *     w = fl(s[o] * W0[o,i]); if r > 0: w = fl(w + d)
 * then, for bf16, one round-to-nearest-even.
 */
wl_status wl_materialize(const void *W0, const float *s, const void *U, const void *V,
                         void *W_eff, int64_t out, int64_t in, int64_t r,
                         wl_out_dtype dt, void *stream);

/*
 * Decomposition of dense projection weights into theta bundles (the pages'
 * weight adapter "auto-decomposes" a checkpoint into the bundle: "Serve and
 * generate with weightless", "How the custom architecture loads").  One call
 * handles one band: the n layers of one projection family that share a W0.
 * Steps (the pages fix only the passthrough point G = num_layers, where each
 * reconstructed weight equals the original; the rest is this library's
 * reading):
 *   W0 = mean of the n weights (fp32 sum, bf16 round-to-nearest-even);
 *   s_l[o] = <W_l[o], W0[o]> / <W0[o], W0[o]> (1 where the W0 row is zero);
 *   U_l, V_l: rank-r truncated SVD of R_l = W_l - diag(s_l) W0, split evenly
 *   (U = U_r S^1/2, V = V_r S^1/2), by randomized subspace iteration from the
 *   caller's Gaussian start omega [in, r + p] fp32 with `iters` power
 *   iterations (Halko, Martinsson and Tropp 2011), then bf16.
 * With n = 1 the bundle is the passthrough one: W0 = W, s = 1, U = V = 0.
 * W: host array of n device pointers to bf16 [out, in] (16-byte aligned).
 * Outputs (device, caller-owned): W0 bf16 [out, in]; s fp32 [n, out];
 * U bf16 [n, out, r]; V bf16 [n, in, r].  workspace: at least
 * wl_decompose_workspace_bytes(out, in, r, p) bytes, 256-byte aligned.
 * Limits: 1 <= n <= 64, in % 8 == 0, 0 <= r <= min(out, in, 128),
 * 0 <= p, r + p <= 160, 0 <= iters <= 64.  Asynchronous on `stream`.
 */
size_t wl_decompose_workspace_bytes(int64_t out, int64_t in, int64_t r, int64_t p);

wl_status wl_decompose_band(const void *const *W, int64_t n, int64_t out, int64_t in, int64_t r,
                            int64_t p, int64_t iters, const float *omega, void *W0, float *s,
                            void *U, void *V, void *workspace, size_t ws_bytes, void *stream);

/*
 * Decoder-layer stacks at decode size, in one launch per step.
 *
 * A weightless decoder layer applies its projections in a chain ("Serve and
 * generate with weightless": every linear layer of the model is a theta
 * bundle; "In-kernel reconstruction", formula section, per projection):
 *     q, k, v = wl(x_l; q), wl(x_l; k), wl(x_l; v)
 *     o       = wl(q; o)                  (q stands in for attention, which
 *                                          is not part of the method)
 *     g, u    = wl(o; gate), wl(o; up);   h = gelu_tanh(g) * u
 *     x_{l+1} = wl(h; down)
 * Every output is bf16 (round-to-nearest-even of the fp32 result, as for
 * wl_linear with WL_OUT_BF16); h keeps fp32 accuracy inside the launch (it
 * enters the down projection as a bf16 pair hi + lo).  Each output of each
 * layer equals, within fp32 accumulation order, the single-projection calls
 * on that layer's bf16 inputs.  At batch 1 a launch per projection costs more than its weight
 * traffic ("What weightless inference costs": at batch-1 decode extra
 * dispatches, not extra arithmetic, dominate), so one launch streams the
 * weights of all L layers and follows the data dependencies inside it.
 */
typedef struct {
    wl_proj q, k, v, o, gate, up, down; /* gate.out == up.out == inter, o.out == down.out == hidden */
} wl_layer;

/* Output buffers of one layer, bf16 [T, n], row-major, 16-byte aligned. */
typedef struct {
    void *yq; /* [T, q.out]  */
    void *yk; /* [T, k.out]  */
    void *yv; /* [T, v.out]  */
    void *yo; /* [T, hidden] */
    void *ym; /* [T, hidden]: the layer's output and the next layer's input */
} wl_layer_out;

typedef struct wl_stack_s *wl_stack;

/*
 * wl_stack_create -- bind L layers and their output buffers (all device
 * memory owned by the caller, which must outlive the stack) into a stack for
 * T tokens on the current device.  Allocates the stack's own device tables
 * and scratch (cudaMalloc; freed by wl_stack_destroy) and uploads them
 * synchronously: call it outside stream capture.
 * Limits: 1 <= T <= 32, 0 <= r <= 32; hidden, q.out and gate.out multiples
 * of 64; every layer with the shapes of layer 0; W0 and V 16-byte aligned.
 * 1..4 tokens and 5..32 tokens run different kernels (the second reduces each
 * output row tile once and hands it on as bf16).
 * Output buffers of different layers must be distinct and may not alias any
 * input.  Sizes outside these limits give WL_ERR_UNSUPPORTED (use the
 * per-projection calls).  On error *out is NULL.
 */
wl_status wl_stack_create(wl_stack *out, const wl_layer *layers, const wl_layer_out *outs,
                          int64_t L, int64_t T, int64_t hidden, int64_t r);

/*
 * wl_stack_decode -- one pass over all layers of the stack for input x
 * [T, hidden] bf16 (device, 16-byte aligned), asynchronous on `stream`.
 * Writes every output of every layer.  Launches must not overlap: calls on
 * one stream never do.  Each step first runs a small kernel that writes V^T
 * of every projection (and, above 4 tokens, clears the step's flags).  The launch is cooperative (one CTA per SM); it
 * cannot be captured into a CUDA graph on drivers that refuse cooperative
 * launches in capture.
 */
wl_status wl_stack_decode(wl_stack stack, const void *x, void *stream);

/* Free the stack's device memory (after its last launch has completed). */
void wl_stack_destroy(wl_stack stack);

/*
 * wl_band_of_layer -- which of the G shared W0 blocks layer `layer` of an
 * L-layer stack uses: floor(layer * G / L) (contiguous bands).  G = L is the
 * passthrough point (one W0 per layer, "Set the fast path on NVIDIA"); G = 1
 * shares one block ("What weightless inference costs", Compression).
 * Returns -1 unless 0 <= layer < L and 1 <= G <= L.  Host-only, exact.
 */
int64_t wl_band_of_layer(int64_t layer, int64_t L, int64_t G);

/*
 * wl_device_status -- synchronise `stream`, then read and clear the device
 * status word of the current device.  Returns WL_ERR_TIMEOUT if a bounded
 * wait in a kernel of this library gave up since the last read, WL_ERR_CUDA
 * if the synchronisation failed, else WL_OK.
 */
wl_status wl_device_status(void *stream);

/*
 * wl_selftest_wait -- diagnostic for the failure detection above (the pages
 * have no counterpart): launches on `stream` one kernel that waits, through
 * the same bounded-wait code as the projection kernels' ring stages, on a
 * barrier that nothing arrives on.  The wait gives up after its limit (4e9 SM
 * cycles, about 2 s), so the next wl_device_status(stream) returns
 * WL_ERR_TIMEOUT; the GPU context stays usable.  Returns WL_OK once launched,
 * WL_ERR_CUDA if the launch failed.
 */
wl_status wl_selftest_wait(void *stream);

/* Message for the last error on the calling thread ("" if none). */
const char *wl_last_error(void);

/* Library version string. */
const char *wl_version(void);

#ifdef __cplusplus
}
#endif

#endif /* WL_H_ */
