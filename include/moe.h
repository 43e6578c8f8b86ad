/*
 * moe.h -- C ABI of a GB300 (sm_103a) forward pass of one Mixture-of-Experts
 * FFN layer of the Hy3 kind: fp32-accurate router GEMM, sigmoid+bias (or
 * softmax) top-k routing, per-expert histogram and permutation, grouped
 * SwiGLU expert GEMMs that read tokens through the route index, an always-on
 * shared expert, and the top-k weighted combine back to token order.
 *
 * Sources (page title, section):
 *   [hy3]   "hy3 -- tencent/Hy3 GGUF Converter and Inference Engine", Model facts
 *           (hidden 4096, 192 routed experts top-8 + 1 shared, expert
 *           intermediate 1536, MoE routing rule, F32 router).
 *   [case]  "Hy3 Preview inference optimisation case", section 2 Router GEMM
 *           (W ~ W_high + W_low/256, two BF16 GEMMs, two accumulators, one FFMA
 *           epilogue) and section 3 FusedMoE (index preprocessing with one
 *           contiguous range per expert, gate-up GEMM through the route index,
 *           compact per-expert down GEMM, top-k aggregation at the end, PDL).
 *   [image] "HunyuanImage 3.0 MoE reading", HunyuanTopKGate easy_topk (softmax,
 *           top-k, clamp(sum, 1e-8)), Routed Experts (eager loop, weighted sum
 *           over k, stacked expert weights), Shared MLP.
 *
 * Conventions for every entry point
 *   - bf16 tensors are passed as moe_bf16 (uint16_t bit patterns of bfloat16).
 *   - Every pointer is a DEVICE pointer owned by the caller, 16-byte aligned
 *     (the workspace 256-byte aligned).  The library never allocates, frees or
 *     synchronises; all work is enqueued on `stream` (a cudaStream_t, NULL for
 *     the legacy default stream) and the call returns once it is enqueued.
 *   - Weights are nn.Linear [out, in] row-major: w_gate, w_up [E, I, H];
 *     w_down [E, H, I]; shared ws_gate, ws_up [I_shared, H]; ws_down [H, I_shared].
 *   - Argument errors are returned before anything is launched:
 *       MOE_ERR_INVALID_ARG  null / misaligned pointer, negative size, bad mode
 *       MOE_ERR_UNSUPPORTED  a shape outside the supported set (below)
 *       MOE_ERR_WORKSPACE    ws_bytes < moe_workspace_bytes(d)
 *       MOE_ERR_CUDA         a launch or driver call failed
 *     Anomalies seen on the device (an index outside its range, a bounded wait
 *     that ran out) are recorded as bits in an error word at the start of the
 *     workspace and read with moe_ws_read_error().
 *   - Supported shapes: T >= 0 (T = 0 is a no-op, and T-sized buffers may
 *     then be NULL; moe_permute still zeroes counts and offsets); H and I (and I_shared when
 *     has_shared) multiples of 64, H <= 16384, I <= 16384; 1 <= E <= 256;
 *     1 <= top_k <= min(E, 16); T * top_k < 2^31.
 *   - The workspace must be zero-filled once after it is allocated (or passed
 *     to moe_ws_init); the library leaves it reusable.  One workspace must not
 *     be used by two calls that overlap on the device.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,
  MOE_ERR_UNSUPPORTED = 2,
  MOE_ERR_WORKSPACE = 3,
  MOE_ERR_CUDA = 4,
  MOE_ERR_DEVICE_TIMEOUT = 5,
  MOE_ERR_DEVICE_INDEX = 6
} moe_status;

typedef enum {
  MOE_SCORE_SIGMOID_BIAS = 0, /* [hy3] Model facts, MoE routing */
  MOE_SCORE_SOFTMAX = 1       /* [image] HunyuanTopKGate easy_topk */
} moe_score_mode;

/* Bits of the device error word (moe_ws_read_error). */
#define MOE_DEVERR_INDEX 0x1u   /* a routing index or permutation entry out of range (clamped) */
#define MOE_DEVERR_TIMEOUT 0x2u /* a bounded wait inside a kernel ran out; that kernel gave up */
#define MOE_DEVERR_OFFSETS 0x4u /* offsets not monotone or offsets[E] != T * top_k; no expert work done */

/* Layer dimensions and routing mode.
 *   T tokens, H hidden size, E routed experts, I expert intermediate size,
 *   I_shared shared-expert intermediate size (ignored when has_shared == 0),
 *   top_k experts per token.
 *   score_mode MOE_SCORE_SIGMOID_BIAS: s = sigmoid(logits); the top_k is chosen
 *     on s + expert_bias; weights = s_sel / sum(s_sel) * route_scale ([hy3]:
 *     route_scale = 2.826).  renorm_eps is not used.
 *   score_mode MOE_SCORE_SOFTMAX: p = softmax(logits) over the E experts; the
 *     top_k of p; weights = p_sel / max(sum(p_sel), renorm_eps) ([image]:
 *     renorm_eps = 1e-8).  route_scale must be 1 and expert_bias is ignored.
 *   Equal keys go to the lower expert index; topk_idx lists each token's
 *   experts in descending key order. */
typedef struct {
  int T, H, E, I, I_shared, top_k;
  int score_mode;
  float route_scale;
  float renorm_eps;
  int has_shared;
} moe_dims;

/* Human-readable name of a status code (static storage). */
const char *moe_status_string(moe_status s);

/* Validate dims against the supported set; MOE_OK, INVALID_ARG or UNSUPPORTED. */
moe_status moe_check_dims(const moe_dims *d);

/* Bytes of workspace every entry point below needs for these dims (the fused
 * layer's need, which covers the others); 0 when the dims are invalid. */
size_t moe_workspace_bytes(const moe_dims *d);

/* Zero the workspace header (error word and tile-scheduler counters, the first
 * 4 KiB) on `stream`. */
moe_status moe_ws_init(void *ws, size_t ws_bytes, void *stream);

/* Read (and, with clear != 0, reset) the device error word.  This is the one
 * call that synchronises `stream`; *bits receives MOE_DEVERR_* flags. */
moe_status moe_ws_read_error(void *ws, size_t ws_bytes, int clear, void *stream, uint32_t *bits);

/* Self-test of the bounded waits inside the kernels: one CTA waits on a
 * barrier phase that nothing completes, gives up after limit_ns (1 ns .. 10 s),
 * records MOE_DEVERR_TIMEOUT in the workspace error word and returns; read it
 * with moe_ws_read_error.  Every wait in this library's kernels is bounded the
 * same way (1 s), so a broken pipeline reports an error instead of hanging. */
moe_status moe_selftest_wait_timeout(void *ws, size_t ws_bytes, unsigned long long limit_ns, void *stream);

/* Self-test of step a6's arithmetic: out[i] = SiLU(g[i]) * u[i] computed by the
 * same device function the expert kernel's gate/up epilogue uses (a hardware
 * base-2 exponential and a Newton-Raphson reciprocal), so that its error can be
 * measured against a float64 reference.  g, u, out: [n] fp32 device arrays,
 * 4-byte aligned; n >= 0 (0 is a no-op).  Async on `stream`. */
moe_status moe_selftest_silu(const float *g, const float *u, float *out, int64_t n, void *stream);

/* Steps a1-a2: router GEMM and routing.  [case] section 2; [hy3] MoE routing;
 * [image] easy_topk.
 *   hidden      [T, H] bf16 row-major (input)
 *   router_w    [E, H] fp32 row-major (input); a first pass writes
 *               W_high = bf16_RNE(W), W_low = bf16_RNE((W - W_high) * 256) into the
 *               workspace, then two BF16 tensor-core GEMMs run into two fp32
 *               accumulators and logits = acc_lo * (1/256) + acc_hi (one FFMA);
 *               the K dimension may be split across CTAs, whose partial logits
 *               are summed in a fixed order
 *   expert_bias [E] fp32 (input, may be NULL = zeros; sigmoid mode only)
 *   logits_out  [T, E] fp32 (output, may be NULL)
 *   topk_idx    [T, top_k] int32 (output), topk_w [T, top_k] fp32 (output) */
moe_status moe_route(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                     const float *expert_bias, float *logits_out, int32_t *topk_idx, float *topk_w,
                     void *ws, size_t ws_bytes, void *stream);

/* Steps a3-a4: per-expert histogram, offsets and permutation.  [case] section 3
 * (routing and index preprocessing: shared-memory block counts, one contiguous
 * range per expert); [image] Routed Experts (flattened slot t * top_k + j).
 *   topk_idx [T, top_k] int32 (input; entries outside [0, E) are clamped and
 *            flagged with MOE_DEVERR_INDEX)
 *   counts   [E] int32, offsets [E + 1] int32 (exclusive prefix of counts)
 *   perm     [T * top_k] int32: perm[p] = flat slot at sorted position p; slots of
 *            one expert are in ascending slot order (deterministic, stable)
 *   inv_perm [T * top_k] int32: inv_perm[slot] = p */
moe_status moe_permute(const moe_dims *d, const int32_t *topk_idx, int32_t *counts, int32_t *offsets,
                       int32_t *perm, int32_t *inv_perm, void *ws, size_t ws_bytes, void *stream);

/* Steps a5-a8: grouped gate/up GEMM reading hidden rows through perm (no gather
 * copy), SiLU(gate) * up, grouped down GEMM, and the shared expert.  [case]
 * section 3; [image] Routed Experts and Shared MLP.
 *   hidden   [T, H] bf16; perm [T * top_k], offsets [E + 1] as moe_permute writes them
 *   w_gate, w_up [E, I, H] bf16; w_down [E, H, I] bf16
 *   ws_gate, ws_up [I_shared, H]; ws_down [H, I_shared] bf16 (NULL when !has_shared)
 *   y_sorted [T * top_k, H] bf16 (output): y_sorted[p] = FFN_e(hidden[perm[p] / top_k])
 *            for p in expert e's range
 *   y_shared [T, H] bf16 (output, NULL when !has_shared): shared FFN of every token */
moe_status moe_expert_ffn(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                          const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                          const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                          const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared, void *ws,
                          size_t ws_bytes, void *stream);

/* The two kernels of moe_expert_ffn as separate calls (same kernels, same
 * results): the gate/up half (a5-a6) writes the bf16 activation
 * SiLU(gate) * up of every routed slot and every token's shared-expert
 * activation into the workspace; the down half (a7-a8) reads them from the
 * same workspace and writes y_sorted / y_shared.  Call them in this order on
 * one stream with one workspace; arguments as for moe_expert_ffn. */
moe_status moe_expert_gate_up(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                              const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                              const moe_bf16 *ws_gate, const moe_bf16 *ws_up, void *ws, size_t ws_bytes,
                              void *stream);
moe_status moe_expert_down(const moe_dims *d, const int32_t *offsets, const moe_bf16 *w_down,
                           const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared, void *ws,
                           size_t ws_bytes, void *stream);

/* moe_expert_ffn for callers that cannot allocate device memory: a plugin
 * running inside a host framework that owns every device allocation and hands
 * its plugins none, or a latency-critical serving loop that must not call
 * cudaMalloc once it is running (cudaMalloc can synchronise the device).  It
 * takes no workspace: its scratch is a 32 MiB array that this library keeps in
 * device memory on every GPU that loads it, until the process exits.  There is
 * no counterpart on the pages: this is an interface convenience, not a step of
 * the layer.
 *   Arguments and results as for moe_expert_ffn (the caller still passes every
 *   input and output).  The scratch holds a 4 KiB header and the bf16
 *   activations, T * top_k * I + T * I_shared values; dims that need more than
 *   32 MiB are rejected with MOE_ERR_WORKSPACE before anything is launched (for
 *   the Hy3 shape that admits batches up to T = 1213 tokens).
 *   The first call in a CUDA context looks up that context's address of the
 *   array (cudaGetSymbolAddress) and caches it under the context's unique id;
 *   make that first call before any stream capture.
 *   Every call uses the same array: calls that overlap on the device (two
 *   streams, or two host threads) race and give wrong results; serialise them.
 *   Device-side anomalies cannot be read back on this path: the error word lives
 *   in the array and every call clears it.  After one (perm or offsets outside
 *   their ranges, or a bounded wait that ran out) y_sorted and y_shared are
 *   undefined; callers that need to detect it use moe_expert_ffn with a
 *   workspace and moe_ws_read_error. */
moe_status moe_expert_ffn_noalloc(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                                  const int32_t *offsets, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                                  const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                                  const moe_bf16 *ws_down, moe_bf16 *y_sorted, moe_bf16 *y_shared, void *stream);

/* Step a9: out[t] = sum_j topk_w[t, j] * y_sorted[inv_perm[t * top_k + j]] + y_shared[t]
 * (fp32 sum in j order, one bf16 rounding).  [case] section 3 (top-k weighted
 * aggregation at the end); [image] Routed Experts (weighted sum over k) and
 * Shared MLP (added).  y_shared may be NULL when !has_shared. */
moe_status moe_combine(const moe_dims *d, const moe_bf16 *y_sorted, const moe_bf16 *y_shared,
                       const int32_t *inv_perm, const float *topk_w, moe_bf16 *out, void *stream);

/* Steps a3-a9 from a given routing, with stacked fused gate/up weights: the
 * shape of the fused-MoE call of [image] ("flashinfer" path: the flattened
 * tokens, the top-k expert indices and routing weights, and the expert
 * weights stacked along an expert dimension, [E, 2I, H] gate/up and
 * [E, H, I] down, handed to one fused kernel chain).  Runs moe_permute,
 * the grouped expert FFN and moe_combine on `stream`; intermediates in `ws`.
 *   hidden      [T, H] bf16 (input)
 *   topk_idx    [T, top_k] int32 expert of each slot, in [0, E) (input)
 *   topk_w      [T, top_k] fp32 combine weight of each slot (input)
 *   w_gate_up   [E, 2I, H] bf16: rows [0, I) of expert e are its gate
 *               projection, rows [I, 2I) its up projection (input)
 *   w_down      [E, H, I] bf16 (input)
 *   ws_gate_up  [2 * I_shared, H] bf16, gate rows then up rows, and
 *   ws_down     [H, I_shared] bf16: the shared expert (NULL when !has_shared)
 *   out         [T, H] bf16 (output)
 * The results equal moe_permute + moe_expert_ffn + moe_combine on the same
 * weights held as separate w_gate / w_up tensors, bit for bit.  Errors as for
 * moe_permute and moe_expert_ffn (an index outside [0, E) sets
 * MOE_DEVERR_INDEX in the workspace error word). */
moe_status moe_fused_moe(const moe_dims *d, const moe_bf16 *hidden, const int32_t *topk_idx, const float *topk_w,
                         const moe_bf16 *w_gate_up, const moe_bf16 *w_down, const moe_bf16 *ws_gate_up,
                         const moe_bf16 *ws_down, moe_bf16 *out, void *ws, size_t ws_bytes, void *stream);

/* ------------------------------------------------------------------ FP8
 * FP8 expert weights ([case] lists W8A8 quantised deployments and quantises
 * inside the FusedMoE chain, but fixes no format).  Reading: every expert matrix row (an output feature) is stored as
 * OCP E4M3 codes plus one fp32 scale, scale = max|row| / 448 (1 for a zero
 * row), code = E4M3 round-to-nearest-even of w / scale, saturated at 448.  The
 * layer uses value(code) * scale as the weight: the expert kernel feeds the
 * code values (exact in bf16) to the MMAs and multiplies each row's fp32
 * accumulator by its scale.  Activations stay bf16 (weight-only quantisation:
 * it halves the weight bytes that bound decode). */
typedef struct {
  const uint8_t *gate, *up;                 /* [E, I, H] E4M3 codes */
  const uint8_t *down;                      /* [E, H, I] */
  const float *gate_scale, *up_scale;       /* [E, I] fp32, one per row */
  const float *down_scale;                  /* [E, H] */
  const uint8_t *s_gate, *s_up;             /* shared expert [I_shared, H] (unused when !has_shared) */
  const uint8_t *s_down;                    /* [H, I_shared] */
  const float *s_gate_scale, *s_up_scale;   /* [I_shared] */
  const float *s_down_scale;                /* [H] */
} moe_fp8_experts;

/* Quantise a bf16 matrix [rows, cols] (cols a multiple of 8) row by row:
 * codes [rows, cols] uint8 and scales [rows] fp32 as described above.  Pointers
 * 16-byte aligned (scales 4-byte).  Async on `stream`. */
moe_status moe_quantize_fp8_rows(const moe_bf16 *src, int64_t rows, int cols, uint8_t *codes, float *scales,
                                 void *stream);

/* moe_expert_ffn with FP8 expert weights (all pointers in *w 16-byte aligned).
 * The FP8 kernel runs tiles of at most 128 tokens; results, layouts and errors
 * as for moe_expert_ffn. */
moe_status moe_expert_ffn_fp8(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                              const int32_t *offsets, const moe_fp8_experts *w, moe_bf16 *y_sorted,
                              moe_bf16 *y_shared, void *ws, size_t ws_bytes, void *stream);

/* moe_layer_forward with FP8 expert weights: moe_route, moe_permute,
 * moe_expert_ffn_fp8, moe_combine on `stream`, intermediates in `ws`. */
moe_status moe_layer_forward_fp8(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                                 const float *expert_bias, const moe_fp8_experts *w, moe_bf16 *out, void *ws,
                                 size_t ws_bytes, void *stream);

/* W8A8: FP8 expert weights (moe_fp8_experts, as above) AND FP8 activations,
 * multiplied on the tensor cores' 8-bit path.  [case] section 3 quantises the
 * activation right before the down GEMM in its W8A8 deployments; the pages fix
 * no format.  Reading: every activation matrix feeding an expert GEMM is
 * quantised per row by the weight rule (E4M3, scale = max|row| / 448, codes
 * nearest-even of value / scale) from its own values at run time -- the hidden
 * state per token before the gate/up GEMM, and the bf16 SiLU(gate) * up
 * activation per routed slot (per token for the shared expert) once the
 * gate/up GEMM has produced the whole row, before the down GEMM reads it (the
 * codes and row scales are kept in the workspace).  Each output element is
 * (sum of code products) * row scale * column scale, accumulated in fp32.  The
 * router stays fp32.
 *   Shapes: H, I and I_shared multiples of 128 (else MOE_ERR_UNSUPPORTED).
 *   moe_expert_ffn_w8a8: arguments and results as for moe_expert_ffn_fp8; it
 *   first quantises `hidden` into the workspace, then runs the expert kernel.
 *   moe_layer_forward_w8a8: quantisation of `hidden`, moe_route, moe_permute,
 *   the W8A8 expert kernel and moe_combine on `stream`, intermediates in `ws`. */
moe_status moe_expert_ffn_w8a8(const moe_dims *d, const moe_bf16 *hidden, const int32_t *perm,
                               const int32_t *offsets, const moe_fp8_experts *w, moe_bf16 *y_sorted,
                               moe_bf16 *y_shared, void *ws, size_t ws_bytes, void *stream);
moe_status moe_layer_forward_w8a8(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                                  const float *expert_bias, const moe_fp8_experts *w, moe_bf16 *out, void *ws,
                                  size_t ws_bytes, void *stream);

/* The whole layer (a1-a9) chained on `stream` with programmatic dependent
 * launch; every intermediate lives in `ws`.  Arguments as above; out [T, H] bf16. */
moe_status moe_layer_forward(const moe_dims *d, const moe_bf16 *hidden, const float *router_w,
                             const float *expert_bias, const moe_bf16 *w_gate, const moe_bf16 *w_up,
                             const moe_bf16 *w_down, const moe_bf16 *ws_gate, const moe_bf16 *ws_up,
                             const moe_bf16 *ws_down, moe_bf16 *out, void *ws, size_t ws_bytes,
                             void *stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
