/*
 * libmoe — a fused Mixture-of-Experts layer (forward and backward) for one
 * GB300 GPU (sm_103a).
 *
 * The layer is the one Prime Mega MoE trains with (Prime Intellect's fused MoE
 * kernel, which adds a fused and overlapped backward pass to DeepSeek's
 * forward-only Mega MoE): a router picks top_k of E experts per token, the
 * tokens are dispatched to their experts, every expert is a gated SwiGLU
 * feed-forward block without bias, and the expert outputs are combined with
 * the router weights ("A Magia da Fusão" and "Detalhes Técnicos Rápidos" on
 * bitsgeniais.com.br/?p=10788; "Qué se ha publicado" on ai-daily-news.org;
 * "Prime Mega MoE: kernel fuso per l'addestramento MoE" on roccomilluzzo.it).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * - All arrays live in device memory, are row-major and contiguous, and are
 *   allocated and freed by the caller.  The library never allocates or frees
 *   device memory; its only host-side state is a per-device cache of launch
 *   attributes.
 * - bf16 arrays hold bfloat16 bit patterns (moe_bf16_t).
 * - Shapes: x, y, dY, dx [T, H]; W_r, dW_r [H, E]; W_gate, W_up, dW_gate,
 *   dW_up [E, H, F]; W_down, dW_down [E, F, H]; logits [T, E];
 *   topk_idx, topk_w, slot_row [T, top_k]; counts [E]; offsets [E + 1];
 *   perm_token [T * top_k].
 * - Every call validates its arguments on the host and returns a status at
 *   once; the GPU work is then queued on `stream` and runs asynchronously.
 *   A device-side failure (a bounded wait that ran out) is recorded in a
 *   status word at the start of the workspace and read with
 *   moe_get_device_status.  Kernels never trap.
 * - Shape limits (the pages' constraints plus this library's own): H a
 *   multiple of 256 and F a multiple of 128 ("Detalhes Técnicos Rápidos"),
 *   1 <= E <= 256, 1 <= top_k <= min(E, 16), 1 <= T, T * top_k < 2^31.
 *   A violation returns MOE_ERR_UNSUPPORTED_SHAPE.
 * - The GPU must be sm_103 (GB300); otherwise MOE_ERR_UNSUPPORTED_DEVICE.
 */
#ifndef LIBMOE_MOE_H
#define LIBMOE_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t moe_bf16_t;               /* bfloat16 bit pattern */
typedef struct CUstream_st* moe_stream_t;  /* the same handle as cudaStream_t */

/* Arithmetic of the six expert GEMMs ("Supporto di precisione" on
 * roccomilluzzo.it): BF16 everywhere; MXFP8 everywhere (E4M3 elements with an
 * E8M0 scale per 32 elements along each GEMM's reduction dimension); or BF16
 * forward with an MXFP8 backward.  Router GEMMs are BF16 in every mode. */
typedef enum {
  MOE_BF16 = 0,
  MOE_MXFP8 = 1,
  MOE_FP8_BWD = 2
} moe_precision_t;

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,          /* null pointer, bad flag or precision  */
  MOE_ERR_UNSUPPORTED_SHAPE = 2,    /* see the shape limits above           */
  MOE_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes below moe_workspace_size    */
  MOE_ERR_CUDA = 4,                 /* a CUDA runtime call failed           */
  MOE_ERR_TIMEOUT = 5,              /* a device-side bounded wait ran out   */
  MOE_ERR_UNSUPPORTED_DEVICE = 6,   /* not an sm_103 GPU                    */
  MOE_ERR_NOT_IMPLEMENTED = 7       /* reserved: a feature this library version lacks */
} moe_status_t;

/* flags */
#define MOE_FLAG_SYNC_CHECK     0x1u  /* synchronise after every kernel and report
                                         launch/runtime errors (debugging aid)   */
#define MOE_FLAG_TEST_TIMEOUT   0x2u  /* test hook: the first grouped GEMM of the
                                         call waits on a barrier that is never
                                         signalled, with a 20 ms limit, so the
                                         timeout path can be exercised; the call
                                         then reports MOE_ERR_TIMEOUT through
                                         moe_get_device_status                   */
#define MOE_FLAG_CTA_PAIRS_OFF  0x4u  /* run every expert GEMM on single-CTA 128-row
                                         tiles                                    */
#define MOE_FLAG_CTA_PAIRS_ON   0x8u  /* use CTA-pair 256-row tiles (cta_group::2)
                                         wherever the shape allows, the MXFP8
                                         GEMMs included (block-scaled pairs; the
                                         MXFP8 down dgrad stays single-CTA); by
                                         default, when experts average >= 512
                                         rows, pairs run every bf16 expert GEMM,
                                         and from 256 rows the two bf16 dgrads
                                         (the down dgrad when F is a multiple of
                                         256), and the MXFP8 GEMMs run single-CTA */
#define MOE_FLAG_RECOMPUTE      0x10u /* activation checkpointing (full activation
                                         checkpointing is the training setting of
                                         the end-to-end runs in "Os Números..." on
                                         bitsgeniais.com.br): ctx keeps only the
                                         routing and permutation; the dispatched
                                         input and the pre-activations h live in
                                         the forward workspace instead, and
                                         moe_backward dispatches x again and
                                         recomputes h with the gate/up GEMM (in
                                         the forward's precision) before the
                                         backward GEMMs.  ctx_bytes shrinks by
                                         h, (T*top_k + 64*E) * 2F * 2 bytes, and
                                         x: x_perm, (T*top_k + 64*E) * H * 2
                                         bytes, or in mxfp8 its E4M3 copy along
                                         the tokens with the scales; forward and
                                         backward must both be given the flag     */

typedef struct {
  int64_t T;           /* tokens                                   */
  int32_t H;           /* hidden size (multiple of 256)            */
  int32_t F;           /* expert FFN width (multiple of 128)       */
  int32_t E;           /* experts                                  */
  int32_t top_k;       /* experts per token                        */
  int32_t precision;   /* moe_precision_t                          */
  uint32_t flags;      /* MOE_FLAG_*                               */
  int32_t max_sms;     /* SM budget: 0 = every SM of the device;
                          else the persistent kernels launch at most
                          this many CTAs (one per SM), leaving the
                          other SMs to work on other streams.  The
                          counterpart of reserving SMs for
                          communication ("Detalhes Técnicos
                          Rápidos" on bitsgeniais.com.br).  CTA
                          pairs need at least 2; below that every
                          GEMM runs single-CTA tiles.  Results are
                          the same for every budget except dW_r,
                          whose split-K depth follows the budget
                          (summation order only).  Must be >= 0. */
  const void* prepared_weights; /* MXFP8 and FP8_BWD: NULL, or a buffer
                          written by moe_prepare_weights for these
                          weights; the MXFP8 GEMMs then read it
                          instead of quantising W_gate, W_up and
                          W_down in every call.  Ignored for BF16.
                          256-byte aligned. */
} moe_config_t;

/* Bytes of device memory each call needs from the caller:
 *   *fwd_ws   — scratch of moe_forward (also enough for moe_route),
 *   *ctx_bytes — the context moe_forward writes and moe_backward reads,
 *   *bwd_ws   — scratch of moe_backward.
 * Any output pointer may be NULL.  Workspaces must be 256-byte aligned. */
moe_status_t moe_workspace_size(const moe_config_t* cfg, size_t* fwd_ws,
                                size_t* ctx_bytes, size_t* bwd_ws);

/* Router and permutation only: the routing half of the forward pass.
 *   logits[t,e] = sum_h x[t,h] W_r[h,e] + logit_bias[e]   (fp32; optional out)
 *   topk_idx[t,:] = the top_k experts by logit, largest first, equal logits
 *                   ordered by lower expert id;
 *   topk_w[t,j] = softmax over all E experts, renormalised over the selected
 *                 top_k (fp32);
 *   counts[e] = tokens routed to e; offsets = exclusive prefix sum of counts
 *               (offsets[E] = T * top_k);
 *   perm_token[r] = token of row r of the expert-major permuted layout
 *                   (ascending token within an expert);
 *   slot_row[t,j] = row of (t, j) in that layout.
 * logit_bias [E] fp32 and logits may be NULL.  Every integer output is
 * deterministic.  ws: at least fwd_ws bytes.
 * Non-finite inputs: a NaN logit (for instance from a NaN or Inf in a row of
 * x) ranks as -inf in the selection, so every slot still gets a valid expert
 * id; a token whose logits are all NaN or -inf is routed to experts
 * 0 .. top_k-1 with NaN weights, and its outputs (and every weight gradient
 * it reaches) are NaN, while other tokens' results are unaffected.  Should an
 * expert id outside [0, E) ever reach the permutation, that (token, slot) is
 * skipped and the status word records MOE_ERR_INVALID_ARG (moe_get_device_status);
 * no kernel indexes with it. */
moe_status_t moe_route(const moe_config_t* cfg, const moe_bf16_t* x, const moe_bf16_t* W_r,
                       const float* logit_bias, float* logits, int32_t* topk_idx,
                       float* topk_w, int32_t* counts, int32_t* offsets,
                       int32_t* perm_token, int32_t* slot_row, void* ws, size_t ws_bytes,
                       moe_stream_t stream);

/* Forward pass: y[t] = sum_j topk_w[t,j] * (silu(x_t W_gate[e]) * (x_t W_up[e])) W_down[e],
 * e = topk_idx[t,j] (y in bf16, fp32 accumulation).  Writes ctx (routing,
 * permutation, the dispatched input and the pre-activations) for moe_backward;
 * ctx must stay unmodified until the matching backward call.  logit_bias may
 * be NULL.  ws: at least fwd_ws bytes; ctx: at least ctx_bytes. */
moe_status_t moe_forward(const moe_config_t* cfg, const moe_bf16_t* x, const moe_bf16_t* W_r,
                         const float* logit_bias, const moe_bf16_t* W_gate,
                         const moe_bf16_t* W_up, const moe_bf16_t* W_down, moe_bf16_t* y,
                         void* ctx, void* ws, size_t ws_bytes, moe_stream_t stream);

/* Backward pass: the exact vector-Jacobian product of moe_forward at dY
 * (routing indices get no gradient).  Outputs dx, dW_r, dW_gate, dW_up and
 * dW_down in bf16 (fp32 accumulation); they are overwritten, not accumulated.
 * An expert that received no token gets exactly-zero weight gradients.
 * The arguments x, W_r, W_gate, W_up, W_down and cfg must be those of the
 * forward call that wrote ctx.  ws: at least bwd_ws bytes. */
moe_status_t moe_backward(const moe_config_t* cfg, const moe_bf16_t* x, const moe_bf16_t* W_r,
                          const moe_bf16_t* W_gate, const moe_bf16_t* W_up,
                          const moe_bf16_t* W_down, const void* ctx, const moe_bf16_t* dY,
                          moe_bf16_t* dx, moe_bf16_t* dW_r, moe_bf16_t* dW_gate,
                          moe_bf16_t* dW_up, moe_bf16_t* dW_down, void* ws, size_t ws_bytes,
                          moe_stream_t stream);

/* MXFP8 weight preparation ("Supporto di precisione" on roccomilluzzo.it
 * names MXFP8 training; the weights change once per optimizer step, however
 * many micro-batches share them).  Quantises W_gate, W_up and W_down (bf16,
 * the layouts above) into wq, in every orientation the MXFP8 GEMMs read:
 * W_gate / W_up along H (forward) and along F (backward), W_down along F
 * (forward) and along H (backward); E4M3 elements with E8M0 scale atoms, the
 * same bytes the calls would compute themselves.  Point
 * cfg->prepared_weights at wq for the forward and backward calls that use
 * these weights; prepare again after the weights change.  cfg->precision
 * must be MOE_MXFP8 or MOE_FP8_BWD.  *bytes receives the size wq needs. */
moe_status_t moe_prepared_weights_size(const moe_config_t* cfg, size_t* bytes);
moe_status_t moe_prepare_weights(const moe_config_t* cfg, const moe_bf16_t* W_gate,
                                 const moe_bf16_t* W_up, const moe_bf16_t* W_down, void* wq,
                                 size_t wq_bytes, moe_stream_t stream);

/* moe_backward for gradient accumulation over micro-batches (the end-to-end
 * runs of "Os Números..." on bitsgeniais.com.br train on micro-batches of
 * 16,384-token sequences): the weight gradients are ADDED into caller-owned
 * fp32 buffers, gW_r [H,E] += dW_r, gW_gate / gW_up [E,H,F] += dW_gate /
 * dW_up, gW_down [E,F,H] += dW_down, straight from the fp32 accumulators
 * (no bf16 rounding of the increment).  dx is written in bf16 as in
 * moe_backward.  An expert that received no token leaves its slices of the
 * buffers unchanged.  The buffers must be 16-byte aligned, hold finite
 * values, and not overlap each other or any input.  Same ctx, cfg, ws and
 * error behaviour as moe_backward. */
moe_status_t moe_backward_accumulate(const moe_config_t* cfg, const moe_bf16_t* x,
                                     const moe_bf16_t* W_r, const moe_bf16_t* W_gate,
                                     const moe_bf16_t* W_up, const moe_bf16_t* W_down,
                                     const void* ctx, const moe_bf16_t* dY, moe_bf16_t* dx,
                                     float* gW_r, float* gW_gate, float* gW_up,
                                     float* gW_down, void* ws, size_t ws_bytes,
                                     moe_stream_t stream);

/* Dense bf16 GEMM on the same tcgen05 engine: D[M,N] = sum_k A(m,k) B(n,k),
 * fp32 accumulation, D written as fp32 row-major [M, N] (ldd = N).
 *   a_kmajor != 0: A is [M, K] row-major; else A is [K, M] row-major.
 *   b_kmajor != 0: B is [N, K] row-major; else B is [K, N] row-major.
 * Limits: M >= 1, K >= 1, N a multiple of 256, and the row length of each
 * operand a multiple of 8 elements (16-byte rows).  ws holds the status word
 * (at least 256 bytes). */
moe_status_t moe_gemm_bf16(int64_t M, int64_t N, int64_t K, const moe_bf16_t* A, int a_kmajor,
                           const moe_bf16_t* B, int b_kmajor, float* D, void* ws,
                           size_t ws_bytes, moe_stream_t stream);

/* Routing without a caller-provided workspace.
 *
 * Same computation and outputs as moe_route, for callers that cannot call
 * cudaMalloc: hosts whose device memory is owned entirely by another
 * allocator or runtime (a framework's memory pool, a fixed budget carved out
 * at start-up), and plain C callers that have no device allocator of their
 * own.  The pages describe no such call; it has no counterpart there.
 *
 * Its scratch is a fixed array of MOE_NOALLOC_SCRATCH_BYTES inside the
 * library; every GPU that loads the library holds that array until the
 * process exits.  A configuration that needs more scratch than that is
 * rejected with MOE_ERR_WORKSPACE_TOO_SMALL before anything is queued.  The
 * scratch takes 2*E*H bytes (the router weight transposed), about
 * 4*(3*top_k + 2*E/128) bytes per token (the permuted-row maps and the
 * per-tile expert histograms) and 512*E bytes of segment padding: at E = 128,
 * H = 4096, top_k = 8 that allows at most T = 69,904 tokens.
 * The call allocates no device memory and calls no allocating routine.
 *
 * The first call on a device looks up the array's device address (once per
 * device and context, with that device current); make that first call before
 * any stream capture.  All calls share the one array and it keeps the last call's
 * contents: calls whose GPU work overlaps (on different streams, or from
 * different host threads) race on it and must be serialised by the caller.
 * device_status (nullable, 4 bytes of device memory) receives the call's
 * device status code (MOE_OK or MOE_ERR_TIMEOUT) once the work has run. */
#define MOE_NOALLOC_SCRATCH_BYTES (8u << 20)
moe_status_t moe_route_noalloc(const moe_config_t* cfg, const moe_bf16_t* x,
                               const moe_bf16_t* W_r, const float* logit_bias, float* logits,
                               int32_t* topk_idx, float* topk_w, int32_t* counts,
                               int32_t* offsets, int32_t* perm_token, int32_t* slot_row,
                               int32_t* device_status, moe_stream_t stream);

/* Dense MXFP8 GEMM on the block-scaled engine: quantises A [M, K] and B [N, K]
 * (bf16, row-major) to E4M3 with an E8M0 scale per 32 elements along K (the
 * OCP MX rule of the precision modes above), then D[M, N] (fp32, row-major) =
 * sum_k A_q(m, k) B_q(n, k) with fp32 accumulation.  Limits: M >= 1; N and K
 * multiples of 128.  Workspace: call with ws = NULL to receive the size in
 * *ws_bytes; otherwise *ws_bytes is the workspace size (256-byte aligned).
 * Used to test the engine's MXFP8 path in isolation: N a multiple of 256 runs
 * the CTA-pair kernel (256 x 256 tiles, block-scaled cta_group::2 MMAs),
 * other N the single-CTA one (128 x 128 tiles). */
moe_status_t moe_gemm_mxfp8(int64_t M, int64_t N, int64_t K, const moe_bf16_t* A,
                            const moe_bf16_t* B, float* D, void* ws, size_t* ws_bytes,
                            moe_stream_t stream);

/* Reads the device status word of a workspace after the work queued on
 * `stream` has finished (this call synchronises the stream).  Returns
 * MOE_OK, MOE_ERR_TIMEOUT (a bounded wait ran out), MOE_ERR_INVALID_ARG (a
 * device-side index check failed: an id or row outside its array was
 * skipped instead of used), or MOE_ERR_CUDA if the read itself failed. */
moe_status_t moe_get_device_status(const void* ws, moe_stream_t stream);

/* Human-readable name of a status code (static string). */
const char* moe_status_string(moe_status_t status);

/* Per-kernel timing with CUDA events recorded on the launch stream around
 * every kernel the library launches while enabled.  moe_profile_read copies
 * up to `cap` records (name, launches, total milliseconds) and returns the
 * number of distinct kernels; it synchronises the recorded events.  Reading
 * resets the counters. */
void moe_profile_enable(int on);
int moe_profile_read(const char** names, int64_t* launches, double* total_ms, int cap);

/* Restricts the per-kernel timing to the launches labelled `name` (the names
 * moe_profile_read returns), so that the other launches run without events
 * between them; NULL times every launch again.  The string is copied. */
void moe_profile_select(const char* name);

/* Number of kernel launches the library has made in this process. */
int64_t moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* LIBMOE_MOE_H */
