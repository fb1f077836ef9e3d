/*
 * moe.h -- C ABI of the sparse token-choice Mixture-of-Experts FFN layer
 * (forward pass) for NVIDIA B300 (sm_103a), library libmoe_b300.so.
 *
 * The layer (notation of the pages): for each token row x (length d),
 *   z      = x . W_g (+ beta)                    router logits, float32, N experts
 *   S_k(x) = the k experts with the largest selection score
 *   g_i    = softmax of z over S_k      (MOE_GATE_SOFTMAX_TOPK), or
 *            s_i / sum_{j in S_k} s_j with s = sigmoid(z), chosen on s + b
 *                                               (MOE_GATE_SIGMOID_BIAS)
 *   y      = sum_{i in S_k, kept} g_i Expert_i(x)  (+ SharedExpert(x))
 *   Expert(x) = W2 (SiLU(W1 x) * W3 x)  (MOE_ACT_SWIGLU) or W2 ReLU(W1 x) (MOE_ACT_RELU)
 * Sources: "Lecture29" (CS25 lecture 29 notes, Mixtral), sections "Top-two
 * routing: from logits to weighted expert output", "A dense Transformer layer"
 * (SwiGLU expert) and "Inference load balance" (capacity); "Chapter 19: MoE"
 * (awesome-ai-roadmap) 19.3.2 (top-k softmax = renormalised full softmax),
 * 19.3.3 (f_i, P_i), 19.3.4 (DeepSeek-V3 selection-only bias), 19.6.1
 * (capacity, dropped overflow); "Stanford CS336 lecture 4: Mixture of Experts",
 * sections 5, 6 (shared expert), 9 (N sum f_i P_i), 10 (dropped token -> zero
 * expert output, residual passes), 11 (float32 router); Shazeer et al. 2017
 * notes (ReLU expert, gate matrix d x n).
 *
 * Conventions (all entry points):
 *  - Every tensor argument is a DEVICE pointer to caller-owned memory on the
 *    current CUDA device; the library never allocates device memory.  Scratch
 *    comes from a caller-provided workspace `ws` of moe_workspace_size() bytes
 *    (256-byte aligned).  The workspace also holds the device status word (and,
 *    after it, a counter the grouped GEMM resets before each launch).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  All work
 *    is enqueued asynchronously on it; no call synchronises except
 *    moe_get_device_status.  Results are deterministic: the same inputs give
 *    bitwise identical outputs.
 *  - Layouts are row-major:
 *      x       [T, d]        activations, dtype cfg->dtype
 *      Wg      [d, N]        float32 router weight (logits = x . Wg)
 *      w1, w3  [N, F, d]     expert e's W1, W3 as F x d ("W1 x" maps d -> F)
 *      w2      [N, d, F]     expert e's W2 as d x F
 *      sw1, sw3 [Fs, d], sw2 [d, Fs]   the shared expert (Fs = cfg->shared_ffn)
 *    bf16 tensors hold raw bfloat16 values (uint16 storage).
 *  - Alignment: every pointer 16-byte aligned; d and ffn (and shared_ffn) a
 *    multiple of 8 (bf16) or 4 (float32).  Otherwise MOE_ERR_UNSUPPORTED.
 *  - Limits: 1 <= N <= 256, 1 <= k <= min(N, 8), T >= 0 (T = 0 is a no-op),
 *    d, ffn <= 65536.  Otherwise MOE_ERR_UNSUPPORTED or MOE_ERR_INVALID_ARG.
 *  - Errors: argument errors are returned synchronously and launch nothing.
 *    Errors found on the device (non-finite logits, a pipeline wait that ran
 *    past its time limit) are recorded in the workspace status word, read by
 *    moe_get_device_status.  Kernels never trap.
 *  - The output is the MoE branch only; the residual add is the caller's.
 */
#ifndef MOE_B300_H
#define MOE_B300_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null pointer, negative size, bad enum */
  MOE_ERR_UNSUPPORTED = 2,  /* shape or alignment outside the limits above */
  MOE_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  MOE_ERR_NONFINITE = 4,    /* device: a router logit was NaN or infinite */
  MOE_ERR_TIMEOUT = 5,      /* device: a pipeline wait exceeded its limit */
  MOE_ERR_BOUNDS = 6        /* device: an index left its range */
} moe_status;

/* MOE_GATE_SOFTMAX_TOPK: softmax over the k selected logits (Mixtral).
 * MOE_GATE_SIGMOID_BIAS: sigmoid affinities, chosen on s + b, weights s / sum s (DeepSeek-V3).
 * MOE_GATE_SOFTMAX_FULL: softmax over all N logits kept on the top-k, not
 *   renormalised (DeepSeek v1; CS336 lecture 4, section 5 pseudocode). */
typedef enum { MOE_GATE_SOFTMAX_TOPK = 0, MOE_GATE_SIGMOID_BIAS = 1, MOE_GATE_SOFTMAX_FULL = 2 } moe_gate;
typedef enum { MOE_ACT_RELU = 0, MOE_ACT_SWIGLU = 1 } moe_act;
typedef enum { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype;
/* MOE_ROUTING_TOKEN_CHOICE: each token picks its top-k experts (the gates above).
 * MOE_ROUTING_EXPERT_CHOICE: each expert picks the `capacity` tokens with the
 *   largest scores, scores = softmax over all N experts of each token's logits;
 *   the gate of (token, expert) is that score; k and gate are ignored. */
typedef enum { MOE_ROUTING_TOKEN_CHOICE = 0, MOE_ROUTING_EXPERT_CHOICE = 1 } moe_routing;

typedef struct {
  int32_t T;          /* tokens */
  int32_t d;          /* hidden size */
  int32_t N;          /* routed experts */
  int32_t k;          /* experts per token */
  int32_t ffn;        /* routed expert hidden width F */
  int32_t shared_ffn; /* shared expert hidden width, 0 = no shared expert */
  int32_t gate;       /* moe_gate */
  int32_t act;        /* moe_act */
  int32_t dtype;      /* moe_dtype of x, weights, out */
  int32_t capacity;   /* per-expert capacity C, <= 0 = unlimited (see moe_capacity);
                         expert choice: tokens per expert (>= 1, capped at T) */
  int32_t routing;    /* moe_routing */
} moe_config;

/* Byte offsets of the intermediates inside the workspace (for inspection after
 * moe_layer_forward; every offset is 256-byte aligned). */
typedef struct {
  size_t status;         /* int32 status word */
  size_t logits;         /* float [T, N] */
  size_t topk_idx;       /* int32 [T, k] (token choice) */
  size_t topk_w;         /* float [T, k]; expert choice: the scores [T, N] */
  size_t counts_routed;  /* int32 [N] */
  size_t counts_kept;    /* int32 [N] */
  size_t offsets;        /* int32 [N + 1] */
  size_t dest_row;       /* int32 [T, k], -1 = dropped; expert choice: [T, N], -1 = not chosen */
  size_t src_token;      /* int32 [R], R = T * k (token choice) or N * min(C, T) (expert choice) */
  size_t x_perm;         /* dtype [R, d] */
  size_t h;              /* dtype [R, F]  expert hidden activations */
  size_t y_perm;         /* bf16 or float [R, d]  expert outputs */
  size_t h_shared;       /* dtype [T, Fs] */
  size_t y_shared;       /* bf16 or float [T, d] */
  size_t scratch;        /* internal scratch */
  size_t total;          /* = moe_workspace_size */
} moe_ws_layout;

/* Human-readable name of a status code (static string, never NULL). */
MOE_API const char *moe_status_string(int status);

/* C = ceil(alpha * T * k / N) computed exactly, alpha taken as the exact value
 * of the double (Lecture29, "Inference load balance": C = ceil(alpha T k / E);
 * Chapter 19, 19.6.1).  alpha > 0, T >= 0, k >= 1, N >= 1; C written to *C. */
MOE_API int moe_capacity(double alpha, int32_t T, int32_t k, int32_t N, int32_t *C);

/* Workspace bytes needed by any call below for this config. */
MOE_API int moe_workspace_size(const moe_config *cfg, size_t *bytes);
MOE_API int moe_workspace_layout(const moe_config *cfg, moe_ws_layout *layout);

/* Router: logits z = x . Wg (+ logit_bias), top-k with ties to the lower expert
 * index, and the gate weights (Lecture29 "Top-two routing"; Chapter 19, 19.3.2
 * and 19.3.4).  logit_bias [N] (float, may be NULL) is added to every logit;
 * sel_bias [N] (float, sigmoid gate only, may be NULL) shifts the selection
 * score s + b but not the weights.  Outputs: logits [T, N] float, topk_idx
 * [T, k] int32 ordered by (selection score desc, index asc), topk_w [T, k]
 * float (sum to 1 per token).  The sigmoid s is fl32(1/(1+exp(-z))) evaluated
 * in double.  Non-finite logits set MOE_ERR_NONFINITE on the device. */
MOE_API int moe_route(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
              const float *sel_bias, float *logits, int32_t *topk_idx, float *topk_w, void *ws,
              void *stream);

/* Dispatch (Lecture29, "Top-k routing semantics"; "Inference load balance"):
 * counts_routed[e] = assignments to e; counts_kept[e] = min(counts_routed, C);
 * offsets [N+1] = exclusive scan of counts_kept; per expert the first C
 * assignments in ascending token order are kept, at rows offsets[e] + rank;
 * dest_row[t, j] = that row or -1 (dropped); src_token[row] = t; and
 * x_perm[row, :] = x[t, :].  x_perm needs room for T * k rows; rows at or
 * beyond offsets[N] are left untouched.  x_perm may be NULL: then the permuted
 * copy is not made (x is not read; moe_expert_ffn_gather reads x by src_token).
 * A token picks an expert at most once:
 * an id in topk_idx outside [0, N) is skipped and sets MOE_ERR_BOUNDS, an id that
 * repeats an earlier slot of the same token is skipped (not counted, dest_row
 * -1) and sets MOE_ERR_INVALID_ARG, both in the device status word.  Token-choice
 * configs only (MOE_ERR_INVALID_ARG for expert choice). */
MOE_API int moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const void *x, int32_t *counts_routed,
                 int32_t *counts_kept, int32_t *offsets, int32_t *dest_row, int32_t *src_token,
                 void *x_perm, void *ws, void *stream);

/* moe_dispatch without a workspace, for callers that cannot allocate device
 * memory and cannot pass a workspace: typically a plug-in or custom operator in a
 * host program that has already reserved the GPU's memory for its own pool and
 * whose interface hands the operator only its input and output buffers.  The
 * pages describe no such variant; it has no counterpart there.
 * Inputs, outputs and results are exactly those of moe_dispatch, token-choice
 * configs only (MOE_ERR_INVALID_ARG for expert choice, as moe_dispatch).  `status`
 * is an optional device int32 (may be NULL) in which bit MOE_ERR_BOUNDS is set
 * when an expert id is out of range and bit MOE_ERR_INVALID_ARG when a token
 * repeats an expert; the caller clears it.
 * Scratch: a fixed 1 MiB array inside the library (a `static __device__`
 * variable), resident on every GPU that loads the library until the process
 * exits.  It bounds the size: ceil(T / 128) * N <= 131072 (for example T up to
 * 65536 with N = 256), else MOE_ERR_UNSUPPORTED.  Every call overwrites every
 * scratch entry it reads, so nothing needs clearing between calls.
 * The first call on each device looks up the array's device address (with that
 * device current); make that first call before any stream capture.  All calls
 * share the one array: calls whose executions overlap on the GPU (two streams,
 * two host threads) race on it and give wrong results; serialise them. */
MOE_API int moe_dispatch_noalloc(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                                 int32_t *counts_routed, int32_t *counts_kept, int32_t *offsets,
                                 int32_t *dest_row, int32_t *src_token, void *x_perm, int32_t *status,
                                 void *stream);

/* Routed experts over the permuted rows: for each expert e, rows
 * [offsets[e], offsets[e+1]) of x_perm go through Expert_e; results in y_perm
 * (same rows).  y_perm is bf16 for bf16 configs, float for float32 configs.
 * The hidden activations (bf16 / float) live in the workspace. */
MOE_API int moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets, const void *w1,
                   const void *w3, const void *w2, void *y_perm, void *ws, void *stream);

/* moe_expert_ffn reading its input rows straight from x: row r of expert e's
 * group (offsets[e] <= r < offsets[e+1]) is x[src_token[r], :], as moe_dispatch
 * would have copied it into x_perm; y_perm as moe_expert_ffn.  bf16 configs only
 * (MOE_ERR_UNSUPPORTED otherwise).  The rows are fetched by TMA row gathers
 * (four indexed rows of x per copy) straight into the tensor cores' operand tiles.
 * A src_token entry outside [0, T) sets MOE_ERR_BOUNDS in the device status word;
 * that row's output is then unspecified (the other rows are unaffected).  It
 * needs no x_perm buffer, at a cost: every N tile of the gate/up GEMM re-gathers
 * its rows, four per TMA instruction, and on large groups that instruction rate
 * limits the GEMM (moe_layer_forward copies x into x_perm once instead). */
MOE_API int moe_expert_ffn_gather(const moe_config *cfg, const void *x, const int32_t *src_token,
                                  const int32_t *offsets, const void *w1, const void *w3, const void *w2,
                                  void *y_perm, void *ws, void *stream);

/* The always-on shared expert on every token (CS336 lecture 4, section 6):
 * y_shared [T, d] (bf16 / float) = SharedExpert(x).  Needs cfg->shared_ffn > 0. */
MOE_API int moe_shared_ffn(const moe_config *cfg, const void *x, const void *sw1, const void *sw3,
                   const void *sw2, void *y_shared, void *ws, void *stream);

/* Combine (Lecture29, "Top-two routing": y = sum_i g_i Expert_i(x)):
 * out[t] = y_shared[t] + sum_{j: dest_row[t,j] >= 0} topk_w[t,j] * y_perm[dest_row[t,j]],
 * accumulated in float32 in slot order j = 0..k-1.  y_shared may be NULL.
 * out [T, d] has the config dtype. */
MOE_API int moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *dest_row, const float *topk_w,
                const void *y_shared, void *out, void *stream);

/* The whole layer: route, dispatch, routed experts, shared expert (if
 * cfg->shared_ffn > 0, sw1/sw3/sw2 non-NULL), combine.  Intermediates stay in
 * the workspace at the offsets of moe_workspace_layout.  With
 * cfg->routing == MOE_ROUTING_EXPERT_CHOICE the routing is moe_ec_route's
 * (sel_bias is ignored) and the combine sums over the experts that chose a token. */
MOE_API int moe_layer_forward(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
                      const float *sel_bias, const void *w1, const void *w3, const void *w2,
                      const void *sw1, const void *sw3, const void *sw2, void *out, void *ws,
                      void *stream);

/* Expert-choice routing (Chapter 19, 19.6.1; CS336 lecture 4, section 4):
 * logits [T, N] as in moe_route; scores [T, N] = softmax over the N experts of
 * each token's logits; expert e takes the C = min(cfg->capacity, T) tokens with
 * the largest scores (ties: lower token index), in ascending token order, at rows
 * e*C .. e*C+C-1: src_token [N*C] holds their tokens, dest_row [T, N] the row of
 * (t, e) or -1, offsets [N+1] = e*C.  Needs cfg->routing == MOE_ROUTING_EXPERT_CHOICE
 * and cfg->capacity >= 1; bf16 or float32 x. */
MOE_API int moe_ec_route(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
                         float *logits, float *scores, int32_t *offsets, int32_t *src_token, int32_t *dest_row,
                         void *ws, void *stream);

/* Switch load statistics (Chapter 19, 19.3.3; CS336 lecture 4, section 9;
 * Lecture29, "Myth 3"): f[e] = counts_routed[e] / (T k); P[e] = mean over
 * tokens of the router probability p_e(t) (full softmax of the logits, or
 * s_e / sum_l s_l for the sigmoid gate); summary[0] = N sum_e f_e P_e,
 * summary[1] = imbalance max_e counts_routed / (T k / N), summary[2] = drop
 * rate 1 - sum(counts_kept) / (T k).  All float device pointers; the per-chunk
 * partial sums use the workspace scratch. */
MOE_API int moe_load_stats(const moe_config *cfg, const float *logits, const int32_t *counts_routed,
                   const int32_t *counts_kept, float *f, float *P, float *summary, void *ws, void *stream);

/* Self-check of the device-side wait limit: launches one kernel whose pipeline
 * wait can never complete (an mbarrier nobody arrives on) with the given limit
 * (0 <= limit_ns <= 1e10).  The wait gives up after limit_ns and records
 * MOE_ERR_TIMEOUT in the workspace status word, exactly as a stalled pipeline in
 * any kernel of this library would; the GPU context stays usable.  The pages
 * have no counterpart: this only tests the library's failure handling. */
MOE_API int moe_check_wait_timeout(void *ws, int64_t limit_ns, void *stream);

/* Measurement aid: samples the SM clock while other work runs on other streams.
 * One thread records n pairs (%globaltimer ns, clock64 cycles) into samples
 * [2 n] (device uint64, 8-byte aligned), the i-th at i * interval_ns after the
 * first, sleeping in between; the kernel ends by itself after (n - 1) *
 * interval_ns.  Cycles over nanoseconds between two samples give the SM clock in
 * that interval.  2 <= n <= 2^20, interval_ns >= 1000, (n - 1) * interval_ns <=
 * 1e10, else MOE_ERR_INVALID_ARG.  The pages have no counterpart. */
MOE_API int moe_clock_probe(uint64_t *samples, int n, int64_t interval_ns, void *stream);

/* Backward pass of the layer, bf16 token-choice configs (Chapter 19, 19.6.2: the
 * top-k choice is discrete, so gradients reach the router through the gate weights
 * of the chosen, kept experts only, and each expert through the tokens it
 * processed; dropped assignments get none -- CS336 lecture 4, section 10).
 * Call it after moe_layer_forward on the same inputs with the same forward
 * workspace `fwd_ws`, whose intermediates it reads (logits, top-k, gate weights,
 * dispatch, x_perm, h, y_perm, the shared expert's h).  dout [T, d] bf16 is the
 * gradient of the loss with respect to the layer output.  Outputs, all float32
 * and fully overwritten: dx [T, d], dWg [d, N], dw1 and dw3 [N, F, d], dw2
 * [N, d, F] (dw3 NULL for ReLU experts), dsw1, dsw3 [Fs, d], dsw2 [d, Fs] when
 * cfg->shared_ffn > 0 (else NULL).  The logit and selection biases are inputs,
 * not parameters: no gradient.  Scratch: `bwd_ws` of moe_backward_workspace_size
 * bytes (256-byte aligned). */
MOE_API int moe_backward_workspace_size(const moe_config *cfg, size_t *bytes);
MOE_API int moe_layer_backward(const moe_config *cfg, const void *x, const float *Wg, const void *w1, const void *w3,
                               const void *w2, const void *sw1, const void *sw3, const void *sw2, const void *dout,
                               float *dx, float *dWg, float *dw1, float *dw3, float *dw2, float *dsw1, float *dsw3,
                               float *dsw2, void *fwd_ws, void *bwd_ws, void *stream);

/* Router z-loss (CS336 lecture 4, section 11; Chapter 19, 19.6.2):
 * *z_loss = mean over tokens of (log sum_i exp(logits[t, i]))^2, a device float.
 * Partial sums use the workspace scratch; the result is deterministic. */
MOE_API int moe_router_zloss(const moe_config *cfg, const float *logits, float *z_loss, void *ws, void *stream);

/* DeepSeek-V3 sequence-wise balance loss (Chapter 19, 19.3.4: a small auxiliary
 * loss kept against extreme imbalance inside one sequence; CS336 lecture 4,
 * section 9: the Switch loss of moe_load_stats with its statistics taken over
 * one sequence instead of the batch).  The T tokens form consecutive sequences
 * of seq_len (>= 1; the last may be shorter, a seq_len above T is one sequence);
 * for each, loss_s = N sum_e f_e P_e with f_e = (assignments of the sequence's
 * tokens to e in topk_idx [T, k], before any capacity) / (L k) and P_e the mean
 * router probability of e over its L tokens (as in moe_load_stats for
 * cfg->gate).  *loss (a device float) = the mean of loss_s over the sequences,
 * summed in a fixed order (deterministic).  Token-choice configs only; T >= 1.
 * An index outside [0, N) in topk_idx is skipped and MOE_ERR_BOUNDS is recorded
 * in the workspace status word. */
MOE_API int moe_seq_balance_loss(const moe_config *cfg, const float *logits, const int32_t *topk_idx,
                                 int32_t seq_len, float *loss, void *ws, void *stream);

/* DeepSeek-V3 auxiliary-loss-free balancing step (CS336 lecture 4, section 9;
 * Chapter 19, 19.3.4): for each expert, sel_bias[e] += gamma when
 * counts_routed[e] < T k / N, -= gamma when it is larger, unchanged when equal
 * (compared exactly as counts_routed[e] * N against T * k).  sel_bias [N] float
 * is updated in place on the device. */
MOE_API int moe_bias_update(const moe_config *cfg, const int32_t *counts_routed, float *sel_bias, float gamma,
                            void *stream);

/* FP8 expert weights ("Stanford CS336 lecture 4", the section on compressing
 * sparse MoEs: quantisation lowers the bytes per weight at the cost of scales and
 * a dequantisation step; the pages leave the scheme open).  Weight-only OCP FP8
 * E4M3 with one float32 scale per row of a weight matrix (its output channel):
 * scales[r] = max_c |w[r, c]| / 448 (1 for an all-zero row), q[r, c] = E4M3 of
 * w[r, c] / scales[r], rounded to nearest even and saturated to +-448.
 * moe_quantize_fp8: w [rows, cols] bf16 device -> q [rows, cols] bytes and scales
 * [rows] float32 device; quantise w1 and w3 as [N * F, d], w2 as [N * d, F]. */
MOE_API int moe_quantize_fp8(const void *w, int64_t rows, int32_t cols, uint8_t *q, float *scales, void *stream);

/* moe_expert_ffn / moe_layer_forward with FP8 expert weights: w1q, w3q [N, F, d]
 * and w2q [N, d, F] E4M3 codes (16-byte aligned), w1s, w3s [N, F] and w2s [N, d]
 * their row scales; the result is the layer whose expert weights are q * s
 * (activations, router, shared expert and accumulation as in the bf16 layer).
 * bf16 configs with d and ffn multiples of 16 (else MOE_ERR_UNSUPPORTED); token or
 * expert choice; the shared expert (sw1, sw3, sw2) stays bf16.  The two NaN codes
 * (0x7F, 0xFF) are not valid weights (moe_quantize_fp8 never writes them).  When
 * no group can exceed 64 rows (T, or the capacity, at most 64: decode) the whole
 * expert FFN is one cooperative launch of one CTA per SM in which the weights
 * stream once per group with the tokens as the narrow side of the product (any
 * offsets still give the right result); if the device cannot run a cooperative
 * launch the call returns MOE_ERR_CUDA. */
MOE_API int moe_expert_ffn_fp8(const moe_config *cfg, const void *x_perm, const int32_t *offsets, const uint8_t *w1q,
                               const float *w1s, const uint8_t *w3q, const float *w3s, const uint8_t *w2q,
                               const float *w2s, void *y_perm, void *ws, void *stream);
MOE_API int moe_layer_forward_fp8(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
                                  const float *sel_bias, const uint8_t *w1q, const float *w1s, const uint8_t *w3q,
                                  const float *w3s, const uint8_t *w2q, const float *w2s, const void *sw1,
                                  const void *sw3, const void *sw2, void *out, void *ws, void *stream);

/* Synchronises `stream`, reads and clears the workspace status word, and
 * writes the first device-side error code found (MOE_OK if none) to *status.
 * Returns MOE_ERR_CUDA if the stream itself reports an error. */
MOE_API int moe_get_device_status(void *ws, void *stream, int *status);

#ifdef __cplusplus
}
#endif

#endif /* MOE_B300_H */
