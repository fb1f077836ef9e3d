// Host-side launchers shared between the translation units of libmoe_b300.
// Every launcher enqueues on `stream` and returns a moe_status code.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

int device_sm_count(int device);

// router: logits = x . Wg (+ logit_bias); then top-k + gate weights
int launch_router_logits(const void *x, bool x_bf16, const float *Wg, const float *logit_bias, int T, int d, int N,
                         int splits, float *logits, cudaStream_t s);
// The whole route (logits, top-k, gate) in one launch on the CUDA cores for N = 4 or 8
// (used for float32 activations).
bool router_fused_fits(int T, int d, int N);
int launch_router_fused(const void *x, bool x_bf16, const float *Wg, const float *logit_bias,
                        const float *sel_bias, int T, int d, int N, int k, int gate, float *logits, int32_t *idx,
                        float *w, int *status, cudaStream_t s);
int launch_router_topk(const float *partial, int S, int pstride, const float *logit_bias, float *logits,
                       const float *sel_bias, int T, int N, int k, int gate, int32_t *idx, float *w, int *status,
                       cudaStream_t s);
// tensor-core router (bf16 x): W_g split into bf16 hi+mid+lo, split-K partial sums
int router_tc_npad(int N);
int router_tc_dpad(int d);
int router_tc_max_splits(int T, int d);
int launch_router_tc(const void *x, const float *Wg, int T, int d, int N, uint16_t *wsplit, float *partial,
                     int *splits_out, int *status, cudaStream_t s);

// dispatch
constexpr int kDispatchChunk = 128;  // tokens per histogram / rank chunk
int launch_dispatch(const int32_t *idx, int T, int k, int N, int capacity, int32_t *hist, int32_t *chunk_base,
                    int32_t *counts_routed, int32_t *counts_kept, int32_t *offsets, int32_t *dest_row,
                    int32_t *src_token, int *status, cudaStream_t s);
// Token choice: x_perm[dest_row[t, j]] = x[t] for the kept slots (k <= 32), x read once per token.
int launch_scatter_rows(const void *x, const int32_t *dest_row, int T, int k, int row_bytes, void *x_perm,
                        cudaStream_t s);
int launch_gather_rows(const void *x, const int32_t *src_token, const int32_t *offsets_end, int64_t max_rows,
                       int row_bytes, void *x_perm, cudaStream_t s);

// grouped GEMM on tcgen05 (bf16); mode 0 = SwiGLU (B0 = W1, B1 = W3), 1 = ReLU, 2 = plain.
// pair_tiles: 256-row tiles on CTA pairs (cta_group::2) instead of 128-row tiles on
// single CTAs -- faster when groups hold many rows, wasteful when they are small.
int tc_grouped_gemm(int mode, const void *A, int64_t a_rows, int K, const void *B0, const void *B1,
                    int64_t b_rows_total, int b_rows_per_group, const int32_t *offsets, int G, int M, int n_out,
                    void *out, int *status, bool pair_tiles, cudaStream_t stream);
// the same with A gathered: row r of A is row src_token[r] of x [x_rows, K] (forward modes)
int tc_grouped_gemm_gather(int mode, const void *x, int64_t x_rows, const int32_t *src_token, int64_t rows, int K,
                           const void *B0, const void *B1, int64_t b_rows_total, int b_rows_per_group,
                           const int32_t *offsets, int G, int n_out, void *out, int *status, bool pair_tiles,
                           cudaStream_t stream);
// The forward GEMM (modes 0-2) with FP8 E4M3 weights Q [G * b_rows, K] bytes and
// per-row float32 scales S [G * b_rows]: out = EPI(S[n] * sum_k A[r, k] Q[n, k]).
// FP8 expert FFN: the two GEMMs for groups of any size, with tokens on the M side.
int tc_grouped_gemm_fp8(int mode, const void *A, int64_t a_rows, int K, const uint8_t *Q0, const float *S0,
                        const uint8_t *Q1, const float *S1, int64_t b_rows_total, int b_rows_per_group,
                        const int32_t *offsets, int G, int M, int n_out, void *out, int *status, cudaStream_t stream);
// The whole FP8 expert FFN in one launch when no group exceeds 64 rows (decode):
// weights on the M side, token tiles of fp8_decode_tile_rows(max_group_rows) rows
// (0: not a decode shape).  dep: G ints of scratch.
inline int fp8_decode_tile_rows(int max_group_rows) {
  return max_group_rows < 0 ? 0 : max_group_rows <= 16 ? 16 : max_group_rows <= 32 ? 32 : max_group_rows <= 64 ? 64 : 0;
}
int tc_expert_ffn_fp8_decode(int act, const void *x_perm, void *h, int64_t rows, int d, int F, int max_group_rows,
                             const uint8_t *w1q, const float *w1s, const uint8_t *w3q, const float *w3s,
                             const uint8_t *w2q, const float *w2s, const int32_t *offsets, int G, void *y, int *dep,
                             int *status, cudaStream_t stream);
int launch_quantize_fp8(const void *w, int64_t rows, int cols, uint8_t *q, float *scales, cudaStream_t s);
// The gate/up GEMM recomputed for the backward with the activation's backward
// fused into its epilogue: a = A W1_g^T (and u = A W3_g^T), dh [rows, F] read,
// dA written: SwiGLU [rows, 2F] = [dh u SiLU'(a) | dh SiLU(a)], ReLU [rows, F] =
// dh [a > 0].  W1/W3 as in tc_grouped_gemm (K-major [G * F, K]).
int tc_grouped_gemm_act_bwd(bool swiglu, const void *A, int64_t a_rows, int K, const void *W1, const void *W3,
                            int64_t b_rows_total, int F, const int32_t *offsets, int G, int M, const void *dh,
                            void *dA, int *status, bool pair_tiles, cudaStream_t stream);
// The same GEMM with each group's B stored [K, n_out] (the stacked weights read in
// place, MN-major tiles): out = A[:, :K1] B0_g, or with A2 (dual) out = A B0_g +
// A2 B1_g where A2 is a second [a_rows, K2] view with the same row stride.
// A rows are a_stride elements apart; B0/B1 are [G][K][n_out] bf16.  Plain epilogue.
int tc_grouped_gemm_bt(const void *A, const void *A2, int64_t a_rows, int64_t a_stride, int K1, int K2,
                       const void *B0, const void *B1, int G, int n_out, const int32_t *offsets, int M, void *out,
                       int *status, bool pair_tiles, cudaStream_t stream);
// Tile choice for expert groups: pairs when the mean group holds >= 512 rows and no
// capacity limit can skew the groups.
inline bool use_pair_tiles(int64_t rows, int groups, int capacity) {
  return capacity <= 0 && rows >= (int64_t)512 * groups;
}

// grouped GEMM on the CUDA cores (float32 workloads); same modes and layouts, float32 out
int simt_grouped_gemm(int mode, const void *A, int64_t a_rows, int K, const void *B0, const void *B1,
                      int b_rows_per_group, const int32_t *offsets, int G, int M, int n_out, void *out,
                      cudaStream_t stream);

// sum of split router partials + logit bias -> logits (no top-k)
int launch_router_sum(const float *partial, int S, int pstride, const float *logit_bias, float *logits, int T, int N,
                      cudaStream_t s);
// counts_routed = counts_kept = C for every expert (expert choice)
int launch_fill_counts(int32_t *counts_routed, int32_t *counts_kept, int N, int C, cudaStream_t s);
// backward pieces
// out[g][m][n] = sum over rows r of group g of A[r][m] B[r][n] (tcgen05, float32
// out); A [rows, M] and B [rows, Nn] bf16 row-major with row strides a_stride /
// b_stride; offsets [G + 1] device (nullptr: one group of all rows).
int tc_wgrad_gemm(const void *A, int64_t a_stride, const void *B, int64_t b_stride, int64_t rows,
                  const int32_t *offsets, int G, int M, int Nn, float *out, int *status, cudaStream_t stream);
int launch_zero_f32(float *p, size_t n, cudaStream_t s);
int launch_dy_dgate(const void *dout, const void *y_perm, const float *topk_w, const int32_t *dest_row,
                    const int32_t *src_token, const int32_t *rows_end, int64_t max_rows, int k, int d, void *dy,
                    float *dgate, cudaStream_t s);
int launch_router_bwd(const float *logits, const int32_t *idx, const float *topk_w, const float *dgate, int gate, int T,
                      int N, int k, float *dz, cudaStream_t s);
// dW_g = x^T dz on the tensor cores: dz split into bf16 [hi | lo] columns (Np =
// N rounded up to 4), one weight-gradient GEMM over all T rows, halves added.
int launch_split_dz(const float *dz, int T, int N, int Np, void *out, cudaStream_t s);
int launch_dwg_sum(const float *part, int d, int N, int Np, float *dWg, cudaStream_t s);
// dz W_g^T on the tensor cores: dz^T and W_g^T split into bf16 [hi; lo; hi] and
// [hi; hi; lo] row blocks (Np = N rounded up to 4, Tp = T rounded up to 8).
int launch_split_router_term(const float *dz, const float *Wg, int T, int d, int N, int Np, int Tp, void *dzT,
                             void *wgT, cudaStream_t s);
// dx = router term + the kept rows of dx_perm (+ the shared expert's dx)
int launch_dx_combine(const void *dxp, const int32_t *dest_row, const float *rterm, const void *dx_sh, int T, int d,
                      int k, float *dx, cudaStream_t s);
int launch_set_offsets2(int32_t *offsets, int rows, cudaStream_t s);

// expert choice: scores + per-expert top-C selection
int launch_expert_choice(const float *logits, int T, int N, int C, float *scores, int32_t *offsets,
                         int32_t *src_token, int32_t *dest_row, cudaStream_t s);

// combine (up to 256 slots per token)
int launch_combine(bool bf16, const void *y_perm, const int32_t *dest_row, const float *w, const void *y_shared,
                   void *out, int T, int d, int k, cudaStream_t s);

// load statistics
constexpr int kStatsChunk = 32;  // tokens per partial-sum chunk
// total = all routed assignments (T * k, or N * C under expert choice)
int launch_load_stats(const float *logits, const int32_t *counts_routed, const int32_t *counts_kept, int T, int N,
                      long long total, int gate, float *partial, int *ticket, float *f, float *P, float *summary,
                      cudaStream_t s);
int launch_router_zloss(const float *logits, int T, int N, float *partial, float *z_loss, cudaStream_t s);
// Sequence-wise balance loss: chunks of the P partials it needs for T tokens in
// sequences of L (at most 2 ceil(T / 32) + 2 rows of N floats), then the launch.
int seq_balance_chunks(int T, int L);
int launch_seq_balance_loss(const float *logits, const int32_t *topk_idx, int T, int N, int k, int gate, int L,
                            float *partial, float *seq_loss, float *loss, int *status, cudaStream_t s);
int launch_bias_update(const int32_t *counts_routed, int T, int k, int N, float *sel_bias, float gamma,
                       cudaStream_t s);

}  // namespace moe
