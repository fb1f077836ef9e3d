// C ABI of libmoe_b300: argument checks, workspace layout and the order of the
// launches.  Every function returns a moe_status; argument errors launch nothing.
#include <algorithm>
#include <mutex>
#include <string.h>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {

int device_sm_count(int device) {
  static std::mutex mu;
  static std::vector<int> cache;
  std::lock_guard<std::mutex> lk(mu);
  if (device < 0) return -1;
  if ((int)cache.size() <= device) cache.resize(device + 1, 0);
  if (cache[device] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) return -1;
    cache[device] = n;
  }
  return cache[device];
}

namespace {

inline size_t align256(size_t v) { return (v + 255) & ~(size_t)255; }
inline bool is_bf16(const moe_config *c) { return c->dtype == MOE_BF16; }
inline size_t esize(const moe_config *c) { return is_bf16(c) ? 2 : 4; }
inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

int check_config(const moe_config *c) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d < 1 || c->N < 1 || c->k < 1 || c->ffn < 1 || c->shared_ffn < 0) return MOE_ERR_INVALID_ARG;
  if (c->gate != MOE_GATE_SOFTMAX_TOPK && c->gate != MOE_GATE_SIGMOID_BIAS && c->gate != MOE_GATE_SOFTMAX_FULL)
    return MOE_ERR_INVALID_ARG;
  if (c->act != MOE_ACT_RELU && c->act != MOE_ACT_SWIGLU) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_F32 && c->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->routing != MOE_ROUTING_TOKEN_CHOICE && c->routing != MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  if (c->routing == MOE_ROUTING_EXPERT_CHOICE && c->capacity < 1) return MOE_ERR_INVALID_ARG;
  if (c->N > 256 || c->k > 8 || c->k > c->N) return MOE_ERR_UNSUPPORTED;
  if (c->d > 65536 || c->ffn > 65536 || c->shared_ffn > 65536) return MOE_ERR_UNSUPPORTED;
  const int q = is_bf16(c) ? 8 : 4;  // 16-byte rows
  if (c->d % q || c->ffn % q || c->shared_ffn % q) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->k >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)c->T * c->N >= (int64_t)1 << 31) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

inline bool is_ec(const moe_config *c) { return c->routing == MOE_ROUTING_EXPERT_CHOICE; }
// tokens per expert under expert choice
inline int ec_c(const moe_config *c) { return c->capacity < c->T ? c->capacity : c->T; }
// routed rows (x_perm, h, y_perm) and routing slots per token (dest_row, gate weights)
inline int64_t routed_rows(const moe_config *c) { return is_ec(c) ? (int64_t)c->N * ec_c(c) : (int64_t)c->T * c->k; }
inline int slots(const moe_config *c) { return is_ec(c) ? c->N : c->k; }

// Scratch for the load statistics, the z-loss and the sequence-wise balance
// loss: up to 2 ceil(T / 32) + 2 rows of N float partials, then T floats.
inline size_t stats_rows_bytes(const moe_config *c) {
  const size_t nch_s = ((size_t)c->T + kStatsChunk - 1) / kStatsChunk;
  return align256((2 * nch_s + 2) * (size_t)c->N * 4);
}
inline size_t stats_bytes(const moe_config *c) { return stats_rows_bytes(c) + align256((size_t)c->T * 4); }

// A group's rows are bounded by T (a token reaches an expert at most once) and by
// the capacity (expert choice's C included).
inline int group_bound(const moe_config *c) { return c->capacity > 0 && c->capacity < c->T ? c->capacity : c->T; }

inline size_t router_scratch_bytes(const moe_config *c) {
  if (!is_bf16(c)) return 0;
  const size_t Np = (size_t)router_tc_npad(c->N), dp = (size_t)router_tc_dpad(c->d);
  return align256(align256(Np * 3 * dp * 2) + (size_t)router_tc_max_splits(c->T, c->d) * c->T * Np * 4);
}

int layout(const moe_config *c, moe_ws_layout *L) {
  const size_t T = (size_t)c->T, N = (size_t)c->N, k = (size_t)c->k, d = (size_t)c->d, F = (size_t)c->ffn;
  const size_t Fs = (size_t)c->shared_ffn, es = esize(c);
  const size_t rows = (size_t)routed_rows(c);
  const size_t sl = (size_t)slots(c);
  const size_t nch_d = (T + kDispatchChunk - 1) / kDispatchChunk;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + (bytes ? bytes : 1));
    return at;
  };
  L->status = take(8);  // the status word, then the CTA-pair GEMM's tile counter
  L->logits = take(T * N * 4);
  L->topk_idx = take(T * k * 4);
  L->topk_w = take(T * sl * 4);
  L->counts_routed = take(N * 4);
  L->counts_kept = take(N * 4);
  L->offsets = take((N + 1) * 4);
  L->dest_row = take(T * sl * 4);
  L->src_token = take(rows * 4);
  L->x_perm = take(rows * d * es);
  L->h = take(rows * F * es);
  L->y_perm = take(rows * d * es);
  L->h_shared = take(Fs ? T * Fs * es : 0);
  L->y_shared = take(Fs ? T * d * es : 0);
  L->scratch = take(align256(2 * nch_d * N * 4) + stats_bytes(c) + router_scratch_bytes(c) + align256(N * 4));
  L->total = o;
  return MOE_OK;
}

struct Ws {
  moe_ws_layout L;
  uint8_t *base;
  template <typename P>
  P *at(size_t off) const {
    return reinterpret_cast<P *>(base + off);
  }
  int *status() const { return at<int>(L.status); }
  int32_t *hist() const { return at<int32_t>(L.scratch); }
  int32_t *chunk_base(const moe_config *c) const {
    const size_t nch = ((size_t)c->T + kDispatchChunk - 1) / kDispatchChunk;
    return at<int32_t>(L.scratch + nch * c->N * 4);
  }
  float *stats_partial(const moe_config *c) const {
    const size_t nch = ((size_t)c->T + kDispatchChunk - 1) / kDispatchChunk;
    return at<float>(L.scratch + align256(2 * nch * c->N * 4));
  }
  float *seq_loss(const moe_config *c) const {
    const size_t nch = ((size_t)c->T + kDispatchChunk - 1) / kDispatchChunk;
    return at<float>(L.scratch + align256(2 * nch * c->N * 4) + stats_rows_bytes(c));
  }
  size_t router_off(const moe_config *c) const {
    const size_t nch = ((size_t)c->T + kDispatchChunk - 1) / kDispatchChunk;
    return L.scratch + align256(2 * nch * c->N * 4) + stats_bytes(c);
  }
  uint16_t *router_wsplit(const moe_config *c) const { return at<uint16_t>(router_off(c)); }
  float *router_partial(const moe_config *c) const {
    const size_t Np = (size_t)router_tc_npad(c->N), dp = (size_t)router_tc_dpad(c->d);
    return at<float>(router_off(c) + align256(Np * 3 * dp * 2));
  }
  // N counters of the one-launch FP8 decode FFN (zeroed before each launch)
  int *fp8_dep(const moe_config *c) const { return at<int>(router_off(c) + router_scratch_bytes(c)); }
};

int make_ws(const moe_config *c, void *ws, Ws *w) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255)) return MOE_ERR_INVALID_ARG;
  layout(c, &w->L);
  w->base = static_cast<uint8_t *>(ws);
  return MOE_OK;
}

#define MOE_TRY(x)        \
  do {                    \
    const int rc_ = (x);  \
    if (rc_) return rc_;  \
  } while (0)

// The routed experts.  bf16 with x and src_token given (x_perm null): the gate/up
// GEMM gathers each row of its A operand from x (row src_token[r]) instead of
// reading a permuted copy.
int ffn_routed(const moe_config *c, const void *x_perm, const void *x, const int32_t *src_token,
               const int32_t *offsets, const void *w1, const void *w3, const void *w2, void *h, void *y_perm,
               int *status, cudaStream_t s) {
  const int64_t rows = routed_rows(c);
  const int mode1 = c->act == MOE_ACT_SWIGLU ? 0 : 1;
  if (is_bf16(c)) {
    // expert choice gives every group exactly C rows: no capacity skew
    const bool pair = use_pair_tiles(rows, c->N, is_ec(c) ? 0 : c->capacity);
    if (x_perm)
      MOE_TRY(tc_grouped_gemm(mode1, x_perm, rows, c->d, w1, w3, (int64_t)c->N * c->ffn, c->ffn, offsets, c->N, 0,
                              c->ffn, h, status, pair, s));
    else
      MOE_TRY(tc_grouped_gemm_gather(mode1, x, c->T, src_token, rows, c->d, w1, w3, (int64_t)c->N * c->ffn, c->ffn,
                                     offsets, c->N, c->ffn, h, status, pair, s));
    MOE_TRY(tc_grouped_gemm(2, h, rows, c->ffn, w2, nullptr, (int64_t)c->N * c->d, c->d, offsets, c->N, 0, c->d,
                            y_perm, status, pair, s));
  } else {
    MOE_TRY(simt_grouped_gemm(mode1, x_perm, rows, c->d, w1, w3, c->ffn, offsets, c->N, 0, c->ffn, h, s));
    MOE_TRY(simt_grouped_gemm(2, h, rows, c->ffn, w2, nullptr, c->d, offsets, c->N, 0, c->d, y_perm, s));
  }
  return MOE_OK;
}

// FP8 E4M3 expert weights with per-row float32 scales (codes [N, rows, K] bytes)
struct Fp8Weights {
  const uint8_t *w1q;
  const float *w1s;
  const uint8_t *w3q;
  const float *w3s;
  const uint8_t *w2q;
  const float *w2s;
};

int check_fp8(const moe_config *c, const Fp8Weights &f) {
  if (!is_bf16(c) || c->d % 16 || c->ffn % 16) return MOE_ERR_UNSUPPORTED;  // code rows: 16-byte multiples
  if (!f.w1q || !f.w1s || !f.w2q || !f.w2s) return MOE_ERR_INVALID_ARG;
  if (c->act == MOE_ACT_SWIGLU && (!f.w3q || !f.w3s)) return MOE_ERR_INVALID_ARG;
  if (!aligned16(f.w1q) || !aligned16(f.w2q) || (f.w3q && !aligned16(f.w3q))) return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

int ffn_routed_fp8(const moe_config *c, const Ws &w, const void *x_perm, const int32_t *offsets,
                   const Fp8Weights &f, void *h, void *y_perm, cudaStream_t s) {
  const int64_t rows = routed_rows(c);
  const int mode1 = c->act == MOE_ACT_SWIGLU ? 0 : 1;
  const int bound = group_bound(c);
  if (fp8_decode_tile_rows(bound))  // decode-sized groups: both GEMMs in one launch, weights on the M side
    return tc_expert_ffn_fp8_decode(mode1, x_perm, h, rows, c->d, c->ffn, bound, f.w1q, f.w1s, f.w3q, f.w3s, f.w2q,
                                    f.w2s, offsets, c->N, y_perm, w.fp8_dep(c), w.status(), s);
  MOE_TRY(tc_grouped_gemm_fp8(mode1, x_perm, rows, c->d, f.w1q, f.w1s, f.w3q, f.w3s, (int64_t)c->N * c->ffn, c->ffn,
                              offsets, c->N, 0, c->ffn, h, w.status(), s));
  return tc_grouped_gemm_fp8(2, h, rows, c->ffn, f.w2q, f.w2s, nullptr, nullptr, (int64_t)c->N * c->d, c->d, offsets,
                             c->N, 0, c->d, y_perm, w.status(), s);
}

int ffn_shared(const moe_config *c, const void *x, const void *sw1, const void *sw3, const void *sw2, void *h,
               void *y, int *status, cudaStream_t s) {
  const int mode1 = c->act == MOE_ACT_SWIGLU ? 0 : 1;
  const int Fs = c->shared_ffn;
  if (is_bf16(c)) {
    const bool pair = use_pair_tiles(c->T, 1, 0);
    MOE_TRY(tc_grouped_gemm(mode1, x, c->T, c->d, sw1, sw3, Fs, Fs, nullptr, 1, c->T, Fs, h, status, pair, s));
    MOE_TRY(tc_grouped_gemm(2, h, c->T, Fs, sw2, nullptr, c->d, c->d, nullptr, 1, c->T, c->d, y, status, pair, s));
  } else {
    MOE_TRY(simt_grouped_gemm(mode1, x, c->T, c->d, sw1, sw3, Fs, nullptr, 1, c->T, Fs, h, s));
    MOE_TRY(simt_grouped_gemm(2, h, c->T, Fs, sw2, nullptr, c->d, nullptr, 1, c->T, c->d, y, s));
  }
  return MOE_OK;
}

// logits, top-k and gate weights: tensor-core router for bf16 x, CUDA-core router for float32 x
// A handful of tokens (decode): the tensor-core router's fixed costs (splitting W_g,
// tensor memory, its pipeline) outweigh its work, so float32 FMA on the CUDA cores,
// split along K over CTAs, computes the logits; the top-k kernel adds the splits.
inline bool small_router(const moe_config *c) { return is_bf16(c) && c->T <= 64; }
inline int small_router_splits(const moe_config *c) {
  return std::min(router_tc_max_splits(c->T, c->d), (c->d + 127) / 128);
}

int route(const moe_config *c, const Ws &w, const void *x, const float *Wg, const float *logit_bias,
          const float *sel_bias, float *logits, int32_t *idx, float *gw, cudaStream_t s) {
  const float *sb = c->gate == MOE_GATE_SIGMOID_BIAS ? sel_bias : nullptr;
  if (!is_bf16(c) && c->T > 64 && router_fused_fits(c->T, c->d, c->N) && aligned16(Wg))
    return launch_router_fused(x, is_bf16(c), Wg, logit_bias, sb, c->T, c->d, c->N, c->k, c->gate, logits, idx, gw,
                               w.status(), s);
  if (small_router(c)) {
    const int S = small_router_splits(c);
    float *part = w.router_partial(c);  // [S][T][N] within the [max splits][T][Npad] scratch
    MOE_TRY(launch_router_logits(x, true, Wg, nullptr, c->T, c->d, c->N, S, part, s));
    const int nkc = (c->d + 127) / 128, kc_per = (nkc + S - 1) / S;
    return launch_router_topk(part, (nkc + kc_per - 1) / kc_per, c->N, logit_bias, logits, sb, c->T, c->N, c->k,
                              c->gate, idx, gw, w.status(), s);
  }
  if (is_bf16(c)) {
    int S = 1;
    float *part = w.router_partial(c);
    MOE_TRY(launch_router_tc(x, Wg, c->T, c->d, c->N, w.router_wsplit(c), part, &S, w.status(), s));
    return launch_router_topk(part, S, router_tc_npad(c->N), logit_bias, logits, sb, c->T, c->N, c->k, c->gate, idx,
                              gw, w.status(), s);
  }
  MOE_TRY(launch_router_logits(x, false, Wg, logit_bias, c->T, c->d, c->N, 1, logits, s));
  return launch_router_topk(logits, 1, c->N, nullptr, logits, sb, c->T, c->N, c->k, c->gate, idx, gw, w.status(), s);
}

// expert choice: logits, scores, per-expert top-C; counts in the workspace read C
int ec_route(const moe_config *c, const Ws &w, const void *x, const float *Wg, const float *logit_bias,
             float *logits, float *scores, int32_t *offsets, int32_t *src_token, int32_t *dest_row, cudaStream_t s) {
  if (is_bf16(c)) {
    int S = 1;
    float *part = w.router_partial(c);
    MOE_TRY(launch_router_tc(x, Wg, c->T, c->d, c->N, w.router_wsplit(c), part, &S, w.status(), s));
    MOE_TRY(launch_router_sum(part, S, router_tc_npad(c->N), logit_bias, logits, c->T, c->N, s));
  } else {
    MOE_TRY(launch_router_logits(x, false, Wg, logit_bias, c->T, c->d, c->N, 1, logits, s));
  }
  MOE_TRY(launch_expert_choice(logits, c->T, c->N, ec_c(c), scores, offsets, src_token, dest_row, s));
  return launch_fill_counts(w.at<int32_t>(w.L.counts_routed), w.at<int32_t>(w.L.counts_kept), c->N, ec_c(c), s);
}

// ---------------------------------------------------------------- backward workspace
struct BwdLayout {
  size_t dgate, dz, dz2, dwg2, dzT3, wgT3, rterm, off_sh, dy, dh, dA, dxp;
  size_t dh_s, dA_s, dx_s, total;
};

BwdLayout bwd_layout(const moe_config *c) {
  BwdLayout L{};
  const size_t T = c->T, N = c->N, k = c->k, d = c->d, F = c->ffn, Fs = c->shared_ffn;
  const size_t R = (size_t)c->T * c->k;
  const bool sw = c->act == MOE_ACT_SWIGLU;
  const size_t FA = sw ? 2 * F : F, FAs = sw ? 2 * Fs : Fs;  // width of dA
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align256(o + (bytes ? bytes : 1));
    return at;
  };
  L.dgate = take(T * k * 4);
  L.dz = take(T * N * 4);
  const size_t Np = (N + 3) / 4 * 4;
  L.dz2 = take(T * 2 * Np * 2);  // dz as bf16 [hi | lo]
  L.dwg2 = take(d * 2 * Np * 4);  // x^T [hi | lo]
  const size_t Tp = (T + 7) / 8 * 8;
  L.dzT3 = take(3 * Np * Tp * 2);  // dz^T [hi; lo; hi]
  L.wgT3 = take(3 * Np * d * 2);   // W_g^T [hi; hi; lo]
  L.rterm = take(T * d * 4);       // dz W_g^T
  L.off_sh = take(2 * 4);
  L.dy = take(R * d * 2);
  L.dh = take(R * F * 2);
  L.dA = take(R * FA * 2);
  L.dxp = take(R * d * 2);
  if (Fs) {
    L.dh_s = take(T * Fs * 2);
    L.dA_s = take(T * FAs * 2);
    L.dx_s = take(T * d * 2);
  }
  L.total = o;
  return L;
}

int check_backward(const moe_config *c) {
  MOE_TRY(check_config(c));
  if (!is_bf16(c) || is_ec(c)) return MOE_ERR_UNSUPPORTED;  // bf16 token choice only
  return MOE_OK;
}

// One expert set (routed: G = N with offsets; shared: G = 1) through the FFN backward.
// dy [R, d], the forward's x rows (x_perm or x), h; writes dx rows (bf16) and float32 grads.
int ffn_backward(const moe_config *c, bool shared, int G, int64_t R, const int32_t *offsets, const int32_t *off_dev,
                 const void *xrows, const void *h, const void *dy, const void *w1, const void *w3, const void *w2,
                 int F, uint8_t *bws, const BwdLayout &L, float *dw1, float *dw3, float *dw2, void *dxrows,
                 int *status, cudaStream_t s) {
  const bool sw = c->act == MOE_ACT_SWIGLU;
  const int d = c->d, FA = sw ? 2 * F : F;
  const bool pair = use_pair_tiles(R, G, shared ? 0 : c->capacity);
  auto B = [&](size_t off) { return bws + off; };
  void *dh = B(shared ? L.dh_s : L.dh);
  void *dA = B(shared ? L.dA_s : L.dA);
  const int M = shared ? c->T : 0;
  // dh = dy W2, W2 read in place as [G][d][F]
  MOE_TRY(tc_grouped_gemm_bt(dy, nullptr, R, d, d, 0, w2, nullptr, G, F, offsets, M, dh, status, pair, s));
  // a = x W1^T and u = x W3^T recomputed, the activation's backward in the epilogue: dA = [da | du]
  MOE_TRY(tc_grouped_gemm_act_bwd(sw, xrows, R, d, w1, sw ? w3 : nullptr, (int64_t)G * F, F, offsets, G, M, dh, dA,
                                  status, pair, s));
  // dx rows = da W1 + du W3, W1 and W3 read in place as [G][F][d]
  MOE_TRY(tc_grouped_gemm_bt(dA, sw ? static_cast<uint8_t *>(dA) + (size_t)F * 2 : nullptr, R, FA, F, F, w1,
                             sw ? w3 : nullptr, G, d, offsets, M, dxrows, status, pair, s));
  // weight gradients: sums over each expert's rows, the activations read in place
  const int64_t rows = shared ? (int64_t)c->T : R;
  const int32_t *goff = shared ? nullptr : off_dev;
  MOE_TRY(tc_wgrad_gemm(dy, d, h, F, rows, goff, G, d, F, dw2, status, s));
  MOE_TRY(tc_wgrad_gemm(dA, FA, xrows, d, rows, goff, G, F, d, dw1, status, s));
  if (sw)
    MOE_TRY(tc_wgrad_gemm(static_cast<uint8_t *>(dA) + (size_t)F * 2, FA, xrows, d, rows, goff, G, F, d, dw3, status,
                          s));
  return MOE_OK;
}

bool weights_ok(const moe_config *c, const void *w1, const void *w3, const void *w2) {
  if (!w1 || !w2 || !aligned16(w1) || !aligned16(w2)) return false;
  if (c->act == MOE_ACT_SWIGLU && (!w3 || !aligned16(w3))) return false;
  return true;
}

// A wait that nothing can end: an mbarrier expecting one arrival that never
// comes.  The bounded wait gives up after limit_ns and records MOE_ERR_TIMEOUT.
__global__ void wait_timeout_kernel(int *status, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, status, limit_ns);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or alignment";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_NONFINITE: return "non-finite router logit";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    case MOE_ERR_BOUNDS: return "index out of range";
    default: return "unknown status";
  }
}

int moe_capacity(double alpha, int32_t T, int32_t k, int32_t N, int32_t *C) {
  if (!C || !(alpha > 0.0) || alpha > 1e9 || T < 0 || k < 1 || N < 1) return MOE_ERR_INVALID_ARG;
  // alpha = m * 2^e exactly, m a 53-bit integer
  int e = 0;
  const double fr = frexp(alpha, &e);        // alpha = fr * 2^e, fr in [0.5, 1)
  const int64_t m = (int64_t)ldexp(fr, 53);  // exact
  e -= 53;
  // C = ceil(m * T * k * 2^e / N)
  __int128 num = (__int128)m * T * k;
  __int128 den = N;
  if (e >= 0) {
    if (e > 60) return MOE_ERR_UNSUPPORTED;
    num <<= e;
  } else {
    if (-e > 100) return MOE_ERR_UNSUPPORTED;
    den <<= -e;
  }
  const __int128 q = (num + den - 1) / den;
  if (q > 0x7FFFFFFF) return MOE_ERR_UNSUPPORTED;
  *C = (int32_t)q;
  return MOE_OK;
}

int moe_workspace_layout(const moe_config *cfg, moe_ws_layout *out) {
  MOE_TRY(check_config(cfg));
  if (!out) return MOE_ERR_INVALID_ARG;
  return layout(cfg, out);
}

int moe_workspace_size(const moe_config *cfg, size_t *bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  moe_ws_layout L;
  MOE_TRY(moe_workspace_layout(cfg, &L));
  *bytes = L.total;
  return MOE_OK;
}

int moe_route(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias, const float *sel_bias,
              float *logits, int32_t *topk_idx, float *topk_w, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (is_ec(cfg)) return MOE_ERR_INVALID_ARG;  // expert choice: moe_ec_route
  if (cfg->T == 0) return MOE_OK;
  if (!x || !Wg || !logits || !topk_idx || !topk_w || !aligned16(x)) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return route(cfg, w, x, Wg, logit_bias, sel_bias, logits, topk_idx, topk_w, static_cast<cudaStream_t>(stream));
}

int moe_dispatch(const moe_config *cfg, const int32_t *topk_idx, const void *x, int32_t *counts_routed,
                 int32_t *counts_kept, int32_t *offsets, int32_t *dest_row, int32_t *src_token, void *x_perm,
                 void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (is_ec(cfg)) return MOE_ERR_INVALID_ARG;  // expert choice routes and dispatches in moe_ec_route
  if (!counts_routed || !counts_kept || !offsets) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cfg->T > 0 && (!topk_idx || !dest_row || !src_token || (x_perm && (!x || !aligned16(x) || !aligned16(x_perm)))))
    return MOE_ERR_INVALID_ARG;
  MOE_TRY(launch_dispatch(topk_idx, cfg->T, cfg->k, cfg->N, cfg->capacity, w.hist(), w.chunk_base(cfg), counts_routed,
                          counts_kept, offsets, dest_row, src_token, w.status(), s));
  if (cfg->T == 0 || !x_perm) return MOE_OK;  // no permuted copy asked for
  return launch_scatter_rows(x, dest_row, cfg->T, cfg->k, (int)(cfg->d * esize(cfg)), x_perm, s);
}

int moe_expert_ffn(const moe_config *cfg, const void *x_perm, const int32_t *offsets, const void *w1, const void *w3,
                   const void *w2, void *y_perm, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (!x_perm || !offsets || !y_perm || !aligned16(x_perm) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(cfg, w1, w3, w2)) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return ffn_routed(cfg, x_perm, nullptr, nullptr, offsets, w1, w3, w2, w.at<void>(w.L.h), y_perm, w.status(),
                    static_cast<cudaStream_t>(stream));
}

int moe_expert_ffn_gather(const moe_config *cfg, const void *x, const int32_t *src_token, const int32_t *offsets,
                          const void *w1, const void *w3, const void *w2, void *y_perm, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (!is_bf16(cfg)) return MOE_ERR_UNSUPPORTED;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !src_token || !offsets || !y_perm || !aligned16(x) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  if (!weights_ok(cfg, w1, w3, w2)) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return ffn_routed(cfg, nullptr, x, src_token, offsets, w1, w3, w2, w.at<void>(w.L.h), y_perm, w.status(),
                    static_cast<cudaStream_t>(stream));
}

int moe_shared_ffn(const moe_config *cfg, const void *x, const void *sw1, const void *sw3, const void *sw2,
                   void *y_shared, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->shared_ffn <= 0) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !y_shared || !aligned16(x) || !aligned16(y_shared) || !weights_ok(cfg, sw1, sw3, sw2))
    return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return ffn_shared(cfg, x, sw1, sw3, sw2, w.at<void>(w.L.h_shared), y_shared, w.status(),
                    static_cast<cudaStream_t>(stream));
}

int moe_combine(const moe_config *cfg, const void *y_perm, const int32_t *dest_row, const float *topk_w,
                const void *y_shared, void *out, void *stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (!y_perm || !dest_row || !topk_w || !out || !aligned16(y_perm) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (y_shared && !aligned16(y_shared)) return MOE_ERR_INVALID_ARG;
  return launch_combine(is_bf16(cfg), y_perm, dest_row, topk_w, y_shared, out, cfg->T, cfg->d, slots(cfg),
                        static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {
// The layer with bf16 / float32 expert weights (f8 == nullptr) or FP8 ones.
int layer_forward_impl(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
                       const float *sel_bias, const void *w1, const void *w3, const void *w2, const Fp8Weights *f8,
                       const void *sw1, const void *sw3, const void *sw2, void *out, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (!x || !Wg || !out || !aligned16(x) || !aligned16(out)) return MOE_ERR_INVALID_ARG;
  if (f8) {
    MOE_TRY(check_fp8(cfg, *f8));
  } else if (!weights_ok(cfg, w1, w3, w2)) {
    return MOE_ERR_INVALID_ARG;
  }
  const bool shared = cfg->shared_ffn > 0;
  if (shared && !weights_ok(cfg, sw1, sw3, sw2)) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const moe_ws_layout &L = w.L;
  float *logits = w.at<float>(L.logits);
  int32_t *idx = w.at<int32_t>(L.topk_idx);
  float *gw = w.at<float>(L.topk_w);
  int32_t *offsets = w.at<int32_t>(L.offsets);
  int32_t *dest_row = w.at<int32_t>(L.dest_row);
  int32_t *src_token = w.at<int32_t>(L.src_token);
  void *x_perm = w.at<void>(L.x_perm);
  void *y_perm = w.at<void>(L.y_perm);
  if (is_ec(cfg)) {
    MOE_TRY(ec_route(cfg, w, x, Wg, logit_bias, logits, gw, offsets, src_token, dest_row, s));
  } else {
    MOE_TRY(route(cfg, w, x, Wg, logit_bias, sel_bias, logits, idx, gw, s));
    MOE_TRY(launch_dispatch(idx, cfg->T, cfg->k, cfg->N, cfg->capacity, w.hist(), w.chunk_base(cfg),
                            w.at<int32_t>(L.counts_routed), w.at<int32_t>(L.counts_kept), offsets, dest_row,
                            src_token, w.status(), s));
  }
  // the experts read a permuted copy of x: one coalesced pass here costs far less than
  // gathering rows into the GEMM's operand tiles, which re-fetch them once per N tile
  if (is_ec(cfg))
    MOE_TRY(launch_gather_rows(x, src_token, offsets + cfg->N, routed_rows(cfg), (int)(cfg->d * esize(cfg)), x_perm,
                               s));
  else
    MOE_TRY(launch_scatter_rows(x, dest_row, cfg->T, cfg->k, (int)(cfg->d * esize(cfg)), x_perm, s));
  if (f8)
    MOE_TRY(ffn_routed_fp8(cfg, w, x_perm, offsets, *f8, w.at<void>(L.h), y_perm, s));
  else
    MOE_TRY(ffn_routed(cfg, x_perm, nullptr, nullptr, offsets, w1, w3, w2, w.at<void>(L.h), y_perm, w.status(), s));
  void *y_sh = nullptr;
  if (shared) {
    y_sh = w.at<void>(L.y_shared);
    MOE_TRY(ffn_shared(cfg, x, sw1, sw3, sw2, w.at<void>(L.h_shared), y_sh, w.status(), s));
  }
  return launch_combine(is_bf16(cfg), y_perm, dest_row, gw, y_sh, out, cfg->T, cfg->d, slots(cfg), s);
}
}  // namespace

extern "C" {

int moe_layer_forward(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
                      const float *sel_bias, const void *w1, const void *w3, const void *w2, const void *sw1,
                      const void *sw3, const void *sw2, void *out, void *ws, void *stream) {
  return layer_forward_impl(cfg, x, Wg, logit_bias, sel_bias, w1, w3, w2, nullptr, sw1, sw3, sw2, out, ws, stream);
}

int moe_layer_forward_fp8(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias,
                          const float *sel_bias, const uint8_t *w1q, const float *w1s, const uint8_t *w3q,
                          const float *w3s, const uint8_t *w2q, const float *w2s, const void *sw1, const void *sw3,
                          const void *sw2, void *out, void *ws, void *stream) {
  const Fp8Weights f{w1q, w1s, w3q, w3s, w2q, w2s};
  return layer_forward_impl(cfg, x, Wg, logit_bias, sel_bias, nullptr, nullptr, nullptr, &f, sw1, sw3, sw2, out, ws,
                            stream);
}

int moe_expert_ffn_fp8(const moe_config *cfg, const void *x_perm, const int32_t *offsets, const uint8_t *w1q,
                       const float *w1s, const uint8_t *w3q, const float *w3s, const uint8_t *w2q, const float *w2s,
                       void *y_perm, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  const Fp8Weights f{w1q, w1s, w3q, w3s, w2q, w2s};
  MOE_TRY(check_fp8(cfg, f));
  if (cfg->T == 0) return MOE_OK;
  if (!x_perm || !offsets || !y_perm || !aligned16(x_perm) || !aligned16(y_perm)) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return ffn_routed_fp8(cfg, w, x_perm, offsets, f, w.at<void>(w.L.h), y_perm, static_cast<cudaStream_t>(stream));
}

int moe_quantize_fp8(const void *w, int64_t rows, int32_t cols, uint8_t *q, float *scales, void *stream) {
  if (rows < 0 || cols < 1) return MOE_ERR_INVALID_ARG;
  if (rows == 0) return MOE_OK;
  if (!w || !q || !scales) return MOE_ERR_INVALID_ARG;
  return launch_quantize_fp8(w, rows, cols, q, scales, static_cast<cudaStream_t>(stream));
}

int moe_load_stats(const moe_config *cfg, const float *logits, const int32_t *counts_routed,
                   const int32_t *counts_kept, float *f, float *P, float *summary, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (cfg->T == 0) return MOE_OK;
  if (!logits || !counts_routed || !counts_kept || !f || !P || !summary) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  const long long total = is_ec(cfg) ? (long long)routed_rows(cfg) : (long long)cfg->T * cfg->k;
  // the ticket of the statistics' last CTA lives in the (here unused) sequence-loss scratch
  return launch_load_stats(logits, counts_routed, counts_kept, cfg->T, cfg->N, total,
                           is_ec(cfg) ? MOE_GATE_SOFTMAX_FULL : cfg->gate, w.stats_partial(cfg),
                           reinterpret_cast<int *>(w.seq_loss(cfg)), f, P, summary, static_cast<cudaStream_t>(stream));
}

int moe_ec_route(const moe_config *cfg, const void *x, const float *Wg, const float *logit_bias, float *logits,
                 float *scores, int32_t *offsets, int32_t *src_token, int32_t *dest_row, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (!is_ec(cfg)) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_OK;
  if (!x || !Wg || !logits || !scores || !offsets || !src_token || !dest_row || !aligned16(x))
    return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return ec_route(cfg, w, x, Wg, logit_bias, logits, scores, offsets, src_token, dest_row,
                  static_cast<cudaStream_t>(stream));
}

int moe_router_zloss(const moe_config *cfg, const float *logits, float *z_loss, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (!logits || !z_loss) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_ERR_INVALID_ARG;  // a mean over no tokens
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  return launch_router_zloss(logits, cfg->T, cfg->N, w.stats_partial(cfg), z_loss, static_cast<cudaStream_t>(stream));
}

int moe_seq_balance_loss(const moe_config *cfg, const float *logits, const int32_t *topk_idx, int32_t seq_len,
                         float *loss, void *ws, void *stream) {
  MOE_TRY(check_config(cfg));
  if (is_ec(cfg)) return MOE_ERR_INVALID_ARG;  // expert choice has no per-token top-k to count
  if (!logits || !topk_idx || !loss || seq_len < 1) return MOE_ERR_INVALID_ARG;
  if (cfg->T == 0) return MOE_ERR_INVALID_ARG;  // a mean over no sequences
  Ws w;
  MOE_TRY(make_ws(cfg, ws, &w));
  const int L = seq_len < cfg->T ? seq_len : cfg->T;
  if (L >= kStatsChunk && (size_t)seq_balance_chunks(cfg->T, L) * cfg->N * 4 > stats_rows_bytes(cfg))
    return MOE_ERR_UNSUPPORTED;  // cannot happen: the bound above holds for every L >= 32
  return launch_seq_balance_loss(logits, topk_idx, cfg->T, cfg->N, cfg->k, cfg->gate, L, w.stats_partial(cfg),
                                 w.seq_loss(cfg), loss, w.status(), static_cast<cudaStream_t>(stream));
}

int moe_bias_update(const moe_config *cfg, const int32_t *counts_routed, float *sel_bias, float gamma, void *stream) {
  MOE_TRY(check_config(cfg));
  if (!counts_routed || !sel_bias || !(gamma >= 0.0f) || gamma > 1e30f) return MOE_ERR_INVALID_ARG;
  return launch_bias_update(counts_routed, cfg->T, cfg->k, cfg->N, sel_bias, gamma, static_cast<cudaStream_t>(stream));
}

int moe_backward_workspace_size(const moe_config *cfg, size_t *bytes) {
  if (!bytes) return MOE_ERR_INVALID_ARG;
  MOE_TRY(check_backward(cfg));
  *bytes = bwd_layout(cfg).total;
  return MOE_OK;
}

int moe_layer_backward(const moe_config *cfg, const void *x, const float *Wg, const void *w1, const void *w3,
                       const void *w2, const void *sw1, const void *sw3, const void *sw2, const void *dout, float *dx,
                       float *dWg, float *dw1, float *dw3, float *dw2, float *dsw1, float *dsw3, float *dsw2,
                       void *fwd_ws, void *bwd_ws, void *stream) {
  MOE_TRY(check_backward(cfg));
  if (cfg->T == 0) return MOE_OK;
  const bool sw = cfg->act == MOE_ACT_SWIGLU, shared = cfg->shared_ffn > 0;
  if (!x || !Wg || !dout || !dx || !dWg || !dw1 || !dw2 || (sw && !dw3) || !weights_ok(cfg, w1, w3, w2))
    return MOE_ERR_INVALID_ARG;
  if (shared && (!weights_ok(cfg, sw1, sw3, sw2) || !dsw1 || !dsw2 || (sw && !dsw3))) return MOE_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(dout) || !aligned16(dx)) return MOE_ERR_INVALID_ARG;
  if (!bwd_ws || (reinterpret_cast<uintptr_t>(bwd_ws) & 255)) return MOE_ERR_INVALID_ARG;
  Ws w;
  MOE_TRY(make_ws(cfg, fwd_ws, &w));
  const moe_ws_layout &FL = w.L;
  const BwdLayout L = bwd_layout(cfg);
  uint8_t *bws = static_cast<uint8_t *>(bwd_ws);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int T = cfg->T, N = cfg->N, k = cfg->k, d = cfg->d;
  const int64_t R = (int64_t)T * k;
  const int32_t *offsets = w.at<int32_t>(FL.offsets);
  const int32_t *dest_row = w.at<int32_t>(FL.dest_row);
  float *dgate = reinterpret_cast<float *>(bws + L.dgate);
  float *dz = reinterpret_cast<float *>(bws + L.dz);
  // gates and router
  MOE_TRY(launch_zero_f32(dgate, (size_t)T * k, s));
  MOE_TRY(launch_dy_dgate(dout, w.at<void>(FL.y_perm), w.at<float>(FL.topk_w), dest_row, w.at<int32_t>(FL.src_token),
                          offsets + N, R, k, d, bws + L.dy, dgate, s));
  MOE_TRY(launch_router_bwd(w.at<float>(FL.logits), w.at<int32_t>(FL.topk_idx), w.at<float>(FL.topk_w), dgate,
                            cfg->gate, T, N, k, dz, s));
  {  // dW_g = x^T dz
    const int Np = (N + 3) / 4 * 4;
    MOE_TRY(launch_split_dz(dz, T, N, Np, bws + L.dz2, s));
    float *part = reinterpret_cast<float *>(bws + L.dwg2);
    MOE_TRY(tc_wgrad_gemm(x, d, bws + L.dz2, 2 * Np, T, nullptr, 1, d, 2 * Np, part, w.status(), s));
    MOE_TRY(launch_dwg_sum(part, d, N, Np, dWg, s));
  }
  // routed experts
  MOE_TRY(ffn_backward(cfg, false, N, R, offsets, offsets, w.at<void>(FL.x_perm), w.at<void>(FL.h), bws + L.dy, w1, w3,
                       w2, cfg->ffn, bws, L, dw1, dw3, dw2, bws + L.dxp, w.status(), s));
  // the shared expert: one group of all T rows, dy = dout
  void *dx_sh = nullptr;
  if (shared) {
    int32_t *off_sh = reinterpret_cast<int32_t *>(bws + L.off_sh);
    MOE_TRY(launch_set_offsets2(off_sh, T, s));
    dx_sh = bws + L.dx_s;
    MOE_TRY(ffn_backward(cfg, true, 1, T, nullptr, off_sh, x, w.at<void>(FL.h_shared), dout, sw1, sw3, sw2,
                         cfg->shared_ffn, bws, L, dsw1, dsw3, dsw2, dx_sh, w.status(), s));
  }
  // x's router term dz W_g^T, then dx
  const int Np = (N + 3) / 4 * 4, Tp = (T + 7) / 8 * 8;
  float *rterm = reinterpret_cast<float *>(bws + L.rterm);
  MOE_TRY(launch_split_router_term(dz, Wg, T, d, N, Np, Tp, bws + L.dzT3, bws + L.wgT3, s));
  MOE_TRY(tc_wgrad_gemm(bws + L.dzT3, Tp, bws + L.wgT3, d, 3 * Np, nullptr, 1, T, d, rterm, w.status(), s));
  return launch_dx_combine(bws + L.dxp, dest_row, rterm, dx_sh, T, d, k, dx, s);
}

int moe_check_wait_timeout(void *ws, int64_t limit_ns, void *stream) {
  if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255) || limit_ns < 0 || limit_ns > 10000000000ll)
    return MOE_ERR_INVALID_ARG;
  wait_timeout_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(static_cast<int *>(ws), (uint64_t)limit_ns);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_get_device_status(void *ws, void *stream, int *status) {
  if (!ws || !status) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  int word = 0;
  if (cudaMemcpyAsync(&word, ws, sizeof(int), cudaMemcpyDeviceToHost, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  const int zero = 0;
  if (cudaMemcpyAsync(ws, &zero, sizeof(int), cudaMemcpyHostToDevice, s) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_CUDA;
  *status = MOE_OK;
  for (int c = 1; c < 31; ++c)
    if (word & (1 << c)) {
      *status = c;
      break;
    }
  return MOE_OK;
}

}  // extern "C"
