// Per-expert load statistics of the Switch balance loss.
//
// "Chapter 19: MoE" 19.3.3: f_i = fraction of assignments routed to expert i,
// P_i = mean router probability of expert i over the batch.  CS336 lecture 4,
// section 9: loss = N * sum_i f_i P_i.  "Lecture29" (CS25 lecture 29 notes),
// "Myth 3": imbalance I = max_i n_i / (T k / N).  Drop rate = share of
// assignments removed by the capacity limit.
//
// p_i(t) is the full N-way softmax of the logits (softmax gate) or
// s_i / sum_l s_l with s = sigmoid(z) (sigmoid gate), in float32.  Partial sums
// per 32-token chunk are reduced in a fixed order, so the result is deterministic.
//
// The sequence-wise balance loss of DeepSeek-V3 ("Chapter 19: MoE" 19.3.4;
// CS336 lecture 4, section 9) is the same N sum_i f_i P_i taken inside each
// sequence of L consecutive tokens and averaged over the sequences.  For L >= 32
// the P partials come from chunks that never cross a sequence boundary and one
// CTA per sequence finishes it; for L < 32 one warp takes a whole sequence.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SC = kStatsChunk;  // tokens per chunk

// Router probabilities of one token, lane + 32 i holding expert lane + 32 i
// (zero past N); called by a whole warp.
__device__ __forceinline__ void token_probs(const float *__restrict__ zr, int N, bool softmax, int lane, float v[8]) {
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < N) ? zr[e] : -INFINITY;
    m = fmaxf(m, v[i]);
  }
  if (softmax) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  }
  float sum = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    float p = 0.f;
    if (e < N) p = softmax ? expf(v[i] - m) : 1.0f / (1.0f + expf(-v[i]));
    v[i] = p;
    sum += p;
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float inv = 1.0f / sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] *= inv;
}

// Sum of p over one chunk of at most SC tokens.  Chunk c is chunk c % cps of
// sequence c / cps (sequences of L tokens, the last one possibly shorter); a
// chunk past its sequence's end writes zeros.  The batch statistics use L = T.
__global__ void __launch_bounds__(256) stats_partial_kernel(const float *__restrict__ logits, int T, int N, int gate,
                                                            int L, int cps, float *__restrict__ partial,
                                                            int *ticket) {
  __shared__ float red[8][256];
  if (ticket && blockIdx.x == 0 && threadIdx.x == 0) *ticket = 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const int seq = blockIdx.x / cps, j = blockIdx.x - seq * cps;
  const long long s0 = (long long)seq * L;
  const long long tb = s0 + (long long)j * SC;
  const long long te = min(min(s0 + L, (long long)T), tb + SC);
  const bool softmax = gate != MOE_GATE_SIGMOID_BIAS;
  const int cnt = (int)max(0LL, te - tb);
#pragma unroll 4
  for (int tt = warp; tt < cnt; tt += 8) {  // SC / 8 tokens per warp, four in flight
    const long long t = tb + tt;
    float v[8];
    token_probs(logits + (size_t)t * N, N, softmax, lane, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += blockDim.x) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w][e];
    partial[(size_t)blockIdx.x * N + e] = s;
  }
}

// ceil(N / 32) CTAs of 1024 threads: CTA b takes experts 32 b + lane; warp w adds
// the chunks w, w + 32, .. of each (loads coalesced across the experts), then the
// 32 warp sums are added in warp order.  The CTA that finishes last (a ticket
// counter, cleared by stats_partial) forms the summary over all experts in a
// fixed order from f, P and the counts: deterministic.
__global__ void __launch_bounds__(1024) stats_final_kernel(const float *__restrict__ partial, int nchunks,
                                                           const int32_t *__restrict__ counts_routed,
                                                           const int32_t *__restrict__ counts_kept, int T, int N,
                                                           long long total, float *__restrict__ f,
                                                           float *__restrict__ P, float *__restrict__ summary,
                                                           int *ticket) {
  __shared__ float red[32][33];
  __shared__ float fp[256];
  __shared__ int maxc[256];
  __shared__ long long kept[256];
  __shared__ bool last;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  float s = 0.f;
  if (e < N) {
#pragma unroll 8
    for (int c = warp; c < nchunks; c += 32) s += partial[(size_t)c * N + e];
  }
  red[warp][lane] = s;
  __syncthreads();
  if (warp == 0 && e < N) {
    float sum = 0.f;
    for (int w = 0; w < 32; ++w) sum += red[w][lane];
    P[e] = sum / (float)T;
    f[e] = (float)((double)counts_routed[e] / (double)total);
  }
  if (gridDim.x > 1) {
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) last = atomicAdd(ticket, 1) == (int)gridDim.x - 1;
    __syncthreads();
    if (!last) return;
    __threadfence();
  } else {
    __syncthreads();  // one CTA: it is the last
  }
  const int x = threadIdx.x;
  if (x < 256) {
    float fe = 0.f, pe = 0.f;
    int ce = 0;
    long long ke = 0;
    if (x < N) {
      fe = __ldcg(f + x);
      pe = __ldcg(P + x);
      ce = counts_routed[x];
      ke = counts_kept[x];
    }
    fp[x] = fe * pe;
    maxc[x] = ce;
    kept[x] = ke;
  }
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if (x < off) {
      fp[x] += fp[x + off];
      maxc[x] = max(maxc[x], maxc[x + off]);
      kept[x] += kept[x + off];
    }
    __syncthreads();
  }
  if (x == 0) {
    const double tk = (double)total;
    summary[0] = (float)N * fp[0];
    summary[1] = (float)((double)maxc[0] / (tk / (double)N));
    summary[2] = (float)(1.0 - (double)kept[0] / tk);
    if (gridDim.x > 1) *ticket = 0;
  }
}

// T <= 32 (one chunk, e.g. decode): the partial sums, P, f and the summary in one
// CTA of 256 threads -- the same arithmetic, in the same order, as the two kernels
// above, without the launch between them.
__global__ void __launch_bounds__(256) stats_one_chunk_kernel(const float *__restrict__ logits, int T, int N, int gate,
                                                              const int32_t *__restrict__ counts_routed,
                                                              const int32_t *__restrict__ counts_kept,
                                                              long long total, float *__restrict__ f,
                                                              float *__restrict__ P, float *__restrict__ summary) {
  __shared__ float red[8][256];
  __shared__ float fp[256];
  __shared__ int maxc[256];
  __shared__ long long kept[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const bool softmax = gate != MOE_GATE_SIGMOID_BIAS;
  for (int t = warp; t < T; t += 8) {
    float v[8];
    token_probs(logits + (size_t)t * N, N, softmax, lane, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) acc[i] += v[i];
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) red[warp][lane + 32 * i] = acc[i];
  __syncthreads();
  const int x = threadIdx.x;
  float fe = 0.f, pe = 0.f;
  int ce = 0;
  long long ke = 0;
  if (x < N) {
    float sum = 0.f;
    for (int w = 0; w < 8; ++w) sum += red[w][x];
    pe = sum / (float)T;
    fe = (float)((double)counts_routed[x] / (double)total);
    P[x] = pe;
    f[x] = fe;
    ce = counts_routed[x];
    ke = counts_kept[x];
  }
  fp[x] = fe * pe;
  maxc[x] = ce;
  kept[x] = ke;
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if (x < off) {
      fp[x] += fp[x + off];
      maxc[x] = max(maxc[x], maxc[x + off]);
      kept[x] += kept[x + off];
    }
    __syncthreads();
  }
  if (x == 0) {
    const double tk = (double)total;
    summary[0] = (float)N * fp[0];
    summary[1] = (float)((double)maxc[0] / (tk / (double)N));
    summary[2] = (float)(1.0 - (double)kept[0] / tk);
  }
}

// One CTA per sequence (L >= 32): P_e L = the sequence's chunk partials added in
// order, n_e = its assignments to e (counted from topk_idx), and
// loss_s = N sum_e (n_e / (L k)) (P_e L / L).
__global__ void __launch_bounds__(256) seq_final_kernel(const float *__restrict__ partial, int cps,
                                                        const int32_t *__restrict__ topk_idx, int T, int N, int k,
                                                        int L, float *__restrict__ seq_loss, int *status) {
  __shared__ int cnt[256];
  __shared__ float red[256];
  const int e = threadIdx.x;
  const int seq = blockIdx.x;
  const long long t0 = (long long)seq * L, t1 = min((long long)T, t0 + L);
  cnt[e] = 0;
  __syncthreads();
  for (long long i = t0 * k + threadIdx.x; i < t1 * k; i += blockDim.x) {
    const int v = topk_idx[i];
    if ((unsigned)v < (unsigned)N) atomicAdd(&cnt[v], 1);
    else set_status(status, MOE_ERR_BOUNDS);
  }
  float psum = 0.f;
  if (e < N)
    for (int j = 0; j < cps; ++j) psum += partial[((size_t)seq * cps + j) * N + e];
  __syncthreads();
  red[e] = (e < N) ? (float)cnt[e] * psum : 0.f;
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if (e < off) red[e] += red[e + off];
    __syncthreads();
  }
  if (e == 0) {
    const float Ls = (float)(t1 - t0);
    seq_loss[seq] = (float)N * (red[0] / (Ls * (float)k)) / Ls;
  }
}

// One warp per sequence (L < 32): p and the counts of the sequence's tokens in
// registers (lane + 32 i holds expert lane + 32 i), then the same loss_s.
__global__ void __launch_bounds__(256) seq_short_kernel(const float *__restrict__ logits,
                                                        const int32_t *__restrict__ topk_idx, int T, int N, int k,
                                                        int gate, int L, int nseq, float *__restrict__ seq_loss,
                                                        int *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int seq = blockIdx.x * 8 + warp;
  if (seq >= nseq) return;
  const int t0 = seq * L, t1 = min(T, t0 + L);
  const bool softmax = gate != MOE_GATE_SIGMOID_BIAS;
  float P[8];
  int n[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    P[i] = 0.f;
    n[i] = 0;
  }
  for (int t = t0; t < t1; ++t) {
    float v[8];
    token_probs(logits + (size_t)t * N, N, softmax, lane, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) P[i] += v[i];
    for (int j = 0; j < k; ++j) {
      const int e = topk_idx[(size_t)t * k + j];
      if ((unsigned)e >= (unsigned)N) {
        if (lane == 0) set_status(status, MOE_ERR_BOUNDS);
        continue;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) n[i] += (e == lane + 32 * i);
    }
  }
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) acc += (float)n[i] * P[i];
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) {
    const float Ls = (float)(t1 - t0);
    seq_loss[seq] = (float)N * (acc / (Ls * (float)k)) / Ls;
  }
}

// Router z-loss: per token log Z = m + log sum exp(z - m) (one warp per token),
// squared and summed per 32-token chunk; one CTA adds the chunks in order.
__global__ void __launch_bounds__(256) zloss_partial_kernel(const float *__restrict__ logits, int T, int N,
                                                            float *__restrict__ partial) {
  __shared__ float red[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc = 0.f;
  for (int tt = warp; tt < SC; tt += 8) {
    const int t = blockIdx.x * SC + tt;
    if (t >= T) break;
    const float *zr = logits + (size_t)t * N;
    float v[8];
    float m = -INFINITY;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int e = lane + 32 * i;
      v[i] = (e < N) ? zr[e] : -INFINITY;
      m = fmaxf(m, v[i]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i)
      if (lane + 32 * i < N) sum += expf(v[i] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    const float lse = m + logf(sum);
    acc += lse * lse;
  }
  if (lane == 0) red[warp] = acc;
  __syncthreads();
  if (threadIdx.x == 0) {
    float s = 0.f;
    for (int w = 0; w < 8; ++w) s += red[w];
    partial[blockIdx.x] = s;
  }
}

// Sum of partial[0 .. nchunks) in a fixed order, divided by T: the mean of the
// z-loss over tokens, or of the sequence losses over sequences.
__global__ void __launch_bounds__(1024) zloss_final_kernel(const float *__restrict__ partial, int nchunks, int T,
                                                           float *__restrict__ z_loss) {
  __shared__ float red[1024];
  float s = 0.f;
  for (int c = threadIdx.x; c < nchunks; c += 1024) s += partial[c];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int off = 512; off > 0; off >>= 1) {
    if (threadIdx.x < off) red[threadIdx.x] += red[threadIdx.x + off];
    __syncthreads();
  }
  if (threadIdx.x == 0) *z_loss = red[0] / (float)T;
}

__global__ void __launch_bounds__(256) bias_update_kernel(const int32_t *__restrict__ counts, int T, int k, int N,
                                                          float *__restrict__ sel_bias, float gamma) {
  const int e = threadIdx.x;
  if (e >= N) return;
  const long long lhs = (long long)counts[e] * N, rhs = (long long)T * k;
  if (lhs < rhs) sel_bias[e] += gamma;
  else if (lhs > rhs) sel_bias[e] -= gamma;
}

}  // namespace

int launch_router_zloss(const float *logits, int T, int N, float *partial, float *z_loss, cudaStream_t s) {
  const int nchunks = (T + SC - 1) / SC;
  zloss_partial_kernel<<<nchunks, 256, 0, s>>>(logits, T, N, partial);
  zloss_final_kernel<<<1, 1024, 0, s>>>(partial, nchunks, T, z_loss);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_bias_update(const int32_t *counts_routed, int T, int k, int N, float *sel_bias, float gamma,
                       cudaStream_t s) {
  bias_update_kernel<<<1, 256, 0, s>>>(counts_routed, T, k, N, sel_bias, gamma);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_load_stats(const float *logits, const int32_t *counts_routed, const int32_t *counts_kept, int T, int N,
                      long long total, int gate, float *partial, int *ticket, float *f, float *P, float *summary,
                      cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int nchunks = (T + SC - 1) / SC;
  if (nchunks == 1) {
    stats_one_chunk_kernel<<<1, 256, 0, s>>>(logits, T, N, gate, counts_routed, counts_kept, total, f, P, summary);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  stats_partial_kernel<<<nchunks, 256, 0, s>>>(logits, T, N, gate, T, nchunks, partial, ticket);
  stats_final_kernel<<<(N + 31) / 32, 1024, 0, s>>>(partial, nchunks, counts_routed, counts_kept, T, N, total, f, P,
                                                    summary, ticket);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int seq_balance_chunks(int T, int L) {
  L = min(L, T);
  return (int)(((long long)T + L - 1) / L) * ((L + SC - 1) / SC);
}

int launch_seq_balance_loss(const float *logits, const int32_t *topk_idx, int T, int N, int k, int gate, int L,
                            float *partial, float *seq_loss, float *loss, int *status, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  L = min(L, T);
  const int nseq = (int)(((long long)T + L - 1) / L);
  if (L >= SC) {
    const int cps = (L + SC - 1) / SC;
    stats_partial_kernel<<<nseq * cps, 256, 0, s>>>(logits, T, N, gate, L, cps, partial, nullptr);
    seq_final_kernel<<<nseq, 256, 0, s>>>(partial, cps, topk_idx, T, N, k, L, seq_loss, status);
  } else {
    seq_short_kernel<<<(nseq + 7) / 8, 256, 0, s>>>(logits, topk_idx, T, N, k, gate, L, nseq, seq_loss, status);
  }
  zloss_final_kernel<<<1, 1024, 0, s>>>(seq_loss, nseq, nseq, loss);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
