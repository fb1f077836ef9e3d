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
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SC = kStatsChunk;  // tokens per chunk

__global__ void __launch_bounds__(256) stats_partial_kernel(const float *__restrict__ logits, int T, int N, int gate,
                                                            float *__restrict__ partial) {
  __shared__ float red[8][256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;
  const int tb = blockIdx.x * SC;
  for (int tt = warp; tt < SC; tt += 8) {  // SC / 8 tokens per warp
    const int t = tb + tt;
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
    const bool softmax = gate != MOE_GATE_SIGMOID_BIAS;
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
    for (int i = 0; i < 8; ++i) acc[i] += v[i] * inv;
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

// One CTA of 1024 threads: four threads per expert each add every fourth chunk,
// then the four partial sums are added in a fixed order.
__global__ void __launch_bounds__(1024) stats_final_kernel(const float *__restrict__ partial, int nchunks,
                                                           const int32_t *__restrict__ counts_routed,
                                                           const int32_t *__restrict__ counts_kept, int T, int N,
                                                           long long total, float *__restrict__ f,
                                                           float *__restrict__ P, float *__restrict__ summary) {
  __shared__ float quarter[4][256];
  __shared__ float fp[256];
  __shared__ int maxc[256];
  __shared__ long long kept[256];
  const int e = threadIdx.x & 255, q = threadIdx.x >> 8;
  float s = 0.f;
  if (e < N)
    for (int c = q; c < nchunks; c += 4) s += partial[(size_t)c * N + e];
  quarter[q][e] = s;
  __syncthreads();
  if (q == 0) {
    float fe = 0.f, pe = 0.f;
    int ce = 0;
    long long ke = 0;
    if (e < N) {
      pe = (((quarter[0][e] + quarter[1][e]) + quarter[2][e]) + quarter[3][e]) / (float)T;
      ce = counts_routed[e];
      ke = counts_kept[e];
      fe = (float)((double)ce / (double)total);
      f[e] = fe;
      P[e] = pe;
    }
    fp[e] = fe * pe;
    maxc[e] = ce;
    kept[e] = ke;
  }
  __syncthreads();
  for (int off = 128; off > 0; off >>= 1) {
    if (q == 0 && e < off) {
      fp[e] += fp[e + off];
      maxc[e] = max(maxc[e], maxc[e + off]);
      kept[e] += kept[e + off];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double tk = (double)total;
    summary[0] = (float)N * fp[0];
    summary[1] = (float)((double)maxc[0] / (tk / (double)N));
    summary[2] = (float)(1.0 - (double)kept[0] / tk);
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
                      long long total, int gate, float *partial, float *f, float *P, float *summary, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int nchunks = (T + SC - 1) / SC;
  stats_partial_kernel<<<nchunks, 256, 0, s>>>(logits, T, N, gate, partial);
  stats_final_kernel<<<1, 1024, 0, s>>>(partial, nchunks, counts_routed, counts_kept, T, N, total, f, P, summary);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
