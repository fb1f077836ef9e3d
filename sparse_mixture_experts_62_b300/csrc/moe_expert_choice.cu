// Expert-choice routing: every expert picks the C tokens with the largest scores.
//
// "Chapter 19: MoE", 19.6.1: with expert choice each expert selects a fixed
// number of tokens, and a token may be processed by any number of experts.
// CS336 lecture 4, section 4: it is top-K taken along the token axis of the
// score matrix, so every expert receives exactly the same number of tokens.
// Scores are the full softmax over experts of each token's logits (CS336
// lecture 4, section 5); ties go to the lower token index; the gate of (t, e) is
// the score itself.  An expert's rows are its chosen tokens in ascending order.
//
//   ec_scores_kernel  one warp per token: softmax over the N logits -> scores
//                     [T, N]; the token's row map dest_row [T, N] set to -1.
//   ec_select_kernel  one CTA per expert: radix selection of the C-th largest
//                     score (4 passes over the 32-bit orderable score), then a
//                     block-wide compaction in token order that takes every token
//                     above it and the lowest-indexed ones equal to it.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int EC_THREADS = 1024;

__global__ void __launch_bounds__(256) ec_scores_kernel(const float *__restrict__ logits, int T, int N,
                                                        float *__restrict__ scores, int32_t *__restrict__ dest_row) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
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
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    v[i] = (e < N) ? expf(v[i] - m) : 0.f;
    sum += v[i];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  const float inv = 1.0f / sum;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int e = lane + 32 * i;
    if (e < N) {
      scores[(size_t)t * N + e] = v[i] * inv;
      dest_row[(size_t)t * N + e] = -1;
    }
  }
}

__device__ __forceinline__ uint32_t order_bits(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide prefix sum of one int per thread (EC_THREADS threads).
__device__ int block_exclusive_scan(int v, int *warp_sums, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_sums[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int w = warp_sums[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, w, off);
      if (lane >= off) w += y;
    }
    warp_sums[lane] = w;  // inclusive over warps
  }
  __syncthreads();
  const int before = (warp > 0 ? warp_sums[warp - 1] : 0) + x - v;
  if (total) *total = warp_sums[31];
  __syncthreads();
  return before;
}

// One CTA per expert e.  Each thread owns a contiguous run of tokens, so a
// block-wide prefix over threads visits tokens in ascending order.
__global__ void __launch_bounds__(EC_THREADS) ec_select_kernel(const float *__restrict__ scores, int T, int N, int C,
                                                               int32_t *__restrict__ offsets,
                                                               int32_t *__restrict__ src_token,
                                                               int32_t *__restrict__ dest_row) {
  __shared__ int hist[256];
  __shared__ int warp_sums[32];
  __shared__ uint32_t s_prefix;
  __shared__ int s_need;
  __shared__ int s_total;
  const int e = blockIdx.x;
  const int per = (T + EC_THREADS - 1) / EC_THREADS;
  const int t0 = threadIdx.x * per;
  const int t1 = min(T, t0 + per);
  if (threadIdx.x == 0) {
    offsets[e] = e * C;
    if (e == N - 1) offsets[N] = N * C;
    s_prefix = 0;
    s_need = C;  // how many of the largest keys are still to be placed at or below the prefix
  }
  __syncthreads();
  // radix selection of the C-th largest orderable score, most significant byte first
  uint32_t mask = 0;
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += EC_THREADS) hist[i] = 0;
    __syncthreads();
    const uint32_t prefix = s_prefix;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = order_bits(scores[(size_t)t * N + e]);
      if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1);
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int need = s_need, digit = 255;
      for (; digit > 0; --digit) {  // from the largest digit down
        if (hist[digit] >= need) break;
        need -= hist[digit];
      }
      s_need = need;
      s_prefix = prefix | ((uint32_t)digit << shift);
    }
    __syncthreads();
    mask |= 255u << shift;
  }
  const uint32_t kth = s_prefix;  // the C-th largest key
  const int take_equal = s_need;  // how many keys equal to it are chosen (lowest tokens first)
  // ordered compaction: above the threshold, or equal and among the first take_equal
  int n_eq = 0;
  for (int t = t0; t < t1; ++t) n_eq += order_bits(scores[(size_t)t * N + e]) == kth;
  int eq_before = block_exclusive_scan(n_eq, warp_sums, nullptr);
  int n_pick = 0;
  {
    int eq = eq_before;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = order_bits(scores[(size_t)t * N + e]);
      if (k > kth) ++n_pick;
      else if (k == kth) n_pick += (eq++ < take_equal);
    }
  }
  int row = block_exclusive_scan(n_pick, warp_sums, &s_total);
  {
    int eq = eq_before;
    for (int t = t0; t < t1; ++t) {
      const uint32_t k = order_bits(scores[(size_t)t * N + e]);
      bool pick = k > kth;
      if (k == kth) pick = eq++ < take_equal;
      if (pick) {
        const int r = e * C + row++;
        src_token[r] = t;
        dest_row[(size_t)t * N + e] = r;
      }
    }
  }
}

__global__ void fill_counts_kernel(int32_t *counts_routed, int32_t *counts_kept, int N, int C) {
  const int e = blockIdx.x * blockDim.x + threadIdx.x;
  if (e < N) {
    counts_routed[e] = C;
    counts_kept[e] = C;
  }
}

}  // namespace

int launch_fill_counts(int32_t *counts_routed, int32_t *counts_kept, int N, int C, cudaStream_t s) {
  fill_counts_kernel<<<(N + 255) / 256, 256, 0, s>>>(counts_routed, counts_kept, N, C);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_expert_choice(const float *logits, int T, int N, int C, float *scores, int32_t *offsets,
                         int32_t *src_token, int32_t *dest_row, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  ec_scores_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, T, N, scores, dest_row);
  ec_select_kernel<<<N, EC_THREADS, 0, s>>>(scores, T, N, C, offsets, src_token, dest_row);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
