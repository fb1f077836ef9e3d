// Router of the layer: logits z = x . W_g (+ beta), top-k selection with ties to
// the lower expert index, and the gate weights.
//
// "Lecture29" (CS25 lecture 29 notes), section "Top-two routing": z = W_r x,
// S_k(x) = the k largest logits, g_i = exp(z_i) / sum_{j in S_k} exp(z_j).
// "Chapter 19: MoE" 19.3.4 and CS336 lecture 4 section 9: DeepSeek-V3 chooses on
// sigmoid(z) + b and mixes with the raw sigmoid affinities.  CS336 lecture 4,
// section 11: the router runs in float32.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int RT_TOK = 32;   // tokens per CTA (one per lane)
constexpr int RT_KC = 128;   // K chunk staged in shared memory
constexpr int RT_WARPS = 8;  // each warp owns RT_KC / RT_WARPS consecutive k of a chunk

// Logits for 32 tokens x EN experts.  Lane = token; the 8 warps split each K
// chunk, and their partial sums are added in warp order (deterministic).
// blockIdx.z picks a range of kc_per 128-wide K chunks; its sums go to
// logits + blockIdx.z * T * N (split partials, added in split order by the
// top-k kernel; the logit bias is then added there and logit_bias is null here).
template <int EN, bool BF16>
__global__ void __launch_bounds__(256) router_logits_kernel(const void *__restrict__ x, const float *__restrict__ Wg,
                                                            const float *__restrict__ logit_bias, int T, int d, int N,
                                                            int kc_per, float *__restrict__ logits) {
  constexpr int XS_LD = RT_KC + 1;
  constexpr int XS_FLOATS = RT_TOK * XS_LD;
  constexpr int WS_FLOATS = RT_KC * EN;
  constexpr int RED_FLOATS = RT_WARPS * RT_TOK * EN;
  constexpr int SMEM_FLOATS = (XS_FLOATS + WS_FLOATS) > RED_FLOATS ? (XS_FLOATS + WS_FLOATS) : RED_FLOATS;
  __shared__ __align__(16) float sm[SMEM_FLOATS];
  float *xs = sm;
  float *ws = sm + XS_FLOATS;

  const int t0 = blockIdx.x * RT_TOK;
  const int e0 = blockIdx.y * EN;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  float acc[EN];
#pragma unroll
  for (int e = 0; e < EN; ++e) acc[e] = 0.f;

  const int kbeg = blockIdx.z * kc_per * RT_KC;
  const int kend = min(d, kbeg + kc_per * RT_KC);
  logits += (size_t)blockIdx.z * T * N;
  for (int k0 = kbeg; k0 < kend; k0 += RT_KC) {
    // stage x[t0.., k0..k0+127] as float (8-element vectors; d % 8 == 0 / 4)
    for (int v = threadIdx.x; v < RT_TOK * (RT_KC / 8); v += blockDim.x) {
      const int tt = v / (RT_KC / 8), kk = (v % (RT_KC / 8)) * 8;
      const int t = t0 + tt, kg = k0 + kk;
      float f[8];
      if (t < T && kg < kend) {
        if (BF16) {
          const uint4 q = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + (size_t)t * d + kg);
          f[0] = bf16_lo(q.x); f[1] = bf16_hi(q.x); f[2] = bf16_lo(q.y); f[3] = bf16_hi(q.y);
          f[4] = bf16_lo(q.z); f[5] = bf16_hi(q.z); f[6] = bf16_lo(q.w); f[7] = bf16_hi(q.w);
        } else {
          const float *src = static_cast<const float *>(x) + (size_t)t * d + kg;
          const float4 a = *reinterpret_cast<const float4 *>(src);
          const float4 b = *reinterpret_cast<const float4 *>(src + 4);
          f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
        }
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) f[i] = 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) xs[tt * XS_LD + kk + i] = f[i];
    }
    // stage Wg[k0.., e0..e0+EN-1]
    for (int v = threadIdx.x; v < RT_KC * EN; v += blockDim.x) {
      const int kk = v / EN, e = v % EN;
      const int kg = k0 + kk, eg = e0 + e;
      ws[v] = (kg < kend && eg < N) ? Wg[(size_t)kg * N + eg] : 0.f;
    }
    __syncthreads();
    const int kb = warp * (RT_KC / RT_WARPS);
#pragma unroll 4
    for (int kk = kb; kk < kb + RT_KC / RT_WARPS; ++kk) {
      const float xv = xs[lane * XS_LD + kk];
      const float4 *wr = reinterpret_cast<const float4 *>(ws + kk * EN);
#pragma unroll
      for (int q = 0; q < EN / 4; ++q) {
        const float4 w4 = wr[q];
        acc[4 * q + 0] = fmaf(xv, w4.x, acc[4 * q + 0]);
        acc[4 * q + 1] = fmaf(xv, w4.y, acc[4 * q + 1]);
        acc[4 * q + 2] = fmaf(xv, w4.z, acc[4 * q + 2]);
        acc[4 * q + 3] = fmaf(xv, w4.w, acc[4 * q + 3]);
      }
    }
    __syncthreads();
  }
  // deterministic cross-warp reduction
  float *red = sm;
#pragma unroll
  for (int e = 0; e < EN; ++e) red[(warp * RT_TOK + lane) * EN + e] = acc[e];
  __syncthreads();
  for (int v = threadIdx.x; v < RT_TOK * EN; v += blockDim.x) {
    const int tt = v / EN, e = v % EN;
    const int t = t0 + tt, eg = e0 + e;
    if (t >= T || eg >= N) continue;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < RT_WARPS; ++w) s += red[(w * RT_TOK + tt) * EN + e];
    if (logit_bias) s += logit_bias[eg];
    logits[(size_t)t * N + eg] = s;
  }
}

// 32-bit key whose unsigned order is the float order (-0 and +0 equal).
__device__ __forceinline__ uint32_t order_key(float v) {
  if (v == 0.0f) v = 0.0f;
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One round of the warp's top-k: the untaken expert (lane + 32 i) with the largest
// key, the lowest index among equal keys (warp max of the keys, then warp min of
// the indices holding it).  Every valid key is > 0; key 0 marks "none".
template <int NV>
__device__ __forceinline__ int warp_select(const uint32_t (&key)[NV], uint32_t &taken, int lane, uint32_t *kmax) {
  uint32_t best = 0;
  int bi = 0;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (!((taken >> i) & 1u) && key[i] > best) {  // strict: the lowest i wins a tie within the lane
      best = key[i];
      bi = i;
    }
  const uint32_t m = __reduce_max_sync(0xffffffffu, best);
  const uint32_t cand = (best == m && m != 0u) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
  const int e = (int)__reduce_min_sync(0xffffffffu, cand);
  if ((e & 31) == lane) taken |= 1u << (e >> 5);
  *kmax = m;
  return e;
}

__device__ __forceinline__ float sigmoid_f32(float z) {
  // evaluated in double and rounded once, as the selection decision is
  return (float)(1.0 / (1.0 + exp(-(double)z)));
}

// One warp per token; lane l holds experts l, l+32, ... (N <= 256).  The logits
// are the sum of S partial tiles (row stride pstride, tile stride T * pstride),
// added in split order, plus the optional logit bias; they are written to
// `logits` (which may alias the only partial when S == 1 and no bias is added).
template <int NV>  // expert slots per lane: N <= 32 NV
__global__ void __launch_bounds__(256) router_topk_kernel(const float *partial, int S, int pstride,
                                                          const float *__restrict__ logit_bias, float *logits,
                                                          const float *__restrict__ sel_bias, int T, int N, int k,
                                                          int gate, int32_t *__restrict__ idx, float *__restrict__ w,
                                                          int *status) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  float zl[NV];  // this lane's logits, kept in registers
  float sel[NV];
  bool bad = false;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    zl[i] = -INFINITY;
    if (e < N) {
      // four independent running sums over the splits, combined in a fixed order
      const float *p = partial + (size_t)t * pstride + e;
      const size_t tile = (size_t)T * pstride;
      float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
      int sp = 0;
      for (; sp + 4 <= S; sp += 4) {
        z0 += p[(sp + 0) * tile];
        z1 += p[(sp + 1) * tile];
        z2 += p[(sp + 2) * tile];
        z3 += p[(sp + 3) * tile];
      }
      for (; sp < S; ++sp) z0 += p[sp * tile];
      float z = (z0 + z1) + (z2 + z3);
      if (logit_bias) z += logit_bias[e];
      logits[(size_t)t * N + e] = z;
      zl[i] = z;
    }
  }
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int e = lane + 32 * i;
    sel[i] = -INFINITY;
    if (e < N) {
      const float z = zl[i];
      if (!isfinite(z)) bad = true;
      float s = z;
      if (gate == MOE_GATE_SIGMOID_BIAS) {
        s = 1.0f / (1.0f + expf(-z));  // estimate, see below
        if (sel_bias) s = s + sel_bias[e];
      }
      sel[i] = s;
    }
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MOE_ERR_NONFINITE);
  uint32_t key[NV];
#pragma unroll
  for (int i = 0; i < NV; ++i) key[i] = (lane + 32 * i < N) ? order_key(sel[i]) : 0u;
  int chosen[8];
  bool done = false;
  if (gate == MOE_GATE_SIGMOID_BIAS) {
    // The selection score is fl32(s + b) with s = fl32(sigmoid(z)) evaluated in
    // double.  The float32 estimate above (expf within 2 ulp, then one add and
    // one division) is within kEstErr of it.  If the k + 1 largest estimates are
    // more than 2 kEstErr apart from one another (checked with a factor 2 to spare),
    // the exact scores rank exactly as
    // the estimates do (and nothing below the (k+1)-th can overtake the k-th), so
    // the estimates decide.  Otherwise (a near tie) every expert within kSelMargin
    // of the k-th estimate is evaluated in double and ranked again; the rest
    // cannot be in the top k.
    constexpr float kEstErr = 5.4e-7f, kSelMargin = 4e-6f;
    uint32_t taken0 = 0, kv[9];
    int ch0[9];
    const int rounds = min(k + 1, N);
#pragma unroll
    for (int j = 0; j < 9; ++j)
      if (j < rounds) ch0[j] = warp_select(key, taken0, lane, &kv[j]);
    bool clear = true;
#pragma unroll
    for (int j = 0; j < 8; ++j)  // 4 kEstErr: twice the bound, covering the rounding of the gap itself
      if (j + 1 < rounds) clear = clear && (key_value(kv[j]) - key_value(kv[j + 1]) > 4.0f * kEstErr);
    if (clear) {
#pragma unroll
      for (int j = 0; j < 8; ++j) chosen[j] = ch0[j];
      done = true;
    } else {
      uint32_t kk = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j == k - 1) kk = kv[j];
      const float vk = key_value(kk);
#pragma unroll
      for (int i = 0; i < NV; ++i) {
        const int e = lane + 32 * i;
        if (e >= N) continue;
        if (sel[i] >= vk - kSelMargin) {
          float se = sigmoid_f32(zl[i]);
          if (sel_bias) se = se + sel_bias[e];
          key[i] = order_key(se);
        } else {
          key[i] = order_key(-INFINITY);
        }
      }
    }
  }
  if (!done) {
    uint32_t taken = 0, kmax;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k) chosen[j] = warp_select(key, taken, lane, &kmax);
  }
  // the chosen experts' logits, from the lanes that hold them: lane j < k gets slot j's
  float zj = 0.f, m = 0.f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < k) {
      const int e = chosen[j];
      float mine = zl[0];
#pragma unroll
      for (int i = 1; i < NV; ++i)
        if ((e >> 5) == i) mine = zl[i];
      const float ze = __shfl_sync(0xffffffffu, mine, e & 31);
      if (lane == j) zj = ze;
      if (j == 0) m = ze;  // the first pick has the largest logit (softmax gates)
    }
  }
  // full-softmax gate: the normaliser over all N experts (warp sum, fixed order)
  float full_den = 0.f;
  if (gate == MOE_GATE_SOFTMAX_FULL) {
#pragma unroll
    for (int i = 0; i < NV; ++i)
      if (lane + 32 * i < N) full_den += expf(zl[i] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) full_den += __shfl_xor_sync(0xffffffffu, full_den, off);
  }
  // gate weights of the selected experts, in float32: lane j < k takes slot j;
  // the normaliser is a warp sum in a fixed order
  float g = 0.f;
  if (gate == MOE_GATE_SOFTMAX_TOPK || gate == MOE_GATE_SOFTMAX_FULL) {
    if (lane < k) g = expf(zj - m);
  } else if (lane < k) {
    g = 1.0f / (1.0f + expf(-zj));  // float32 affinity (within 3e-7 relative of the rounded exact one)
  }
  float sum = g;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (gate == MOE_GATE_SOFTMAX_FULL) sum = full_den;
  if (lane < k) {
    int cj = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < k && lane == j) cj = chosen[j];
    idx[(size_t)t * k + lane] = cj;
    w[(size_t)t * k + lane] = g / sum;
  }
}

// logits[t, e] = sum of the S split partials in split order + logit bias
__global__ void __launch_bounds__(256) router_sum_kernel(const float *__restrict__ partial, int S, int pstride,
                                                         const float *__restrict__ logit_bias,
                                                         float *__restrict__ logits, int T, int N) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * N) return;
  const int t = (int)(i / N), e = (int)(i % N);
  const float *p = partial + (size_t)t * pstride + e;
  const size_t tile = (size_t)T * pstride;
  float z0 = 0.f, z1 = 0.f, z2 = 0.f, z3 = 0.f;
  int sp = 0;
  for (; sp + 4 <= S; sp += 4) {
    z0 += p[(sp + 0) * tile];
    z1 += p[(sp + 1) * tile];
    z2 += p[(sp + 2) * tile];
    z3 += p[(sp + 3) * tile];
  }
  for (; sp < S; ++sp) z0 += p[sp * tile];
  float z = (z0 + z1) + (z2 + z3);
  if (logit_bias) z += logit_bias[e];
  logits[i] = z;
}

}  // namespace

int launch_router_sum(const float *partial, int S, int pstride, const float *logit_bias, float *logits, int T, int N,
                      cudaStream_t s) {
  const size_t n = (size_t)T * N;
  if (n == 0) return MOE_OK;
  router_sum_kernel<<<(unsigned)((n + 255) / 256), 256, 0, s>>>(partial, S, pstride, logit_bias, logits, T, N);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_router_logits(const void *x, bool x_bf16, const float *Wg, const float *logit_bias, int T, int d, int N,
                         int splits, float *logits, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const int en = N <= 8 ? 8 : (N <= 16 ? 16 : 32);
  const int nkc = (d + RT_KC - 1) / RT_KC;
  if (splits < 1) splits = 1;
  const int kc_per = (nkc + splits - 1) / splits;
  splits = (nkc + kc_per - 1) / kc_per;  // every split non-empty
  dim3 grid((T + RT_TOK - 1) / RT_TOK, (N + en - 1) / en, splits), block(256);
#define MOE_RL(EN)                                                                                           \
  if (x_bf16)                                                                                                \
    router_logits_kernel<EN, true><<<grid, block, 0, s>>>(x, Wg, logit_bias, T, d, N, kc_per, logits);      \
  else                                                                                                       \
    router_logits_kernel<EN, false><<<grid, block, 0, s>>>(x, Wg, logit_bias, T, d, N, kc_per, logits);
  if (en == 8) {
    MOE_RL(8)
  } else if (en == 16) {
    MOE_RL(16)
  } else {
    MOE_RL(32)
  }
#undef MOE_RL
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_router_topk(const float *partial, int S, int pstride, const float *logit_bias, float *logits,
                       const float *sel_bias, int T, int N, int k, int gate, int32_t *idx, float *w, int *status,
                       cudaStream_t s) {
  if (T == 0) return MOE_OK;
  const dim3 grid((T + 7) / 8), block(256);
  if (N <= 32)
    router_topk_kernel<1><<<grid, block, 0, s>>>(partial, S, pstride, logit_bias, logits, sel_bias, T, N, k, gate, idx,
                                                 w, status);
  else if (N <= 64)
    router_topk_kernel<2><<<grid, block, 0, s>>>(partial, S, pstride, logit_bias, logits, sel_bias, T, N, k, gate, idx,
                                                 w, status);
  else if (N <= 128)
    router_topk_kernel<4><<<grid, block, 0, s>>>(partial, S, pstride, logit_bias, logits, sel_bias, T, N, k, gate, idx,
                                                 w, status);
  else
    router_topk_kernel<8><<<grid, block, 0, s>>>(partial, S, pstride, logit_bias, logits, sel_bias, T, N, k, gate, idx,
                                                 w, status);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
