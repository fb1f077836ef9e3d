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
__device__ __forceinline__ int warp_select(const uint32_t (&key)[NV], const float (&zl)[NV], uint32_t &taken,
                                           int lane, uint32_t *kmax, float *zwin) {
  uint32_t best = 0;
  int bi = 0;
  float zb = 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i)
    if (!((taken >> i) & 1u) && key[i] > best) {  // strict: the lowest i wins a tie within the lane
      best = key[i];
      bi = i;
      zb = zl[i];
    }
  const uint32_t m = __reduce_max_sync(0xffffffffu, best);
  const uint32_t cand = (best == m && m != 0u) ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu;
  const int e = (int)__reduce_min_sync(0xffffffffu, cand);
  if ((e & 31) == lane) taken |= 1u << (e >> 5);
  *kmax = m;
  *zwin = __shfl_sync(0xffffffffu, zb, e & 31);  // the winner's logit, from the lane holding it
  return e;
}

__device__ __forceinline__ float sigmoid_f32(float z) {
  // evaluated in double and rounded once, as the selection decision is
  return (float)(1.0 / (1.0 + exp(-(double)z)));
}

// Top-k and gate of token t, called by a whole warp: lane l holds the logits of
// experts l, l + 32, ... (N <= 32 NV; -inf past N).  Writes idx[t, :] and w[t, :];
// a non-finite logit sets MOE_ERR_NONFINITE.
template <int NV>
__device__ __forceinline__ void route_token(const float (&zl)[NV], int t, int lane, int N, int k, int gate,
                                            const float *__restrict__ sel_bias, int32_t *__restrict__ idx,
                                            float *__restrict__ w, int *status) {
  float sel[NV];
  bool bad = false;
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
  // slot j's expert and logit are kept by lane j (j < k), as each round picks them
  int ej = 0;
  float zj = 0.f, m = 0.f;
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
    uint32_t taken0 = 0, kprev = 0, kk = 0;
    bool clear = true;
    const int rounds = min(k + 1, N);
#pragma unroll
    for (int j = 0; j < 9; ++j) {
      if (j >= rounds) break;
      uint32_t kw;
      float zw;
      const int e = warp_select(key, zl, taken0, lane, &kw, &zw);
      // 4 kEstErr: twice the bound, covering the rounding of the gap itself
      if (j > 0) clear = clear && (key_value(kprev) - key_value(kw) > 4.0f * kEstErr);
      if (j == k - 1) kk = kw;
      if (j < k && lane == j) {
        ej = e;
        zj = zw;
      }
      kprev = kw;
    }
    if (clear) {
      done = true;
    } else {
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
    uint32_t taken = 0;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      if (j >= k) break;
      uint32_t kw;
      float zw;
      const int e = warp_select(key, zl, taken, lane, &kw, &zw);
      if (lane == j) {
        ej = e;
        zj = zw;
      }
      if (j == 0) m = zw;  // the first pick has the largest logit (softmax gates)
    }
  } else {
    m = __shfl_sync(0xffffffffu, zj, 0);
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
    idx[(size_t)t * k + lane] = ej;
    w[(size_t)t * k + lane] = g / sum;
  }
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
  route_token<NV>(zl, t, lane, N, k, gate, sel_bias, idx, w, status);
}

// The whole route in one launch for a few experts (N = 4 or 8) and float32
// activations past the decode sizes: logits on the CUDA cores, then top-k and gate
// in the same CTA (the logits never make a round trip through memory before the
// selection).  Used for float32 x, where it replaces the two-launch CUDA-core
// route (9.0 us against 12.5 us on the 256-token, d = 512 float32 layer).  For
// bf16 x the tensor-core route stays faster (18.8 us against 40.8 us on the
// 4096-token Mixtral shape): every CTA reads each W_g row once, so those loads
// miss L1, and with one CTA of eight warps per SM their latency is not hidden.
//
// CTA = 32 tokens x 8 warps.  Warp w takes the K range [w kw, (w + 1) kw) (kw a
// multiple of 16); lane l takes tokens t0 + (l & 15) and t0 + 16 + (l & 15) and,
// of every 16 consecutive k, the 8 at offset 8 (l >> 4), so a load of 8 values of
// x is 16 bytes, the two half-warps together read 32-byte sectors whole, and each
// W_g row (NW floats, 16-byte vectors, the same for the half-warp) feeds 2 NW
// products.  Sums: per 128-wide block of K in float32 (fused multiply-adds in k
// order), the blocks added in order, the two half-warps added (lower half first),
// then the eight warps' sums in warp order plus the logit bias: deterministic.
constexpr int RF_TOK = 32;
constexpr int RF_WARPS = 8;
constexpr int RF_GROUPS = 8;  // 16-wide groups of K per block: 128 k, 8 loads of x in flight per lane

// 8 consecutive values of x at element offset `off`, raw: one 16-byte vector of
// bf16 or two of float32; value j of a raw vector as float32.
template <bool BF16>
struct XRaw {
  uint4 q[BF16 ? 1 : 2];
};
template <bool BF16>
__device__ __forceinline__ XRaw<BF16> load_x8(const void *x, size_t off) {
  XRaw<BF16> r;
  if (BF16) {
    r.q[0] = __ldg(reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(x) + off));
  } else {
    const uint4 *p = reinterpret_cast<const uint4 *>(static_cast<const float *>(x) + off);
    r.q[0] = __ldg(p);
    r.q[BF16 ? 0 : 1] = __ldg(p + 1);
  }
  return r;
}
template <bool BF16>
__device__ __forceinline__ float x_at(const XRaw<BF16> &r, int j) {
  if (BF16) {
    const uint32_t wv = j < 2 ? r.q[0].x : (j < 4 ? r.q[0].y : (j < 6 ? r.q[0].z : r.q[0].w));
    return (j & 1) ? bf16_hi(wv) : bf16_lo(wv);
  }
  const uint4 &q = r.q[j >> 2];
  const uint32_t wv = (j & 3) == 0 ? q.x : ((j & 3) == 1 ? q.y : ((j & 3) == 2 ? q.z : q.w));
  return __uint_as_float(wv);
}

template <bool BF16, int NW>
__global__ void __launch_bounds__(256) router_fused_kernel(const void *__restrict__ x, const float *__restrict__ Wg,
                                                           const float *__restrict__ logit_bias,
                                                           const float *__restrict__ sel_bias, int T, int d, int k,
                                                           int gate, int kw, float *__restrict__ logits,
                                                           int32_t *__restrict__ idx, float *__restrict__ w,
                                                           int *status) {
  __shared__ float red[RF_WARPS][RF_TOK][NW];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tl = lane & 15, h = lane >> 4;
  const int t0 = blockIdx.x * RF_TOK;
  const int ta = t0 + tl, tb = t0 + 16 + tl;
  const bool va = ta < T, vb = tb < T;
  const int kbeg = warp * kw, kend = min(d, kbeg + kw);
  float acc[2][NW];
#pragma unroll
  for (int e = 0; e < NW; ++e) acc[0][e] = acc[1][e] = 0.f;
  for (int k0 = kbeg; k0 < kend; k0 += 16 * RF_GROUPS) {
    XRaw<BF16> xa[RF_GROUPS], xb[RF_GROUPS];
#pragma unroll
    for (int g = 0; g < RF_GROUPS; ++g) {
      const int kk = k0 + 16 * g + 8 * h;
      const bool in = kk < kend;  // the group's 8 values are all in or all out (d % 8 == 0)
      xa[g] = (in && va) ? load_x8<BF16>(x, (size_t)ta * d + kk) : XRaw<BF16>{};
      xb[g] = (in && vb) ? load_x8<BF16>(x, (size_t)tb * d + kk) : XRaw<BF16>{};
    }
    float ca[NW], cb[NW];
#pragma unroll
    for (int e = 0; e < NW; ++e) ca[e] = cb[e] = 0.f;
#pragma unroll
    for (int g = 0; g < RF_GROUPS; ++g) {
      const int kk = k0 + 16 * g + 8 * h;
      if (kk >= kend) continue;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float4 *wr = reinterpret_cast<const float4 *>(Wg + (size_t)(kk + j) * NW);
        const float xja = x_at<BF16>(xa[g], j), xjb = x_at<BF16>(xb[g], j);
#pragma unroll
        for (int q = 0; q < NW / 4; ++q) {
          const float4 w4 = __ldg(wr + q);
          ca[4 * q + 0] = fmaf(xja, w4.x, ca[4 * q + 0]);
          ca[4 * q + 1] = fmaf(xja, w4.y, ca[4 * q + 1]);
          ca[4 * q + 2] = fmaf(xja, w4.z, ca[4 * q + 2]);
          ca[4 * q + 3] = fmaf(xja, w4.w, ca[4 * q + 3]);
          cb[4 * q + 0] = fmaf(xjb, w4.x, cb[4 * q + 0]);
          cb[4 * q + 1] = fmaf(xjb, w4.y, cb[4 * q + 1]);
          cb[4 * q + 2] = fmaf(xjb, w4.z, cb[4 * q + 2]);
          cb[4 * q + 3] = fmaf(xjb, w4.w, cb[4 * q + 3]);
        }
      }
    }
#pragma unroll
    for (int e = 0; e < NW; ++e) {
      acc[0][e] += ca[e];
      acc[1][e] += cb[e];
    }
  }
  // the two halves of K, lower half first
#pragma unroll
  for (int e = 0; e < NW; ++e) {
    const float ua = __shfl_down_sync(0xffffffffu, acc[0][e], 16);
    const float ub = __shfl_down_sync(0xffffffffu, acc[1][e], 16);
    if (h == 0) {
      red[warp][tl][e] = acc[0][e] + ua;
      red[warp][16 + tl][e] = acc[1][e] + ub;
    }
  }
  __syncthreads();
  // warp w routes tokens 4 w .. 4 w + 3 of the CTA; lane e < NW holds expert e
  for (int i = 0; i < RF_TOK / RF_WARPS; ++i) {
    const int tt = warp * (RF_TOK / RF_WARPS) + i;
    const int t = t0 + tt;
    if (t >= T) break;
    float zl[1] = {-INFINITY};
    if (lane < NW) {
      float z = 0.f;
#pragma unroll
      for (int ww = 0; ww < RF_WARPS; ++ww) z += red[ww][tt][lane];
      if (logit_bias) z += logit_bias[lane];
      logits[(size_t)t * NW + lane] = z;
      zl[0] = z;
    }
    route_token<1>(zl, t, lane, NW, k, gate, sel_bias, idx, w, status);
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

bool router_fused_fits(int T, int d, int N) { return T > 0 && (N == 4 || N == 8) && d % 8 == 0 && d > 0; }

int launch_router_fused(const void *x, bool x_bf16, const float *Wg, const float *logit_bias,
                        const float *sel_bias, int T, int d, int N, int k, int gate, float *logits, int32_t *idx,
                        float *w, int *status, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  if (!router_fused_fits(T, d, N) || (reinterpret_cast<uintptr_t>(Wg) & 15) ||
      (reinterpret_cast<uintptr_t>(x) & 15))
    return MOE_ERR_UNSUPPORTED;
  const int kw = (d + 16 * RF_WARPS - 1) / (16 * RF_WARPS) * 16;
  const dim3 grid((T + RF_TOK - 1) / RF_TOK), block(32 * RF_WARPS);
#define MOE_RF(B, NW) \
  router_fused_kernel<B, NW><<<grid, block, 0, s>>>(x, Wg, logit_bias, sel_bias, T, d, k, gate, kw, logits, idx, w, status)
  if (x_bf16) {
    if (N == 8) MOE_RF(true, 8); else MOE_RF(true, 4);
  } else {
    if (N == 8) MOE_RF(false, 8); else MOE_RF(false, 4);
  }
#undef MOE_RF
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
