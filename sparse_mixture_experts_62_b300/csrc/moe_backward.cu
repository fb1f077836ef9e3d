// Backward pass of the layer with the routing held fixed: the element-wise and
// router kernels around the tensor-core GEMMs.
//
// "Chapter 19: MoE", 19.6.2: the top-k choice is discrete, so the task gradient
// reaches the router only through the gate weights of the chosen experts and
// each expert only through the tokens it processed.  With out[t] = sum_j w_tj y_tj:
//   dy_tj = w_tj dout[t]                      (into the expert backward)
//   dw_tj = <dout[t], y_tj>                   (into the gate backward)
//   softmax over the selected:  dz_j = w_j (dw_j - sum_l w_l dw_l)
//   full softmax:               dz_i = p_i (g_i - sum_l p_l g_l), g = dw on the selected
//   sigmoid, w = s / sum s:     dz_j = (dw_j - sum_l w_l dw_l) / sum s * s_j (1 - s_j)
//   SwiGLU h = SiLU(a) u:       da = dh u SiLU'(a), du = dh SiLU(a),
//                               SiLU'(a) = sig(a) (1 + a (1 - sig(a)))
// Dropped assignments contribute nothing (CS336 lecture 4, section 10).
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

__global__ void zero_f32_kernel(float *p, size_t n) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) p[i] = 0.f;
}

// One warp per kept row r: dy[r] = w_tj dout[t] (bf16), dgate[t, j] = <dout[t], y_perm[r]>.
__global__ void __launch_bounds__(256) dy_dgate_kernel(const uint16_t *__restrict__ dout,
                                                       const uint16_t *__restrict__ y_perm,
                                                       const float *__restrict__ topk_w,
                                                       const int32_t *__restrict__ dest_row,
                                                       const int32_t *__restrict__ src_token,
                                                       const int32_t *__restrict__ rows_end, int k, int d,
                                                       uint16_t *__restrict__ dy, float *__restrict__ dgate) {
  const int rows = *rows_end;
  const int warps = gridDim.x * 8;
  for (int r = blockIdx.x * 8 + (threadIdx.x >> 5); r < rows; r += warps) {
    const int lane = threadIdx.x & 31;
    const int t = src_token[r];
    int j = 0;
    while (j < k - 1 && dest_row[(size_t)t * k + j] != r) ++j;
    const float w = topk_w[(size_t)t * k + j];
    float dot = 0.f;
    for (int c = lane * 8; c < d; c += 256) {
      const uint4 g = *reinterpret_cast<const uint4 *>(dout + (size_t)t * d + c);
      const uint4 y = *reinterpret_cast<const uint4 *>(y_perm + (size_t)r * d + c);
      const uint32_t gv[4] = {g.x, g.y, g.z, g.w}, yv[4] = {y.x, y.y, y.z, y.w};
      uint32_t o[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float g0 = bf16_lo(gv[q]), g1 = bf16_hi(gv[q]);
        dot = fmaf(g0, bf16_lo(yv[q]), dot);
        dot = fmaf(g1, bf16_hi(yv[q]), dot);
        o[q] = pack_bf16x2(w * g0, w * g1);
      }
      *reinterpret_cast<uint4 *>(dy + (size_t)r * d + c) = make_uint4(o[0], o[1], o[2], o[3]);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, off);
    if (lane == 0) dgate[(size_t)t * k + j] = dot;
  }
}

// One warp per token: dz [T, N] from the gate gradients of the kept slots.
__global__ void __launch_bounds__(256) router_bwd_kernel(const float *__restrict__ logits,
                                                         const int32_t *__restrict__ idx,
                                                         const float *__restrict__ topk_w,
                                                         const float *__restrict__ dgate, int gate, int T, int N,
                                                         int k, float *__restrict__ dz) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  if (t >= T) return;
  const float *zr = logits + (size_t)t * N;
  float *dzr = dz + (size_t)t * N;
  // sum_l w_l g_l over the selected slots (dropped slots have g = 0)
  float wg = 0.f;
  for (int j = 0; j < k; ++j) wg += topk_w[(size_t)t * k + j] * dgate[(size_t)t * k + j];
  if (gate == MOE_GATE_SOFTMAX_FULL) {
    float m = -INFINITY;
    for (int e = lane; e < N; e += 32) m = fmaxf(m, zr[e]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
    float sum = 0.f;
    for (int e = lane; e < N; e += 32) sum += expf(zr[e] - m);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    // sum_l p_l g_l = sum_l w_l g_l (the gate weights are the selected p)
    for (int e = lane; e < N; e += 32) {
      float g = 0.f;
      for (int j = 0; j < k; ++j)
        if (idx[(size_t)t * k + j] == e) g = dgate[(size_t)t * k + j];
      dzr[e] = expf(zr[e] - m) / sum * (g - wg);
    }
    return;
  }
  for (int e = lane; e < N; e += 32) dzr[e] = 0.f;
  __syncwarp();
  if (lane == 0) {
    float ssum = 0.f;
    if (gate == MOE_GATE_SIGMOID_BIAS)
      for (int j = 0; j < k; ++j) ssum += 1.0f / (1.0f + expf(-zr[idx[(size_t)t * k + j]]));
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      const float g = dgate[(size_t)t * k + j], w = topk_w[(size_t)t * k + j];
      if (gate == MOE_GATE_SOFTMAX_TOPK) {
        dzr[e] = w * (g - wg);
      } else {
        const float s = 1.0f / (1.0f + expf(-zr[e]));
        dzr[e] = (g - wg) / ssum * s * (1.0f - s);
      }
    }
  }
}

// dz [T, N] float32 -> [T, 2 Np] bf16: columns e = bf16(dz), Np + e = bf16(dz -
// bf16(dz)), zero past N.  With x exact in bf16, x^T [hi | lo] on the tensor cores
// gives x^T dz to about 2^-16 relative (two-term split, every product exact).
__global__ void split_dz_kernel(const float *__restrict__ dz, int T, int N, int Np, uint16_t *__restrict__ out) {
  const size_t n = (size_t)T * Np;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int t = (int)(i / Np), e = (int)(i % Np);
    const float v = e < N ? dz[(size_t)t * N + e] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    out[(size_t)t * 2 * Np + e] = __bfloat16_as_ushort(hi);
    out[(size_t)t * 2 * Np + Np + e] = __bfloat16_as_ushort(lo);
  }
}

// dWg[c][e] = part[c][e] + part[c][Np + e]: the hi and lo halves of x^T [hi | lo].
__global__ void dwg_sum_kernel(const float *__restrict__ part, int d, int N, int Np, float *__restrict__ dWg) {
  const size_t n = (size_t)d * N;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int c = (int)(i / N), e = (int)(i % N);
    dWg[i] = part[(size_t)c * 2 * Np + e] + part[(size_t)c * 2 * Np + Np + e];
  }
}

// dx[t] = sum_j kept dx_perm[row_tj] + sum_e dz[t][e] Wg[:, e] (+ the shared expert's dx).
// dx[t] = sum_j kept dx_perm[row_tj] + router term [t] (+ the shared expert's dx);
// 8 columns per thread with 16-byte loads (d is a multiple of 8).
__global__ void __launch_bounds__(256) dx_combine_kernel(const uint16_t *__restrict__ dxp,
                                                         const int32_t *__restrict__ dest_row,
                                                         const float *__restrict__ rterm,
                                                         const uint16_t *__restrict__ dx_sh, int T, int d, int k,
                                                         float *__restrict__ dx) {
  const int t = blockIdx.x;
  __shared__ int rows[8];
  if (threadIdx.x < k) rows[threadIdx.x] = dest_row[(size_t)t * k + threadIdx.x];
  __syncthreads();
  for (int c = threadIdx.x * 8; c < d; c += blockDim.x * 8) {
    float acc[8];
    const float4 r0 = *reinterpret_cast<const float4 *>(rterm + (size_t)t * d + c);
    const float4 r1 = *reinterpret_cast<const float4 *>(rterm + (size_t)t * d + c + 4);
    acc[0] = r0.x, acc[1] = r0.y, acc[2] = r0.z, acc[3] = r0.w, acc[4] = r1.x, acc[5] = r1.y, acc[6] = r1.z,
    acc[7] = r1.w;
    if (dx_sh) {
      const uint4 q = *reinterpret_cast<const uint4 *>(dx_sh + (size_t)t * d + c);
      const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += bf16_lo(v[i]);
        acc[2 * i + 1] += bf16_hi(v[i]);
      }
    }
    for (int j = 0; j < k; ++j) {
      if (rows[j] < 0) continue;
      const uint4 q = *reinterpret_cast<const uint4 *>(dxp + (size_t)rows[j] * d + c);
      const uint32_t v[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        acc[2 * i] += bf16_lo(v[i]);
        acc[2 * i + 1] += bf16_hi(v[i]);
      }
    }
    *reinterpret_cast<float4 *>(dx + (size_t)t * d + c) = make_float4(acc[0], acc[1], acc[2], acc[3]);
    *reinterpret_cast<float4 *>(dx + (size_t)t * d + c + 4) = make_float4(acc[4], acc[5], acc[6], acc[7]);
  }
}

// The router term dz W_g^T as a weight-gradient GEMM over the experts: rows e,
// Np + e, 2 Np + e of A = dz^T [hi; lo; hi] ([3 Np, Tp] bf16, zero past N and T)
// and of B = W_g^T [hi; hi; lo] ([3 Np, d] bf16), so the sum over the rows gives
// dz_hi W_hi + dz_lo W_hi + dz_hi W_lo (the lo x lo term is below 2^-16 relative).
__global__ void split_dzT_kernel(const float *__restrict__ dz, int T, int N, int Np, int Tp,
                                 uint16_t *__restrict__ out) {
  const size_t n = (size_t)Np * Tp;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / Tp), t = (int)(i % Tp);
    const float v = (e < N && t < T) ? dz[(size_t)t * N + e] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    out[(size_t)e * Tp + t] = __bfloat16_as_ushort(hi);
    out[(size_t)(Np + e) * Tp + t] = __bfloat16_as_ushort(lo);
    out[(size_t)(2 * Np + e) * Tp + t] = __bfloat16_as_ushort(hi);
  }
}

__global__ void split_wgT_kernel(const float *__restrict__ Wg, int d, int N, int Np, uint16_t *__restrict__ out) {
  const size_t n = (size_t)Np * d;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
    const int e = (int)(i / d), c = (int)(i % d);
    const float v = e < N ? Wg[(size_t)c * N + e] : 0.f;
    const __nv_bfloat16 hi = __float2bfloat16_rn(v);
    const __nv_bfloat16 lo = __float2bfloat16_rn(v - __bfloat162float(hi));
    out[(size_t)e * d + c] = __bfloat16_as_ushort(hi);
    out[(size_t)(Np + e) * d + c] = __bfloat16_as_ushort(hi);
    out[(size_t)(2 * Np + e) * d + c] = __bfloat16_as_ushort(lo);
  }
}

__global__ void set_offsets2_kernel(int32_t *offsets, int rows) {
  if (threadIdx.x == 0) {
    offsets[0] = 0;
    offsets[1] = rows;
  }
}

inline int grid_for(size_t n, int per_block) {
  size_t g = (n + per_block - 1) / per_block;
  return (int)(g > 65535 * 8 ? 65535 * 8 : (g < 1 ? 1 : g));
}

}  // namespace

int launch_set_offsets2(int32_t *offsets, int rows, cudaStream_t s) {
  set_offsets2_kernel<<<1, 32, 0, s>>>(offsets, rows);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_zero_f32(float *p, size_t n, cudaStream_t s) {
  if (n == 0) return MOE_OK;
  zero_f32_kernel<<<grid_for(n, 256 * 4), 256, 0, s>>>(p, n);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dy_dgate(const void *dout, const void *y_perm, const float *topk_w, const int32_t *dest_row,
                    const int32_t *src_token, const int32_t *rows_end, int64_t max_rows, int k, int d, void *dy,
                    float *dgate, cudaStream_t s) {
  if (max_rows <= 0) return MOE_OK;
  dy_dgate_kernel<<<grid_for((size_t)max_rows, 8), 256, 0, s>>>(
      static_cast<const uint16_t *>(dout), static_cast<const uint16_t *>(y_perm), topk_w, dest_row, src_token, rows_end,
      k, d, static_cast<uint16_t *>(dy), dgate);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_router_bwd(const float *logits, const int32_t *idx, const float *topk_w, const float *dgate, int gate, int T,
                      int N, int k, float *dz, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  router_bwd_kernel<<<(T + 7) / 8, 256, 0, s>>>(logits, idx, topk_w, dgate, gate, T, N, k, dz);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_split_dz(const float *dz, int T, int N, int Np, void *out, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  split_dz_kernel<<<grid_for((size_t)T * Np, 256), 256, 0, s>>>(dz, T, N, Np, static_cast<uint16_t *>(out));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dwg_sum(const float *part, int d, int N, int Np, float *dWg, cudaStream_t s) {
  dwg_sum_kernel<<<grid_for((size_t)d * N, 256), 256, 0, s>>>(part, d, N, Np, dWg);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_split_router_term(const float *dz, const float *Wg, int T, int d, int N, int Np, int Tp, void *dzT,
                             void *wgT, cudaStream_t s) {
  split_dzT_kernel<<<grid_for((size_t)Np * Tp, 256), 256, 0, s>>>(dz, T, N, Np, Tp, static_cast<uint16_t *>(dzT));
  split_wgT_kernel<<<grid_for((size_t)Np * d, 256), 256, 0, s>>>(Wg, d, N, Np, static_cast<uint16_t *>(wgT));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_dx_combine(const void *dxp, const int32_t *dest_row, const float *rterm, const void *dx_sh, int T, int d,
                      int k, float *dx, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  dx_combine_kernel<<<T, 256, 0, s>>>(static_cast<const uint16_t *>(dxp), dest_row, rterm,
                                      static_cast<const uint16_t *>(dx_sh), T, d, k, dx);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
