// Combine: weight each kept expert output by its gate and restore token order.
//
// "Lecture29" (CS25 lecture 29 notes), section "Top-two routing":
// y = sum_i g_i(x) Expert_i(x); section "Top-k routing semantics": results are
// inverse-permuted back to the tokens.  CS336 lecture 4, section 6: the shared
// expert's output is added for every token; section 10: a dropped assignment
// adds nothing.
//
// out[t] = y_shared[t] + sum_{j=0..k-1, dest_row[t,j] >= 0} w[t,j] * y_perm[dest_row[t,j]]
// in float32, slot order fixed, no atomics; 8 elements per thread per step.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

template <bool BF16>
__device__ __forceinline__ void load8(const void *base, size_t off, float *v) {
  if (BF16) {
    const uint4 q = *reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(base) + off);
    v[0] = bf16_lo(q.x); v[1] = bf16_hi(q.x); v[2] = bf16_lo(q.y); v[3] = bf16_hi(q.y);
    v[4] = bf16_lo(q.z); v[5] = bf16_hi(q.z); v[6] = bf16_lo(q.w); v[7] = bf16_hi(q.w);
  } else {
    const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off);
    const float4 b = *reinterpret_cast<const float4 *>(static_cast<const float *>(base) + off + 4);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// One CTA per token; d % 8 == 0 for bf16 (8-wide steps), d % 4 == 0 for float32 (4-wide).
template <bool BF16>
__global__ void __launch_bounds__(128) combine_kernel(const void *__restrict__ y_perm,
                                                      const int32_t *__restrict__ dest_row,
                                                      const float *__restrict__ w, const void *__restrict__ y_shared,
                                                      void *__restrict__ out, int T, int d, int k) {
  const int t = blockIdx.x;
  __shared__ int rows[256];
  __shared__ float gates[256];
  __shared__ int nslots;
  // the token's kept slots, in slot order (k <= 8 for token choice, N <= 256 for expert choice)
  if (threadIdx.x == 0) {
    int n = 0;
    for (int j = 0; j < k; ++j) {
      const int r = dest_row[(size_t)t * k + j];
      if (r >= 0) {
        rows[n] = r;
        gates[n] = w[(size_t)t * k + j];
        ++n;
      }
    }
    nslots = n;
  }
  __syncthreads();
  const int ns = nslots;
  const int step = BF16 ? 8 : 4;
  for (int c = threadIdx.x * step; c < d; c += blockDim.x * step) {
    if (BF16) {
      float acc[8];
      if (y_shared)
        load8<true>(y_shared, (size_t)t * d + c, acc);
      else
        for (int i = 0; i < 8; ++i) acc[i] = 0.f;
      for (int j = 0; j < ns; ++j) {
        const int r = rows[j];
        float v[8];
        load8<true>(y_perm, (size_t)r * d + c, v);
        const float g = gates[j];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = fmaf(g, v[i], acc[i]);
      }
      uint4 o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                           pack_bf16x2(acc[6], acc[7]));
      *reinterpret_cast<uint4 *>(static_cast<uint16_t *>(out) + (size_t)t * d + c) = o;
    } else {
      float4 acc = y_shared ? *reinterpret_cast<const float4 *>(static_cast<const float *>(y_shared) + (size_t)t * d + c)
                            : make_float4(0.f, 0.f, 0.f, 0.f);
      for (int j = 0; j < ns; ++j) {
        const int r = rows[j];
        const float4 v = *reinterpret_cast<const float4 *>(static_cast<const float *>(y_perm) + (size_t)r * d + c);
        const float g = gates[j];
        acc.x = fmaf(g, v.x, acc.x);
        acc.y = fmaf(g, v.y, acc.y);
        acc.z = fmaf(g, v.z, acc.z);
        acc.w = fmaf(g, v.w, acc.w);
      }
      *reinterpret_cast<float4 *>(static_cast<float *>(out) + (size_t)t * d + c) = acc;
    }
  }
}

}  // namespace

int launch_combine(bool bf16, const void *y_perm, const int32_t *dest_row, const float *w, const void *y_shared,
                   void *out, int T, int d, int k, cudaStream_t s) {
  if (T == 0) return MOE_OK;
  if (bf16)
    combine_kernel<true><<<T, 128, 0, s>>>(y_perm, dest_row, w, y_shared, out, T, d, k);
  else
    combine_kernel<false><<<T, 128, 0, s>>>(y_perm, dest_row, w, y_shared, out, T, d, k);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
