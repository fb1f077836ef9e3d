// Combine: weight each kept expert output by its gate and restore token order.
//
// "Lecture29" (CS25 lecture 29 notes), section "Top-two routing":
// y = sum_i g_i(x) Expert_i(x); section "Top-k routing semantics": results are
// inverse-permuted back to the tokens.  CS336 lecture 4, section 6: the shared
// expert's output is added for every token; section 10: a dropped assignment
// adds nothing.
//
// out[t] = y_shared[t] + sum_{j=0..k-1, dest_row[t,j] >= 0} w[t,j] * y_perm[dest_row[t,j]]
// in float32, slot order fixed, no atomics.
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

// One warp per token (grid-stride), for token choice (k <= 8 slots).  Lane j < k
// reads slot j's row and gate; the kept slots are compacted in slot order with a
// ballot and broadcast.  Each lane then takes 16-byte chunks of the row
// (8 bf16 or 4 float) and, per chunk, issues the loads of every kept slot before
// the fused multiply-adds, which run in slot order.  KS (2, 4 or 8) bounds the
// slots; each lane keeps 16 / KS chunks in flight per pass (16 loads).
template <bool BF16, int KS>
__global__ void __launch_bounds__(256) combine_warp_kernel(const void *__restrict__ y_perm,
                                                           const int32_t *__restrict__ dest_row,
                                                           const float *__restrict__ w,
                                                           const void *__restrict__ y_shared, void *__restrict__ out,
                                                           int T, int d, int k) {
  constexpr int EPC = BF16 ? 8 : 4;  // elements per 16-byte chunk
  const int lane = threadIdx.x & 31;
  const int nchunk = d / EPC;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps_total) {
    int r = -1;
    float g = 0.f;
    if (lane < k) {
      r = dest_row[(size_t)t * k + lane];
      g = w[(size_t)t * k + lane];
    }
    const uint32_t kept = __ballot_sync(0xffffffffu, r >= 0);
    const int ns = __popc(kept);
    int rows[KS];
    float gates[KS];
    uint32_t m = kept;
#pragma unroll
    for (int j = 0; j < KS; ++j) {
      const int src = m ? __ffs(m) - 1 : 0;
      rows[j] = __shfl_sync(0xffffffffu, r, src);
      gates[j] = __shfl_sync(0xffffffffu, g, src);
      m &= m - 1;
    }
    constexpr int U = 16 / KS;  // chunks per lane per pass, their loads in flight together
    for (int c0 = lane; c0 < nchunk; c0 += 32 * U) {
      uint4 q[U][KS];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
#pragma unroll
        for (int j = 0; j < KS; ++j)
          if (j < ns && c < nchunk)
            q[u][j] = __ldg(reinterpret_cast<const uint4 *>(y_perm) + (size_t)rows[j] * nchunk + c);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + 32 * u;
        if (c >= nchunk) break;
        float acc[EPC];
        if (y_shared) {
          const uint4 sq = __ldg(reinterpret_cast<const uint4 *>(y_shared) + (size_t)t * nchunk + c);
          if (BF16) {
            acc[0] = bf16_lo(sq.x); acc[1] = bf16_hi(sq.x); acc[2] = bf16_lo(sq.y); acc[3] = bf16_hi(sq.y);
            acc[4] = bf16_lo(sq.z); acc[5] = bf16_hi(sq.z); acc[6] = bf16_lo(sq.w); acc[7] = bf16_hi(sq.w);
          } else {
            acc[0] = __uint_as_float(sq.x); acc[1] = __uint_as_float(sq.y);
            acc[2] = __uint_as_float(sq.z); acc[3] = __uint_as_float(sq.w);
          }
        } else {
#pragma unroll
          for (int i = 0; i < EPC; ++i) acc[i] = 0.f;
        }
#pragma unroll
        for (int j = 0; j < KS; ++j) {
          if (j >= ns) break;
          const uint4 v = q[u][j];
          const float gj = gates[j];
          if (BF16) {
            acc[0] = fmaf(gj, bf16_lo(v.x), acc[0]); acc[1] = fmaf(gj, bf16_hi(v.x), acc[1]);
            acc[2] = fmaf(gj, bf16_lo(v.y), acc[2]); acc[3] = fmaf(gj, bf16_hi(v.y), acc[3]);
            acc[4] = fmaf(gj, bf16_lo(v.z), acc[4]); acc[5] = fmaf(gj, bf16_hi(v.z), acc[5]);
            acc[6] = fmaf(gj, bf16_lo(v.w), acc[6]); acc[7] = fmaf(gj, bf16_hi(v.w), acc[7]);
          } else {
            acc[0] = fmaf(gj, __uint_as_float(v.x), acc[0]); acc[1] = fmaf(gj, __uint_as_float(v.y), acc[1]);
            acc[2] = fmaf(gj, __uint_as_float(v.z), acc[2]); acc[3] = fmaf(gj, __uint_as_float(v.w), acc[3]);
          }
        }
        uint4 o;
        if (BF16)
          o = make_uint4(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]), pack_bf16x2(acc[4], acc[5]),
                         pack_bf16x2(acc[6], acc[7]));
        else
          o = make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                         __float_as_uint(acc[3]));
        reinterpret_cast<uint4 *>(out)[(size_t)t * nchunk + c] = o;
      }
    }
  }
}

// Expert choice (up to 256 slots per token): one CTA per token; d % 8 == 0 for
// bf16 (8-wide steps), d % 4 == 0 for float32 (4-wide).
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
  if (k <= 8) {  // token choice
    int dev = 0;
    cudaGetDevice(&dev);
    const int sms = device_sm_count(dev);
    int64_t blocks = ((int64_t)T + 7) / 8;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 4;
    if (blocks > cap) blocks = cap;
#define MOE_CMB(B, KS) combine_warp_kernel<B, KS><<<(int)blocks, 256, 0, s>>>(y_perm, dest_row, w, y_shared, out, T, d, k)
    if (bf16) {
      if (k <= 2) MOE_CMB(true, 2); else if (k <= 4) MOE_CMB(true, 4); else MOE_CMB(true, 8);
    } else {
      if (k <= 2) MOE_CMB(false, 2); else if (k <= 4) MOE_CMB(false, 4); else MOE_CMB(false, 8);
    }
#undef MOE_CMB
  } else if (bf16) {
    combine_kernel<true><<<T, 128, 0, s>>>(y_perm, dest_row, w, y_shared, out, T, d, k);
  } else {
    combine_kernel<false><<<T, 128, 0, s>>>(y_perm, dest_row, w, y_shared, out, T, d, k);
  }
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
