// Grouped GEMM over ragged expert row groups on the CUDA cores, float32
// accumulation.  It serves the float32 workload (Shazeer-style ReLU experts,
// 512 -> 1024 -> 512, from the "Outrageously Large Neural Networks" notes),
// where tensor-core TF32 would not hold 1e-4 relative accuracy.
//
//   out[r, n] = EPI( sum_k A[r, k] * B_g[n, k] )     rows r of group g
// with the same modes and operand layouts as the tensor-core kernel
// (SwiGLU: B0 = W1, B1 = W3; ReLU; plain).  64 x 64 output tile per CTA,
// 4 x 4 per thread, K staged 16 at a time through shared memory.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SB_M = 64, SB_N = 64, SB_K = 16;

template <bool BF16>
__device__ __forceinline__ float ld_elem(const void *p, size_t i) {
  if (BF16) return __uint_as_float((uint32_t) static_cast<const uint16_t *>(p)[i] << 16);
  return static_cast<const float *>(p)[i];
}

template <bool BF16>
__device__ __forceinline__ void st_elem(void *p, size_t i, float v) {
  if (BF16) {
    __nv_bfloat16 b = __float2bfloat16_rn(v);
    static_cast<uint16_t *>(p)[i] = *reinterpret_cast<uint16_t *>(&b);
  } else {
    static_cast<float *>(p)[i] = v;
  }
}

template <bool BF16, int MODE>
__global__ void __launch_bounds__(256) simt_gemm_kernel(const void *__restrict__ A, int K, const void *__restrict__ B0,
                                                        const void *__restrict__ B1, int b_rows,
                                                        const int32_t *__restrict__ offsets, int M, int a_rows,
                                                        int n_out, void *__restrict__ out) {
  const int g = blockIdx.z;
  const int rb = offsets ? offsets[g] : 0;
  const int re = offsets ? offsets[g + 1] : M;
  if (rb < 0 || re > a_rows) return;  // malformed group: nothing to do (the tensor-core path flags it)
  const int row0 = rb + blockIdx.y * SB_M;
  if (row0 >= re) return;
  const int n0 = blockIdx.x * SB_N;
  __shared__ float As[SB_K][SB_M + 4];
  __shared__ float Bs[SB_K][SB_N + 4];
  __shared__ float Cs[SB_K][SB_N + 4];  // W3 tile for SwiGLU
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;
  float acc[4][4] = {}, acc3[4][4] = {};
  const size_t bbase = (size_t)g * b_rows;
  for (int k0 = 0; k0 < K; k0 += SB_K) {
    for (int v = threadIdx.x; v < SB_M * SB_K; v += 256) {
      const int m = v / SB_K, kk = v % SB_K;
      const int r = row0 + m, kg = k0 + kk;
      As[kk][m] = (r < re && kg < K) ? ld_elem<BF16>(A, (size_t)r * K + kg) : 0.f;
      const int n = n0 + m;
      const bool bok = n < n_out && kg < K;
      Bs[kk][m] = bok ? ld_elem<BF16>(B0, (bbase + n) * K + kg) : 0.f;
      if (MODE == 0) Cs[kk][m] = bok ? ld_elem<BF16>(B1, (bbase + n) * K + kg) : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < SB_K; ++kk) {
      float a[4], b[4], c[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        a[i] = As[kk][ty * 4 + i];
        b[i] = Bs[kk][tx * 4 + i];
        if (MODE == 0) c[i] = Cs[kk][tx * 4 + i];
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
          if (MODE == 0) acc3[i][j] = fmaf(a[i], c[j], acc3[i][j]);
        }
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = row0 + ty * 4 + i;
    if (r >= re) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= n_out) continue;
      float v = acc[i][j];
      if (MODE == 0) v = v / (1.0f + expf(-v)) * acc3[i][j];
      if (MODE == 1) v = fmaxf(v, 0.f);
      st_elem<BF16>(out, (size_t)r * n_out + n, v);
    }
  }
}

}  // namespace

int simt_grouped_gemm(int mode, bool bf16, const void *A, int64_t a_rows, int K, const void *B0, const void *B1,
                      int b_rows_per_group, const int32_t *offsets, int G, int M, int n_out, void *out,
                      cudaStream_t stream) {
  if (a_rows <= 0) return MOE_OK;
  const int64_t mt = (a_rows + SB_M - 1) / SB_M;  // a group never exceeds a_rows rows
  if (mt > 65535 || G > 65535 || a_rows > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (n_out > b_rows_per_group) return MOE_ERR_INVALID_ARG;
  dim3 grid((n_out + SB_N - 1) / SB_N, (unsigned)mt, G), block(256);
#define MOE_SG(BF, MD) \
  simt_gemm_kernel<BF, MD><<<grid, block, 0, stream>>>(A, K, B0, B1, b_rows_per_group, offsets, M, (int)a_rows, \
                                                       n_out, out)
  if (bf16) {
    if (mode == 0) MOE_SG(true, 0); else if (mode == 1) MOE_SG(true, 1); else MOE_SG(true, 2);
  } else {
    if (mode == 0) MOE_SG(false, 0); else if (mode == 1) MOE_SG(false, 1); else MOE_SG(false, 2);
  }
#undef MOE_SG
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
