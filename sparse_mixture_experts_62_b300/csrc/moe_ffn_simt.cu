// Grouped GEMM over ragged expert row groups on the CUDA cores, float32
// throughout.  It serves the float32 workload (Shazeer-style ReLU experts,
// 512 -> 1024 -> 512, from the "Outrageously Large Neural Networks" notes),
// where tensor-core TF32 would not hold 1e-4 relative accuracy.
//
//   out[r, n] = EPI( sum_k A[r, k] * B_g[n, k] )     rows r of group g
// with the same modes and operand layouts as the tensor-core kernel
// (SwiGLU: B0 = W1, B1 = W3; ReLU; plain).  32 x 64 output tile per CTA (small
// tiles: the expert groups of this workload hold ~64 rows), 4 x 4 per thread, K
// staged 32 at a time through shared memory with the next slice prefetched into
// registers while the current one is multiplied.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int SB_M = 32, SB_N = 64, SB_K = 32, SB_T = 128;

template <int MODE>
__global__ void __launch_bounds__(SB_T) simt_gemm_kernel(const float *__restrict__ A, int K, const float *__restrict__ B0,
                                                         const float *__restrict__ B1, int b_rows,
                                                         const int32_t *__restrict__ offsets, int M, int a_rows,
                                                         int n_out, float *__restrict__ out) {
  constexpr bool TWO = MODE == 0;  // SwiGLU: a second weight matrix
  const int g = blockIdx.z;
  const int rb = offsets ? offsets[g] : 0;
  const int re = offsets ? offsets[g + 1] : M;
  if (rb < 0 || re > a_rows) return;  // malformed group: nothing to do
  const int row0 = rb + blockIdx.y * SB_M;
  if (row0 >= re) return;
  const int n0 = blockIdx.x * SB_N;
  __shared__ __align__(16) float As[SB_K][SB_M + 4];
  __shared__ __align__(16) float Bs[SB_K][SB_N + 4];
  __shared__ __align__(16) float Cs[TWO ? SB_K : 1][SB_N + 4];
  const int tx = threadIdx.x % 16, ty = threadIdx.x / 16;  // 16 x 8 threads, 4 x 4 outputs each
  const size_t bbase = (size_t)g * b_rows;
  // loader mapping: 8 float4 per row of a tile; A has 32 rows (two float4 per
  // thread), B and C 64 rows (four per thread)
  constexpr int AQ = SB_M * (SB_K / 4) / SB_T, BQ = SB_N * (SB_K / 4) / SB_T;
  float4 ra[AQ], rb4[BQ], rc[TWO ? BQ : 1];
  auto load = [&](int k0) {
    const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int q = 0; q < AQ; ++q) {
      const int v = threadIdx.x + q * SB_T, m = v / (SB_K / 4), kg = k0 + (v % (SB_K / 4)) * 4;
      const int r = row0 + m;
      ra[q] = (r < re && kg < K) ? *reinterpret_cast<const float4 *>(A + (size_t)r * K + kg) : z;
    }
#pragma unroll
    for (int q = 0; q < BQ; ++q) {
      const int v = threadIdx.x + q * SB_T, m = v / (SB_K / 4), kg = k0 + (v % (SB_K / 4)) * 4;
      const int n = n0 + m;
      const bool bok = n < n_out && kg < K;
      rb4[q] = bok ? *reinterpret_cast<const float4 *>(B0 + (bbase + n) * K + kg) : z;
      if (TWO) rc[q] = bok ? *reinterpret_cast<const float4 *>(B1 + (bbase + n) * K + kg) : z;
    }
  };
  auto stash = [&]() {
#pragma unroll
    for (int q = 0; q < AQ; ++q) {
      const int v = threadIdx.x + q * SB_T, m = v / (SB_K / 4), kk = (v % (SB_K / 4)) * 4;
      As[kk][m] = ra[q].x; As[kk + 1][m] = ra[q].y; As[kk + 2][m] = ra[q].z; As[kk + 3][m] = ra[q].w;
    }
#pragma unroll
    for (int q = 0; q < BQ; ++q) {
      const int v = threadIdx.x + q * SB_T, m = v / (SB_K / 4), kk = (v % (SB_K / 4)) * 4;
      Bs[kk][m] = rb4[q].x; Bs[kk + 1][m] = rb4[q].y; Bs[kk + 2][m] = rb4[q].z; Bs[kk + 3][m] = rb4[q].w;
      if (TWO) {
        Cs[kk][m] = rc[q].x; Cs[kk + 1][m] = rc[q].y; Cs[kk + 2][m] = rc[q].z; Cs[kk + 3][m] = rc[q].w;
      }
    }
  };
  float acc[4][4] = {}, acc3[4][4] = {};
  load(0);
  for (int k0 = 0; k0 < K; k0 += SB_K) {
    __syncthreads();
    stash();
    __syncthreads();
    if (k0 + SB_K < K) load(k0 + SB_K);  // in flight while this slice is multiplied
#pragma unroll
    for (int kk = 0; kk < SB_K; ++kk) {
      const float4 a = *reinterpret_cast<const float4 *>(&As[kk][ty * 4]);
      const float4 b = *reinterpret_cast<const float4 *>(&Bs[kk][tx * 4]);
      const float av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
      float cv[4];
      if (TWO) {
        const float4 c = *reinterpret_cast<const float4 *>(&Cs[kk][tx * 4]);
        cv[0] = c.x; cv[1] = c.y; cv[2] = c.z; cv[3] = c.w;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
          if (TWO) acc3[i][j] = fmaf(av[i], cv[j], acc3[i][j]);
        }
    }
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
      out[(size_t)r * n_out + n] = v;
    }
  }
}

}  // namespace

int simt_grouped_gemm(int mode, const void *A, int64_t a_rows, int K, const void *B0, const void *B1,
                      int b_rows_per_group, const int32_t *offsets, int G, int M, int n_out, void *out,
                      cudaStream_t stream) {
  if (a_rows <= 0) return MOE_OK;
  const int64_t mt = (a_rows + SB_M - 1) / SB_M;  // a group never exceeds a_rows rows
  if (mt > 65535 || G > 65535 || a_rows > INT32_MAX) return MOE_ERR_UNSUPPORTED;
  if (n_out > b_rows_per_group || K % 4) return MOE_ERR_INVALID_ARG;
  dim3 grid((n_out + SB_N - 1) / SB_N, (unsigned)mt, G), block(SB_T);
  const float *a = static_cast<const float *>(A), *b0 = static_cast<const float *>(B0);
  const float *b1 = static_cast<const float *>(B1);
  float *o = static_cast<float *>(out);
  if (mode == 0)
    simt_gemm_kernel<0><<<grid, block, 0, stream>>>(a, K, b0, b1, b_rows_per_group, offsets, M, (int)a_rows, n_out, o);
  else if (mode == 1)
    simt_gemm_kernel<1><<<grid, block, 0, stream>>>(a, K, b0, b1, b_rows_per_group, offsets, M, (int)a_rows, n_out, o);
  else
    simt_gemm_kernel<2><<<grid, block, 0, stream>>>(a, K, b0, b1, b_rows_per_group, offsets, M, (int)a_rows, n_out, o);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
