// Weight-gradient GEMM of the expert FFN backward on the tensor cores: for each
// expert g, a sum over the rows that expert processed,
//
//   out[g][m][n] = sum_{r in rows of g} A[r][m] * B[r][n]      (float32 out)
//
// with A and B given transposed (AT [M, Kp], BT [Nn, Kp], both bf16, K = rows
// contiguous) and each expert's rows padded to a multiple of 64 with zeros, so
// expert g owns columns koff[g] .. koff[g+1] of AT and BT.  This is the ragged-K
// counterpart of the forward's ragged-M grouped GEMM: dW2 = dy^T h,
// dW1 = da^T x, dW3 = du^T x ("Chapter 19: MoE", 19.6.2: gradients reach an
// expert only through the tokens it processed).
//
// Same machinery as the forward kernel: one CTA per SM, warp 0 loads 128x64 A
// and 256x64 B tiles by TMA (128-byte swizzle) into a 4-stage ring, warp 1 issues
// tcgen05.mma M=128 N=256 K=16 into one of two TMEM accumulators, warps 2-5
// drain the other and store float32 rows.  Empty K ranges store zeros.
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace wg {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4, THREADS = 192;
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_G = 257;
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + (size_t)(MAX_G + 8) * 4;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

struct Args {
  const int32_t *koff;  // [G + 1] column offsets of each group in AT / BT (multiples of 64)
  int32_t G;
  int32_t M;            // rows of AT = output rows per group
  int32_t Nn;           // rows of BT = output columns
  int64_t kp;           // columns of AT and BT
  float *out;           // [G][M][Nn]
  int *status;
};

__global__ void __launch_bounds__(THREADS, 1)
    wgrad_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  int *kb_of = reinterpret_cast<int *>(smem + STAGES * STAGE_BYTES + 256);  // [G + 1] k-block offsets

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tiles = (args.M + BM - 1) / BM, n_tiles = (args.Nn + BN - 1) / BN;
  const int per_group = m_tiles * n_tiles;
  const int total_tiles = args.G * per_group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    fence_barrier_init();
    int prev = 0;
    for (int g = 0; g <= args.G; ++g) {
      int k = args.koff[g];
      if (k < prev || (k & (BK - 1)) || k > args.kp) {  // malformed: treat the group as empty
        set_status(args.status, MOE_ERR_BOUNDS);
        k = prev;
      }
      kb_of[g] = k / BK;
      prev = k;
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      int issued_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        const int g = tile / per_group, rem = tile % per_group;
        const int n_tile = rem / m_tiles, m_tile = rem % m_tiles;
        for (int kb = kb_of[g]; kb < kb_of[g + 1]; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
          tma_load_2d(sa, &tmA, &full[stage], kb * BK, m_tile * BM);
          tma_load_2d(sa + A_BYTES, &tmB, &full[stage], kb * BK, n_tile * BN);
          tma_load_2d(sa + A_BYTES + B_BYTES / 2, &tmB, &full[stage], kb * BK, n_tile * BN + BN / 2);
          issued_parity[stage] = (int)phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_parity[s], args.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
        const int g = tile / per_group;
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        const int kb0 = kb_of[g];
        for (int kb = kb0; kb < kb_of[g + 1]; ++kb) {
          if (!mbar_wait(&full[stage], phase, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = smem_desc_sw128(sa);
          const uint64_t bdesc = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, IDESC, (kb > kb0 || kk > 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(&tfull[acc]);  // with no MMA issued (empty group) it arrives at once
      }
    }
  } else {
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      const int g = tile / per_group, rem = tile % per_group;
      const int n_tile = rem / m_tiles, m_tile = rem % m_tiles;
      const bool empty_k = kb_of[g + 1] == kb_of[g];
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
      const int row = m_tile * BM + r;
      const bool row_ok = row < args.M;
      float *orow = args.out + ((size_t)g * args.M + (row_ok ? row : 0)) * args.Nn;
      const int n0 = n_tile * BN;
#pragma unroll 1
      for (int c = 0; c < BN; c += 32) {
        float v0[16], v1[16];
        tmem_ld16x2(taddr + c, taddr + c + 16, v0, v1);
        if (empty_k) {
#pragma unroll
          for (int i = 0; i < 16; ++i) v0[i] = v1[i] = 0.f;
        }
        if (row_ok) {
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const int col = n0 + c + 4 * q;
            const float *src = q < 4 ? v0 + 4 * q : v1 + 4 * (q - 4);
            if (col + 4 <= args.Nn) *reinterpret_cast<float4 *>(orow + col) = make_float4(src[0], src[1], src[2], src[3]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static int make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  if (!fn) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16 || rows == 0 || cols == 0) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, 128};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace wg

int tc_wgrad_gemm(const void *AT, const void *BT, const int32_t *koff, int G, int M, int Nn, int64_t kp, float *out,
                  int *status, cudaStream_t stream) {
  using namespace wg;
  if (G < 1 || G > MAX_G - 1 || M < 1 || Nn < 1 || kp < BK || (kp % BK) || (Nn % 4)) return MOE_ERR_INVALID_ARG;
  CUtensorMap ma, mb;
  int rc;
  if ((rc = make_map(&ma, AT, (uint64_t)M, (uint64_t)kp))) return rc;
  if ((rc = make_map(&mb, BT, (uint64_t)Nn, (uint64_t)kp))) return rc;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  {
    static std::mutex mu;
    static std::vector<int> done;
    std::lock_guard<std::mutex> lk(mu);
    if ((int)done.size() <= dev) done.resize(dev + 1, 0);
    if (!done[dev]) {
      if (cudaFuncSetAttribute(wgrad_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM_BYTES) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
      done[dev] = 1;
    }
  }
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  Args a{koff, G, M, Nn, kp, out, status};
  wgrad_kernel<<<sms, THREADS, SMEM_BYTES, stream>>>(ma, mb, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
