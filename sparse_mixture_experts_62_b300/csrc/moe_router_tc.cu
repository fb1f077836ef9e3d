// Router logits on the tensor cores for bf16 activations: z = x . W_g with
// float32 accuracy (the CS336 lecture 4 notes, section 11, keep the router in
// float32; "Lecture29", section "Top-two routing": z = W_r x).
//
// x is bf16, so it is exact as a tensor-core operand; the float32 router weight
// is split into three bf16 terms, W_g = hi + mid + lo (each the bf16 rounding of
// what the previous terms left; the remainder is below 2^-24 relative), and
//   z = x.hi + x.mid + x.lo
// is computed on the tensor cores -- the bf16x3 method of Henry, Tang &
// Heinecke, "Leveraging the bfloat16 artificial intelligence datatype for
// higher-precision computations" (ARITH 2019).  Every product of two bf16
// values is exact in float32; each 64-wide slice of K is summed by the tensor
// core and the slices are added in float32 registers (see the kernel), so the
// result carries float32 accumulation error only.  The three terms are laid out
// along K: B = [hi | mid | lo], and the A tile of x for k-block kb is x's k-block
// kb mod (d/64).
//
// One CTA per (128-token tile, K split); the K splits fill the GPU when T is
// small.  Each CTA writes its raw float32 partial sums; the top-k kernel adds
// the splits in a fixed order (deterministic) plus the logit bias.
#include <algorithm>
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace rtc {

constexpr int BM = 128, BK = 64, STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;

struct Args {
  int T;
  int Npad;     // experts padded to 32, 64, 128 or 256 (MMA N)
  int nkb_d;    // k-blocks per copy of d
  int kb_per;   // k-blocks per split
  int nkb;      // 3 * nkb_d
  int S;        // splits
  uint32_t idesc;
  float *partial;  // [S][T][Npad]
  int *status;
};

// W_g [d, N] float32 -> B [Npad, 3*dp] bf16: B[e, s*dp + j] = term s of W_g[j, e];
// zero for e >= N or j >= d.  32x32 tiles transposed through shared memory.
__global__ void __launch_bounds__(256) split_wg_kernel(const float *__restrict__ Wg, int d, int N, int dp, int Npad,
                                                       uint16_t *__restrict__ B) {
  __shared__ float tile[32][33];
  const int j0 = blockIdx.x * 32, e0 = blockIdx.y * 32;
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
  for (int r = ty; r < 32; r += 8) {
    const int j = j0 + r, e = e0 + tx;
    tile[r][tx] = (j < d && e < N) ? Wg[(size_t)j * N + e] : 0.f;
  }
  __syncthreads();
  for (int r = ty; r < 32; r += 8) {
    const int e = e0 + r, j = j0 + tx;
    if (e >= Npad || j >= dp) continue;
    const float w = tile[tx][r];
    const __nv_bfloat16 hi = __float2bfloat16_rn(w);
    const float r1 = w - __bfloat162float(hi);
    const __nv_bfloat16 mid = __float2bfloat16_rn(r1);
    const float r2 = r1 - __bfloat162float(mid);
    const __nv_bfloat16 lo = __float2bfloat16_rn(r2);
    uint16_t *row = B + (size_t)e * 3 * dp;
    row[j] = *reinterpret_cast<const uint16_t *>(&hi);
    row[dp + j] = *reinterpret_cast<const uint16_t *>(&mid);
    row[2 * dp + j] = *reinterpret_cast<const uint16_t *>(&lo);
  }
}

// The tensor core adds each MMA's products into its float32 accumulator with a
// rounding that drifts by about one unit in the last place per MMA, always the
// same way; over a K of several thousand that bias reaches 1e-4.  So the MMAs
// of one k-block (K = 64, four MMAs) go into a fresh tensor-memory buffer and
// the epilogue warps add that buffer into float32 registers (round to nearest)
// while the MMAs of the next k-blocks fill the other buffers (up to eight in
// rotation, so the MMAs are not held up by each buffer's round trip).
template <int NP>
__global__ void __launch_bounds__(64 + 32 * (NP > 128 ? 8 : 4), 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args a) {
  constexpr int EW = NP > 128 ? 8 : 4;          // epilogue warps
  constexpr int COLS = NP / (EW / 4);           // accumulator columns per epilogue thread
  constexpr int B_BYTES = NP * BK * 2;
  constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
  // tensor-memory buffers in rotation, sized so that the CTAs that fit on one SM
  // by shared memory (two for NP <= 64, one above) share its 512 columns
  constexpr int NBUF = NP == 32 ? 8 : (NP == 64 ? 4 : (NP == 128 ? 4 : 2));
  constexpr uint32_t TMEM_COLS = NBUF * NP;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + NBUF;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + NBUF);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int m_tile = blockIdx.x / a.S, split = blockIdx.x % a.S;
  const int kb0 = split * a.kb_per;
  const int kb1 = min(kb0 + a.kb_per, a.nkb);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EW);
    }
    fence_barrier_init();
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
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, a.status)) break;
        uint8_t *sa = smem + stage * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)STAGE_BYTES);
        tma_load_2d(sa, &tmA, &full[stage], (kb % a.nkb_d) * BK, m_tile * BM);
        tma_load_2d(sa + A_BYTES, &tmB, &full[stage], kb * BK, 0);
        issued_parity[stage] = (int)phase;
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_parity[s], a.status);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
        const int b = it % NBUF;
        const uint32_t use = (uint32_t)(it / NBUF);
        if (!mbar_wait(&tempty[b], (use & 1u) ^ 1u, a.status)) break;
        if (!mbar_wait(&full[stage], phase, a.status)) break;
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
        const uint64_t adesc = smem_desc_sw128(sa);
        const uint64_t bdesc = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_bf16(tmem_base + (uint32_t)(b * NP), adesc + 2ull * kk, bdesc + 2ull * kk, a.idesc, kk > 0 ? 1u : 0u);
        tc_commit(&empty[stage]);
        tc_commit(&tfull[b]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
  } else {
    const int ew = warp - 2;
    const int quad = warp & 3;
    const int col0 = (ew / 4) * COLS;
    const int r = quad * 32 + lane;
    const int t = m_tile * BM + r;
    float acc[COLS];
#pragma unroll
    for (int i = 0; i < COLS; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int b = it % NBUF;
      const uint32_t use = (uint32_t)(it / NBUF);
      if (!mbar_wait(&tfull[b], use & 1u, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(b * NP + col0) + ((uint32_t)(quad * 32) << 16);
#pragma unroll
      for (int c = 0; c < COLS; c += 32) {
        float v0[16], v1[16];
        tmem_ld16x2(taddr + c, taddr + c + 16, v0, v1);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          acc[c + i] += v0[i];
          acc[c + 16 + i] += v1[i];
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
    if (ok && t < a.T) {
      float4 *prow = reinterpret_cast<float4 *>(a.partial + ((size_t)split * a.T + t) * NP + col0);
#pragma unroll
      for (int q = 0; q < COLS / 4; ++q) prow[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
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

static EncodeTiledFn get_encode() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

static int make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

static size_t smem_bytes(int Npad) { return 1024 + (size_t)STAGES * (A_BYTES + Npad * BK * 2) + 256; }
static int threads_for(int Npad) { return 64 + 32 * (Npad > 128 ? 8 : 4); }

template <int NP>
static int launch_np(const CUtensorMap &ma, const CUtensorMap &mb, const Args &a, int grid, int dev, cudaStream_t s) {
  static std::mutex mu;
  static std::vector<int> done;
  {
    std::lock_guard<std::mutex> lk(mu);
    if ((int)done.size() <= dev) done.resize(dev + 1, 0);
    if (!done[dev]) {
      if (cudaFuncSetAttribute(router_gemm_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem_bytes(NP)) != cudaSuccess)
        return MOE_ERR_CUDA;
      done[dev] = 1;
    }
  }
  router_gemm_kernel<NP><<<grid, threads_for(NP), smem_bytes(NP), s>>>(ma, mb, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace rtc

int router_tc_npad(int N) { return N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256)); }
int router_tc_dpad(int d) { return (d + 63) / 64 * 64; }
// Largest split count the planner may choose (bounds the partial-sum scratch).
int router_tc_max_splits(int T, int d) {
  const int mtiles = std::max(1, (T + 127) / 128);
  const int nkb = 3 * (router_tc_dpad(d) / 64);
  return std::max(1, std::min(std::min(nkb, 64), 512 / mtiles));
}

static int plan_splits(int T, int d, int Npad, int sms) {
  const int mtiles = std::max(1, (T + 127) / 128);
  const int nkb = 3 * (router_tc_dpad(d) / 64);
  const size_t smem = rtc::smem_bytes(Npad);
  const int per_sm = std::max(1, std::min(4, (int)((size_t)(227 * 1024) / smem)));
  const long slots = (long)sms * per_sm;
  const int smax = router_tc_max_splits(T, d);
  int best = 1;
  long best_cost = -1;
  for (int S = 1; S <= smax; ++S) {
    const int kb_per = (nkb + S - 1) / S;
    const int S_eff = (nkb + kb_per - 1) / kb_per;
    if (S_eff != S) continue;  // every split non-empty
    const long waves = ((long)mtiles * S + slots - 1) / slots;
    const long cost = waves * kb_per;
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = S;
    }
  }
  return best;
}

int launch_router_tc(const void *x, const float *Wg, int T, int d, int N, uint16_t *wsplit, float *partial,
                     int *splits_out, int *status, cudaStream_t s) {
  using namespace rtc;
  const int Npad = router_tc_npad(N), dp = router_tc_dpad(d);
  if (Npad > 256) return MOE_ERR_UNSUPPORTED;
  dim3 sg((dp + 31) / 32, (Npad + 31) / 32);
  split_wg_kernel<<<sg, 256, 0, s>>>(Wg, d, N, dp, Npad, wsplit);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  const int S = plan_splits(T, d, Npad, sms);
  const int nkb_d = dp / BK, nkb = 3 * nkb_d;
  const int kb_per = (nkb + S - 1) / S;
  CUtensorMap ma, mb;
  int rc;
  if ((rc = make_map(&ma, x, (uint64_t)T, (uint64_t)d, BM))) return rc;
  if ((rc = make_map(&mb, wsplit, (uint64_t)Npad, (uint64_t)(3 * dp), (uint32_t)Npad))) return rc;
  Args a{T, Npad, nkb_d, kb_per, nkb, S, idesc_bf16_f32(BM, Npad), partial, status};
  const int grid = ((T + BM - 1) / BM) * S;
  switch (Npad) {
    case 32: rc = launch_np<32>(ma, mb, a, grid, dev, s); break;
    case 64: rc = launch_np<64>(ma, mb, a, grid, dev, s); break;
    case 128: rc = launch_np<128>(ma, mb, a, grid, dev, s); break;
    default: rc = launch_np<256>(ma, mb, a, grid, dev, s); break;
  }
  if (rc) return rc;
  *splits_out = S;
  return MOE_OK;
}

}  // namespace moe
