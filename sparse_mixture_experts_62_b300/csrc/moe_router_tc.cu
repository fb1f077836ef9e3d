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
// values is exact in float32; the hi term's 64-wide slices of K are summed by
// the tensor core one at a time and added in float32 registers (see the
// kernel), so the result carries float32 accumulation error only.  The three
// terms are laid out along K: B = [hi | mid | lo], each dp = d rounded up to 64
// columns wide.
//
// One CTA per (128-token tile, tile of up to 128 experts, K split); the K splits
// fill the GPU when T is small.  Each CTA writes its raw float32 partial sums;
// the top-k kernel adds the splits in a fixed order (deterministic) plus the
// logit bias.
#include <algorithm>
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace rtc {

constexpr int BM = 128, BK = 64;
constexpr int A_BYTES = BM * BK * 2;

struct Args {
  int T;
  int Npad;     // experts padded to 32, 64, 128 or 256
  int ntiles;   // N tiles of NT experts (Npad / NT)
  int nkb_d;    // 64-wide k-blocks of d
  int kb_per;   // k-blocks per split
  int dp;       // d padded to 64: the column offset between the hi, mid and lo terms
  int S;        // splits
  uint32_t idesc;   // M = 128, N = NT
  uint32_t idesc2;  // M = 128, N = 2 NT
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
// same way; over a K of several thousand that bias reaches 1e-4.  So the MMAs of
// one k-block of the hi term (K = 64, four MMAs) go into a fresh tensor-memory
// buffer, which the epilogue warps add into float32 registers (round to nearest)
// while the next k-blocks fill the other buffers.  The mid and lo terms are 2^-8
// and 2^-16 of the weights, so the same drift on their running sums is below
// 2^-24 of the logit over any K here (at most 4 x 112 MMAs): they accumulate in
// a running buffer (mid and lo side by side) for the CTA's whole K range,
// drained once at the end.
//
// A stage holds one 64-wide k-block of x (128 tokens) and the same k-block of all
// three weight terms for this CTA's NT experts, so x is read once per N tile.
// The mid and lo tiles sit back to back and form one 2 NT-row operand.  MMAs per
// stage: 4 with N = NT (hi, fresh buffer) + 4 with N = 2 NT (mid and lo side by
// side in the running buffer): each MMA re-reads the x tile from shared memory,
// so fewer, wider MMAs move fewer shared-memory bytes per k-block.
template <int NT>
struct RouterShape {
  static constexpr int CPT = NT >= 64 ? 64 : 32;             // accumulator columns per epilogue thread
  static constexpr int EW = 4 * (NT / CPT);                  // epilogue warps (4 lane quadrants)
  static constexpr int THREADS = 64 + 32 * EW;
  static constexpr int STAGES = NT == 32 ? 3 : (NT == 64 ? 4 : 3);
  static constexpr int B_BYTES = NT * BK * 2;                // one term's k-block
  static constexpr int STAGE_BYTES = A_BYTES + 3 * B_BYTES;
  // two CTAs per SM (by shared memory) for NT = 32, one otherwise
  static constexpr uint32_t TMEM_COLS = NT == 32 ? 256 : 512;
  static constexpr int NBUF = (int)TMEM_COLS / NT - 2;       // hi buffers; the last 2 NT columns hold mid, lo
  static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + 256;
};

// 32 consecutive 32-bit TMEM columns of this thread's lane, waited for.
MOE_DEV void tmem_ld32(uint32_t taddr, float *v) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
// 64 columns with one wait.
MOE_DEV void tmem_ld64(uint32_t taddr, float *v) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr), "r"(taddr + 32)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}
template <int CPT>
MOE_DEV void tmem_ld_cols(uint32_t taddr, float *v) {
  if (CPT == 64)
    tmem_ld64(taddr, v);
  else
    tmem_ld32(taddr, v);
}

template <int NT>
__global__ void __launch_bounds__(RouterShape<NT>::THREADS, 1)
    router_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, const Args a) {
  using Sh = RouterShape<NT>;
  constexpr int CPT = Sh::CPT, EW = Sh::EW, STAGES = Sh::STAGES, NBUF = Sh::NBUF;
  constexpr int B_BYTES = Sh::B_BYTES, STAGE_BYTES = Sh::STAGE_BYTES;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + NBUF;
  uint64_t *mlfull = tempty + NBUF;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mlfull + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // blockIdx.x = (m_tile * ntiles + n_tile) * S + split
  const int split = blockIdx.x % a.S;
  const int mn = blockIdx.x / a.S;
  const int n_tile = mn % a.ntiles, m_tile = mn / a.ntiles;
  const int kb0 = split * a.kb_per;
  const int kb1 = min(kb0 + a.kb_per, a.nkb_d);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], EW);
    }
    mbar_init(mlfull, 1);
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc(tmem_slot, Sh::TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t ml_col = (uint32_t)(NBUF * NT);

  if (warp == 0) {
    if (lane == 0) {
      int issued_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      const int n0 = n_tile * NT;
      for (int kb = kb0; kb < kb1; ++kb) {
        if (!mbar_wait(&empty[stage], phase ^ 1u, a.status)) break;
        uint8_t *sa = smem + stage * STAGE_BYTES;
        mbar_arrive_expect_tx(&full[stage], (uint32_t)STAGE_BYTES);
        tma_load_2d(sa, &tmA, &full[stage], kb * BK, m_tile * BM);
#pragma unroll
        for (int term = 0; term < 3; ++term)
          tma_load_2d(sa + A_BYTES + term * B_BYTES, &tmB, &full[stage], term * a.dp + kb * BK, n0);
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
      bool ok = true;
      for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
        const int b = it % NBUF;
        const uint32_t use = (uint32_t)(it / NBUF);
        if (!mbar_wait(&tempty[b], (use & 1u) ^ 1u, a.status) || !mbar_wait(&full[stage], phase, a.status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
        const uint64_t adesc = smem_desc_sw128(sa);
        const uint64_t bhi = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_bf16(tmem_base + (uint32_t)(b * NT), adesc + 2ull * kk, bhi + 2ull * kk, a.idesc, kk > 0 ? 1u : 0u);
        tc_commit(&tfull[b]);
        const uint64_t bml = smem_desc_sw128(sa + A_BYTES + B_BYTES);  // [mid; lo], 2 NT rows
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk)
          tc_mma_bf16(tmem_base + ml_col, adesc + 2ull * kk, bml + 2ull * kk, a.idesc2,
                      (it == 0 && kk == 0) ? 0u : 1u);
        tc_commit(&empty[stage]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok) tc_commit(mlfull);
    }
  } else {
    const int ew = warp - 2;
    const int quad = warp & 3;                  // TMEM lanes 32 quad .. 32 quad + 31
    const int col0 = (ew / 4) * CPT;            // this thread's columns of the N tile
    const int r = quad * 32 + lane;
    const int t = m_tile * BM + r;
    const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
    float acc[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) acc[i] = 0.f;
    bool ok = true;
    for (int kb = kb0, it = 0; kb < kb1; ++kb, ++it) {
      const int b = it % NBUF;
      const uint32_t use = (uint32_t)(it / NBUF);
      if (!mbar_wait(&tfull[b], use & 1u, a.status)) {
        ok = false;
        break;
      }
      tc_fence_after();
      float v[CPT];
      tmem_ld_cols<CPT>(tmem_base + (uint32_t)(b * NT + col0) + lane_off, v);
#pragma unroll
      for (int i = 0; i < CPT; ++i) acc[i] += v[i];
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[b]);
    }
    if (ok && kb1 > kb0 && mbar_wait(mlfull, 0u, a.status)) {
      tc_fence_after();
      float v[CPT];
      tmem_ld_cols<CPT>(tmem_base + ml_col + (uint32_t)col0 + lane_off, v);  // mid
#pragma unroll
      for (int i = 0; i < CPT; ++i) acc[i] += v[i];
      tmem_ld_cols<CPT>(tmem_base + ml_col + (uint32_t)(NT + col0) + lane_off, v);  // lo
      if (t < a.T) {
        float4 *prow = reinterpret_cast<float4 *>(a.partial + ((size_t)split * a.T + t) * a.Npad + n_tile * NT + col0);
#pragma unroll
        for (int q = 0; q < CPT / 4; ++q)
          prow[q] = make_float4(acc[4 * q] + v[4 * q], acc[4 * q + 1] + v[4 * q + 1], acc[4 * q + 2] + v[4 * q + 2],
                                acc[4 * q + 3] + v[4 * q + 3]);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, Sh::TMEM_COLS);
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

// N tile: every expert in one tile up to 128, two tiles of 128 for 256
static int n_tile_width(int Npad) { return Npad > 128 ? 128 : Npad; }
static int ctas_per_sm(int NT) { return NT == 32 ? 2 : 1; }

template <int NT>
static int launch_nt(const CUtensorMap &ma, const CUtensorMap &mb, const Args &a, int grid, int dev, cudaStream_t s) {
  using Sh = RouterShape<NT>;
  static std::mutex mu;
  static std::vector<int> done;
  {
    std::lock_guard<std::mutex> lk(mu);
    if ((int)done.size() <= dev) done.resize(dev + 1, 0);
    if (!done[dev]) {
      if (cudaFuncSetAttribute(router_gemm_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::SMEM) !=
          cudaSuccess)
        return MOE_ERR_CUDA;
      done[dev] = 1;
    }
  }
  router_gemm_kernel<NT><<<grid, Sh::THREADS, Sh::SMEM, s>>>(ma, mb, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace rtc

int router_tc_npad(int N) { return N <= 32 ? 32 : (N <= 64 ? 64 : (N <= 128 ? 128 : 256)); }
int router_tc_dpad(int d) { return (d + 63) / 64 * 64; }
// Largest split count the planner may choose (bounds the partial-sum scratch).
int router_tc_max_splits(int T, int d) {
  const int mtiles = std::max(1, (T + 127) / 128);
  const int nkb = router_tc_dpad(d) / 64;
  return std::max(1, std::min(std::min(nkb, 64), 512 / mtiles));
}

// Split count with the fewest k-blocks on the busiest CTA slot: waves of CTAs
// (CTAs per SM from shared memory) times k-blocks per CTA.
static int plan_splits(int T, int d, int Npad, int sms) {
  const int mtiles = std::max(1, (T + 127) / 128);
  const int NT = rtc::n_tile_width(Npad);
  const int ntiles = Npad / NT;
  const int nkb = router_tc_dpad(d) / 64;
  const long slots = (long)sms * rtc::ctas_per_sm(NT);
  const int smax = router_tc_max_splits(T, d);
  int best = 1;
  long best_cost = -1;
  for (int S = 1; S <= smax; ++S) {
    const int kb_per = (nkb + S - 1) / S;
    const int S_eff = (nkb + kb_per - 1) / kb_per;
    if (S_eff != S) continue;  // every split non-empty
    const long waves = ((long)mtiles * ntiles * S + slots - 1) / slots;
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
  const int NT = n_tile_width(Npad);
  const int nkb_d = dp / BK;
  const int kb_per = (nkb_d + S - 1) / S;
  CUtensorMap ma, mb;
  int rc;
  if ((rc = make_map(&ma, x, (uint64_t)T, (uint64_t)d, BM))) return rc;
  if ((rc = make_map(&mb, wsplit, (uint64_t)Npad, (uint64_t)(3 * dp), (uint32_t)NT))) return rc;
  Args a{T, Npad, Npad / NT, nkb_d, kb_per, dp, S, idesc_bf16_f32(BM, NT), idesc_bf16_f32(BM, 2 * NT), partial, status};
  const int grid = ((T + BM - 1) / BM) * (Npad / NT) * S;
  switch (NT) {
    case 32: rc = launch_nt<32>(ma, mb, a, grid, dev, s); break;
    case 64: rc = launch_nt<64>(ma, mb, a, grid, dev, s); break;
    default: rc = launch_nt<128>(ma, mb, a, grid, dev, s); break;
  }
  if (rc) return rc;
  *splits_out = S;
  return MOE_OK;
}

}  // namespace moe
