// Weight-gradient GEMM of the expert FFN backward on the tensor cores: for each
// expert g, a sum over the rows that expert processed,
//
//   out[g][m][n] = sum_{r in rows of g} A[r][m] * B[r][n]      (float32 out)
//
// with A [rows, M] and B [rows, Nn] the row-major activations as the forward and
// the dgrad GEMMs left them (bf16, rows a_stride / b_stride elements apart) and
// the rows of expert g = offsets[g] .. offsets[g+1].  This is the ragged-K
// counterpart of the forward's ragged-M grouped GEMM: dW2 = dy^T h,
// dW1 = da^T x, dW3 = du^T x ("Chapter 19: MoE", 19.6.2: gradients reach an
// expert only through the tokens it processed).
//
// Both operands are MN-major: TMA copies 64-row x 64-column boxes (128-byte
// swizzle), K running along the rows.  A group's K blocks start at its first row,
// so its last block may hold rows of the next group (or rows past the data): the
// MMA warp issues that block's K=16 MMAs only up to the group's last row and
// zeroes the rows of the last one that lie past the group (a 128-byte row of a
// swizzled box stays one row of shared memory).
//
// Same machinery as the forward kernel: one CTA per SM, warp 0 loads a 128x64 A
// and a 256x64 B tile per stage into a 4-stage ring, warp 1 issues tcgen05.mma
// M=128 N=256 K=16 into one of two TMEM accumulators, warps 2-5 drain the other
// and store float32 rows.  Empty groups store zeros.
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace wg {

constexpr int BM = 128, BN = 256, BK = 64, STAGES = 4, THREADS = 192;
constexpr int SLICE = BK * 64 * 2;  // one box: 64 K rows x 64 columns = 8 KB
constexpr int A_BYTES = BM * BK * 2, B_BYTES = BN * BK * 2, STAGE_BYTES = A_BYTES + B_BYTES;
constexpr uint32_t TMEM_COLS = 512;
constexpr int MAX_G = 257;
constexpr int TABLE_BYTES = ((2 * MAX_G + 8) * 4 + 15) / 16 * 16;  // keeps the staging area 16-byte aligned
constexpr int STG_PITCH = 36;                          // floats per staged row (32 + 4: no bank conflicts)
constexpr int STG_BYTES = 4 * 32 * STG_PITCH * 4;      // one 32 x 32 float block per epilogue warp
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + TABLE_BYTES + STG_BYTES;
constexpr uint32_t IDESC = idesc_bf16_f32_major(BM, BN, true, true);

struct Args {
  const int32_t *offsets;  // [G + 1] row offsets of the groups, or nullptr: one group of `rows` rows
  int32_t G;
  int32_t M;               // columns of A used = output rows per group
  int32_t Nn;              // columns of B used = output columns
  int32_t rows;            // rows of A and B
  float *out;              // [G][M][Nn]
  int *status;
};

// Epilogue of one warp: its 32 accumulator rows (TMEM lanes at taddr) x 256
// columns -> out rows row0 .. row0 + 31 of group g, columns n0 ..  Each 32 x 32
// block goes through the warp's staging area so that global stores cover whole
// 128-byte row segments (4 rows per instruction).
__device__ __forceinline__ void store_tile_rows(uint32_t taddr, float *stg, const Args &args, int g, int row0, int n0,
                                                bool empty_k, int lane) {
#pragma unroll 1
  for (int c = 0; c < BN; c += 32) {
    float v0[16], v1[16];
    tmem_ld16x2(taddr + c, taddr + c + 16, v0, v1);
    if (empty_k) {
#pragma unroll
      for (int i = 0; i < 16; ++i) v0[i] = v1[i] = 0.f;
    }
    float4 *mine = reinterpret_cast<float4 *>(stg + lane * STG_PITCH);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      mine[q] = make_float4(v0[4 * q], v0[4 * q + 1], v0[4 * q + 2], v0[4 * q + 3]);
      mine[4 + q] = make_float4(v1[4 * q], v1[4 * q + 1], v1[4 * q + 2], v1[4 * q + 3]);
    }
    __syncwarp();
    const int cc = (lane & 7) * 4;
    const int col = n0 + c + cc;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int rr = i * 4 + (lane >> 3);
      const int row = row0 + rr;
      const float4 v = *reinterpret_cast<const float4 *>(stg + rr * STG_PITCH + cc);
      if (row < args.M && col + 4 <= args.Nn)
        *reinterpret_cast<float4 *>(args.out + ((size_t)g * args.M + row) * args.Nn + col) = v;
    }
    __syncwarp();
  }
}

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
  int *rowbeg = reinterpret_cast<int *>(smem + STAGES * STAGE_BYTES + 256);  // [G]
  int *rowend = rowbeg + MAX_G;                                               // [G]
  float *staging = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES + 256 + TABLE_BYTES);

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
    for (int g = 0; g < args.G; ++g) {
      int b = args.offsets ? args.offsets[g] : 0;
      int e = args.offsets ? args.offsets[g + 1] : args.rows;
      if (b < 0 || e < b || e > args.rows) {  // malformed: flag it, treat the group as empty
        set_status(args.status, MOE_ERR_BOUNDS);
        b = e = 0;
      }
      rowbeg[g] = b;
      rowend[g] = e;
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
        for (int k0 = rowbeg[g]; k0 < rowend[g]; k0 += BK) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + stage * STAGE_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
#pragma unroll
          for (int j = 0; j < BM / 64; ++j) tma_load_2d(sa + j * SLICE, &tmA, &full[stage], m_tile * BM + 64 * j, k0);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)
            tma_load_2d(sa + A_BYTES + j * SLICE, &tmB, &full[stage], n_tile * BN + 64 * j, k0);
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
    // the whole warp follows the pipeline (it zeroes tail rows); lane 0 issues the MMAs
    int stage = 0;
    uint32_t phase = 0;
    int it = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
      const int g = tile / per_group;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!__all_sync(0xffffffffu, mbar_wait(&tempty[acc], (use & 1u) ^ 1u, args.status))) break;
      tc_fence_after();
      const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
      const int kbeg = rowbeg[g], kend = rowend[g];
      for (int k0 = kbeg; k0 < kend; k0 += BK) {
        if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, args.status))) {
          ok = false;
          break;
        }
        uint8_t *st = smem + stage * STAGE_BYTES;
        // a group's last block: MMAs of K=16 up to its last row; the rows of the
        // last MMA past the group belong to no row of this group: zero them
        const int valid = kend - k0;
        const int nk = valid >= BK ? BK / 16 : (valid + 15) / 16;
        if (valid < nk * 16) {
          const int nrow = nk * 16 - valid;
          for (int v = lane; v < (STAGE_BYTES / SLICE) * nrow * 8; v += 32) {
            const int box = v / (nrow * 8), rr = (v / 8) % nrow, ch = v % 8;
            *reinterpret_cast<uint4 *>(st + box * SLICE + (valid + rr) * 128 + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
          }
          asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        }
        __syncwarp();
        if (lane == 0) {
          tc_fence_after();
          const uint32_t sa = smem_u32(st);
          const uint64_t adesc = smem_desc_sw128_mn(sa, SLICE);
          const uint64_t bdesc = smem_desc_sw128_mn(sa + A_BYTES, SLICE);
          for (int kk = 0; kk < nk; ++kk)  // +16 K rows = +2048 bytes in both tiles
            tc_mma_bf16(d_tmem, adesc + 128ull * kk, bdesc + 128ull * kk, IDESC, (k0 > kbeg || kk > 0) ? 1u : 0u);
          tc_commit(&empty[stage]);
        }
        __syncwarp();
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (ok && lane == 0) tc_commit(&tfull[acc]);  // with no MMA issued (empty group) it arrives at once
      __syncwarp();
    }
  } else {
    const int quad = warp & 3;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      const int g = tile / per_group, rem = tile % per_group;
      const int n_tile = rem / m_tiles, m_tile = rem % m_tiles;
      const bool empty_k = rowend[g] == rowbeg[g];
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
      store_tile_rows(taddr, staging + quad * 32 * STG_PITCH, args, g, m_tile * BM + quad * 32, n_tile * BN, empty_k,
                      lane);
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

// ---------------------------------------------------------------- CTA-pair form
// The same sums on pairs of SMs (clusters of two) with tcgen05.mma.cta_group::2:
// a pair computes a 256 x 256 output tile, each CTA staging 128 columns of A and
// 128 of B per K block (32 KB, 6 stages), which halves the shared-memory traffic
// per MMA of the single-CTA form.  Both CTAs' copies complete on the leader's
// full[s] and the leader issues the MMAs.  In a group's last block the leader's
// warp zeroes the rows past the group (up to the last K=16 step) in its own tiles
// and, through distributed shared memory, in the peer's, then fences them for the
// tensor core: no round trip between the CTAs.
//   empty[s], tfull[a]  in each CTA: the leader's multicast commits.
//   tempty[a]           in the leader: the 8 epilogue warps of the pair.
namespace pr {
constexpr int STAGES = 6;
constexpr int HALF = 128;                         // columns of A and of B per CTA
constexpr int A_BYTES = HALF * BK * 2;            // 16 KB
constexpr int STAGE_BYTES = 2 * A_BYTES;          // 32 KB
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + TABLE_BYTES + STG_BYTES;
constexpr uint32_t IDESC = idesc_bf16_f32_major(2 * HALF, 2 * HALF, true, true);
}  // namespace pr

// Zero rows valid .. end-1 of every 64-row box of a staged K block (a 128-byte
// row of a swizzled box stays one row), in this CTA and, through its cluster
// address, in the peer's copy at the same offset; then order the writes before
// the tensor core's reads of both.
__device__ __forceinline__ void zero_tail_rows_pair(uint8_t *st, int nbox, int valid, int end, int lane) {
  const int nrow = end - valid;
  const uint32_t local = smem_u32(st);
  const uint32_t remote = mapa_shared(local, 1);
  for (int v = lane; v < nbox * nrow * 8; v += 32) {
    const int box = v / (nrow * 8), rr = (v / 8) % nrow, ch = v % 8;
    const uint32_t off = (uint32_t)(box * SLICE + (valid + rr) * 128 + ch * 16);
    *reinterpret_cast<uint4 *>(st + off) = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(remote + off), "r"(0u) : "memory");
  }
  asm volatile("fence.proxy.async.shared::cluster;" ::: "memory");
}

__global__ void __launch_bounds__(THREADS, 1)
    wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                      const Args args) {
  constexpr int STAGES = pr::STAGES, STAGE_BYTES = pr::STAGE_BYTES, A_BYTES = pr::A_BYTES, HALF = pr::HALF;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  int *rowbeg = reinterpret_cast<int *>(smem + STAGES * STAGE_BYTES + 256);
  int *rowend = rowbeg + MAX_G;
  float *staging = reinterpret_cast<float *>(smem + STAGES * STAGE_BYTES + 256 + TABLE_BYTES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int pair_id = blockIdx.x >> 1, npairs = gridDim.x >> 1;
  const int m_tiles = (args.M + 2 * HALF - 1) / (2 * HALF), n_tiles = (args.Nn + 2 * HALF - 1) / (2 * HALF);
  const int per_group = m_tiles * n_tiles;
  const int total_tiles = args.G * per_group;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    fence_barrier_init();
    for (int g = 0; g < args.G; ++g) {
      int b = args.offsets ? args.offsets[g] : 0;
      int e = args.offsets ? args.offsets[g + 1] : args.rows;
      if (b < 0 || e < b || e > args.rows) {
        set_status(args.status, MOE_ERR_BOUNDS);
        b = e = 0;
      }
      rowbeg[g] = b;
      rowend[g] = e;
    }
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const uint32_t full_lead = mapa_shared(smem_u32(&full[0]), 0);
  const uint32_t tempty_lead = mapa_shared(smem_u32(&tempty[0]), 0);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int issued_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int tile = pair_id; tile < total_tiles && ok; tile += npairs) {
        const int g = tile / per_group, rem = tile % per_group;
        const int n_tile = rem / m_tiles, m_tile = rem % m_tiles;
        const int m0 = m_tile * 2 * HALF + (int)rank * HALF, n0 = n_tile * 2 * HALF + (int)rank * HALF;
        for (int k0 = rowbeg[g]; k0 < rowend[g]; k0 += BK) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + stage * STAGE_BYTES;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2u * STAGE_BYTES);
          const uint32_t fb = full_lead + 8u * stage;
          tma_load_2d_pair(sa, &tmA, fb, m0, k0);
          tma_load_2d_pair(sa + SLICE, &tmA, fb, m0 + 64, k0);
          tma_load_2d_pair(sa + A_BYTES, &tmB, fb, n0, k0);
          tma_load_2d_pair(sa + A_BYTES + SLICE, &tmB, fb, n0 + 64, k0);
          issued_parity[stage] = (int)phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // the leader's full barriers count both CTAs' copies: wait for the last ones
      if (leader)
        for (int s = 0; s < STAGES; ++s)
          if (issued_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_parity[s], args.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issue and tail zeroing (leader)
    if (leader) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      for (int tile = pair_id; tile < total_tiles && ok; tile += npairs, ++it) {
        const int g = tile / per_group;
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!__all_sync(0xffffffffu, mbar_wait_cluster(&tempty[acc], (use & 1u) ^ 1u, args.status))) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * 2 * HALF);
        const int kbeg = rowbeg[g], kend = rowend[g];
        for (int k0 = kbeg; k0 < kend; k0 += BK) {
          if (!__all_sync(0xffffffffu, mbar_wait(&full[stage], phase, args.status))) {
            ok = false;
            break;
          }
          uint8_t *st = smem + stage * STAGE_BYTES;
          // a group's last block: MMAs of K=16 up to its last row, the rows of
          // the last MMA past the group zeroed
          const int valid = kend - k0;
          const int nk = valid >= BK ? BK / 16 : (valid + 15) / 16;
          if (valid < nk * 16) zero_tail_rows_pair(st, STAGE_BYTES / SLICE, valid, nk * 16, lane);
          __syncwarp();
          if (lane == 0) {
            tc_fence_after();
            const uint32_t sa = smem_u32(st);
            const uint64_t adesc = smem_desc_sw128_mn(sa, SLICE);
            const uint64_t bdesc = smem_desc_sw128_mn(sa + A_BYTES, SLICE);
            for (int kk = 0; kk < nk; ++kk)
              tc_mma_bf16_pair(d_tmem, adesc + 128ull * kk, bdesc + 128ull * kk, pr::IDESC,
                               (k0 > kbeg || kk > 0) ? 1u : 0u);
            tc_commit_pair(&empty[stage], 0x3);
          }
          __syncwarp();
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok && lane == 0) tc_commit_pair(&tfull[acc], 0x3);
        __syncwarp();
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    int it = 0;
    for (int tile = pair_id; tile < total_tiles; tile += npairs, ++it) {
      const int g = tile / per_group, rem = tile % per_group;
      const int n_tile = rem / m_tiles, m_tile = rem % m_tiles;
      const bool empty_k = rowend[g] == rowbeg[g];
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * 2 * HALF) + ((uint32_t)(quad * 32) << 16);
      store_tile_rows(taddr, staging + quad * 32 * STG_PITCH, args, g, m_tile * 2 * HALF + (int)rank * HALF + quad * 32,
                      n_tile * 2 * HALF, empty_k, lane);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty_lead + 8u * acc);
    }
  }
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal its barriers
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// [rows, cols] bf16, rows `stride` elements apart; box 64 (cols) x 64 (rows),
// 128-byte swizzle; reads past the matrix are zero.
static int make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint64_t stride) {
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
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (stride * 2) % 16 || rows == 0 || cols == 0 || stride < cols)
    return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride * 2};
  cuuint32_t box[2] = {64, BK};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// CTA pairs that can run at once (cluster occupancy), per device.
static int pair_grid(int device) {
  static std::mutex mu;
  static std::vector<int> cache;
  std::lock_guard<std::mutex> lk(mu);
  if ((int)cache.size() <= device) cache.resize(device + 1, 0);
  if (!cache[device]) {
    if (cudaFuncSetAttribute(wgrad_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)pr::SMEM_BYTES) !=
        cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * device_sm_count(device));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = pr::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, wgrad_pair_kernel, &cfg) != cudaSuccess || clusters < 1) return -1;
    cache[device] = 2 * clusters;
  }
  return cache[device];
}

}  // namespace wg

int tc_wgrad_gemm(const void *A, int64_t a_stride, const void *B, int64_t b_stride, int64_t rows,
                  const int32_t *offsets, int G, int M, int Nn, float *out, int *status, cudaStream_t stream) {
  using namespace wg;
  if (G < 1 || G > MAX_G - 1 || M < 1 || Nn < 1 || rows < 1 || rows > INT32_MAX || (Nn % 4) || !A || !B || !out)
    return MOE_ERR_INVALID_ARG;
  CUtensorMap ma, mb;
  int rc;
  if ((rc = make_map(&ma, A, (uint64_t)rows, (uint64_t)M, (uint64_t)a_stride))) return rc;
  if ((rc = make_map(&mb, B, (uint64_t)rows, (uint64_t)Nn, (uint64_t)b_stride))) return rc;
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
  Args a{offsets, G, M, Nn, (int32_t)rows, out, status};
  if (M >= 2 * pr::HALF) {  // 256-row output tiles on CTA pairs
    const int grid = pair_grid(dev);
    if (grid < 2) return MOE_ERR_CUDA;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = pr::SMEM_BYTES;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, wgrad_pair_kernel, ma, mb, a) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  wgrad_kernel<<<sms, THREADS, SMEM_BYTES, stream>>>(ma, mb, a);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
