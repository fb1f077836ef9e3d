// Grouped GEMM over ragged per-expert row groups on the 5th-generation tensor
// cores (tcgen05, accumulators in tensor memory), operands staged by TMA.
//
// This is the expert FFN of the layer: "Lecture29" (CS25 lecture 29 notes),
// section "A dense Transformer layer" (expert = W2(SiLU(W1 x) * W3 x)) and the
// Shazeer et al. notes (expert = one ReLU hidden layer); grouped over experts
// the way the CS336 lecture 4 notes, section 10, describe the block-sparse
// matmul: every expert's rows form one contiguous group, no padding per expert.
//
//   out[r, n] = EPI( sum_k A[r, k] * B_g[n, k] )        for rows r of group g
//
// A: [rows, K] bf16 row-major (x_perm or h), one TMA map over all groups (or the
//    rows of x gathered by index, see below).
// B_g: rows [g * b_rows, (g + 1) * b_rows) of a [G * b_rows, K] bf16 view of the
//      stacked expert weights (K-major, i.e. the "W x" layout).
// Modes:
//   kSwiGLU: two weight maps (W1, W3); a 128x256 accumulator holds W1 rows
//            n0..n0+127 in columns 0..127 and W3 rows in 128..255; the epilogue
//            writes SiLU(a) * u as bf16, 128 output columns per tile.
//   kReLU:   one map; 256 output columns per tile; epilogue max(acc, 0) -> bf16.
//   kPlain:  one map; 256 output columns per tile; epilogue acc -> bf16.
//   kPlainBT: B_g stored the other way round, [K, n_out] per group (the stacked
//            weights read in place as [G][K][n_out] through a 3-D map, MN-major
//            tiles); epilogue as kPlain.  dh = dy W2 in the backward.
//   kDualBT: two (A, B) pairs concatenated along K, both B's as in kPlainBT:
//            out = A1 B1 + A2 B2.  dx rows = da W1 + du W3 in the backward.
//   kSwiGLUBwd: the kSwiGLU tile (a = x W1^T, u = x W3^T recomputed), epilogue
//            the activation's backward with dh read from memory:
//            da = dh u SiLU'(a) into columns n, du = dh SiLU(a) into n_out + n.
//   kReLUBwd: the kReLU tile (a = x W1^T), epilogue da = dh [a > 0].
//
// Kernel shape (one CTA per SM, persistent over output tiles):
//   warp 0      TMA producer (one lane): 4-stage ring of {A 128x64, B 256x64}.
//   warp 1      TMEM owner + MMA issuer (one lane): 4 x tcgen05.mma
//               M=128,N=256,K=16 per stage into one of two TMEM accumulators.
//   warps 2..5  epilogue: tcgen05.ld of its 32-lane quadrant, activation,
//               16-byte stores masked to the group's rows and the output width.
// Tiles are enumerated group by group, n-tile-major within a group, so the
// CTAs of one wave share each weight tile through L2.  Single CTAs take tiles
// round robin; CTA pairs take them in issue order from a counter (see the tile
// queue below), so the pairs that share a weight tile run it together.
//
// Small groups (forward modes, single-CTA form): a group of at most 128 rows
// pays a whole 128-row MMA per tile however few its rows.  Its tiles run with the
// operands swapped instead: the two 128-row halves of the stage's weight tile are
// each the MMA's M side and the group's rows, padded to a multiple of 16, its N
// side (D1, D2 = 128 weight rows x N_t in tensor memory), so the MMA work shrinks
// to N_t / 128 of a tile while the same bytes stream through the same ring.  The
// epilogue thread of weight row f writes output column f of every row of the
// group (32 consecutive columns per warp store).
//
// Gathered A (forward modes, `tc_grouped_gemm_gather`): instead of x_perm, the A
// tile's rows are rows src_token[r] of x, fetched by TMA row gathers
// (`tile::gather4` on a one-row-high map over x: four indexed 128-byte rows per
// copy, 32 copies per 128-row stage, one per producer lane) into the same
// 128-byte-swizzled layout; the rest of the kernel is unchanged.
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace tc {

constexpr int BM = 128;              // rows per tile (TMEM lanes)
constexpr int BN = 256;              // accumulator columns per tile
constexpr int BK = 64;               // K per stage: 64 bf16 = one 128-byte swizzle row
constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;            // 16 KB
constexpr int B_BYTES = BN * BK * 2;            // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // 48 KB
constexpr uint32_t STAGE_TX = STAGE_BYTES;
constexpr int MAX_GROUPS = 257;
constexpr int THREADS = 192;
constexpr uint32_t TMEM_COLS = 512;  // two 256-column accumulators
constexpr size_t SMEM_BYTES = 1024 /*alignment slack*/ + (size_t)STAGES * STAGE_BYTES + 256 /*barriers*/ +
                              (size_t)(4 * MAX_GROUPS + 8) * 4;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

enum Mode { kSwiGLU = 0, kReLU = 1, kPlain = 2, kPlainBT = 3, kDualBT = 4, kSwiGLUBwd = 5, kReLUBwd = 6 };
// groups of at most this many rows run swapped tiles (forward modes, single-CTA form)
constexpr int SWAP_ROWS = 128;
__host__ __device__ constexpr bool swappable(int mode) { return mode == kSwiGLU || mode == kReLU || mode == kPlain; }
// modes whose tile pairs W1 and W3 rows (128 output columns per tile)
__host__ __device__ constexpr bool paired_b(int mode) { return mode == kSwiGLU || mode == kSwiGLUBwd; }
constexpr uint32_t IDESC_BT = idesc_bf16_f32_major(BM, BN, false, true);
constexpr int B_SLICE = BK * 64 * 2;  // one MN-major B slice: 64 K rows x 64 columns = 8 KB

struct Args {
  const int32_t *offsets;  // [G + 1] group row offsets in A / out, or nullptr: one group of M rows
  int32_t G;
  int32_t M;
  int32_t a_rows;      // rows of A and out; a group reaching past them is rejected
  int32_t n_out;       // output columns of every group
  int32_t K;           // reduction length
  int32_t b_rows;      // weight-view rows per group
  uint16_t *out;       // [rows, n_out] bf16
  int *status;
  int32_t num_kb;      // K blocks per tile
  int32_t kb1;         // kDualBT: K blocks taken from the first (A, B) pair
  int32_t out_stride;  // elements between output rows
  const uint16_t *dh;  // kSwiGLUBwd / kReLUBwd: [rows, n_out] bf16 gradient of h
  // Gathered A (forward modes): row r of A is row src[r] of gx [gx_rows, K] instead
  // of row r of the A tensor map; null: A through its tensor map.
  const uint16_t *gx;
  const int32_t *gsrc;
  int32_t gx_rows;
  // CTA-pair form: tiles are taken from this counter in issue order (zeroed before
  // each launch)
  int *tile_counter;
};

__device__ __forceinline__ float silu(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// Epilogue of one accumulator row (this thread's TMEM lane at taddr): output row
// `row`, columns n0 .. of the tile; nothing is stored when !row_ok.
template <int MODE>
__device__ __forceinline__ void epilogue_row(uint32_t taddr, const Args &args, int row, bool row_ok, int n0) {
  uint16_t *orow = args.out + (size_t)(row_ok ? row : 0) * args.out_stride;
  if (MODE == kSwiGLU) {
#pragma unroll 1
    for (int c = 0; c < 128; c += 16) {
      float a[16], u[16];
      tmem_ld16x2(taddr + c, taddr + 128 + c, a, u);
      uint32_t p[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) p[i] = pack_bf16x2(silu(a[2 * i]) * u[2 * i], silu(a[2 * i + 1]) * u[2 * i + 1]);
      const int col = n0 + c;
      if (row_ok) {
        if (col + 8 <= args.n_out) *reinterpret_cast<uint4 *>(orow + col) = make_uint4(p[0], p[1], p[2], p[3]);
        if (col + 16 <= args.n_out) *reinterpret_cast<uint4 *>(orow + col + 8) = make_uint4(p[4], p[5], p[6], p[7]);
      }
    }
  } else if (MODE == kSwiGLUBwd) {
    const uint16_t *grow = args.dh + (size_t)(row_ok ? row : 0) * args.n_out;
#pragma unroll 1
    for (int c = 0; c < 128; c += 16) {
      float a[16], u[16];
      tmem_ld16x2(taddr + c, taddr + 128 + c, a, u);
      const int col = n0 + c;
      if (!row_ok) continue;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        if (col + 8 * h + 8 > args.n_out) break;
        const uint4 gq = *reinterpret_cast<const uint4 *>(grow + col + 8 * h);
        const uint32_t gv[4] = {gq.x, gq.y, gq.z, gq.w};
        uint32_t pa[4], pu[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          float da[2], du[2];
#pragma unroll
          for (int j = 0; j < 2; ++j) {
            const float av = a[8 * h + 2 * i + j], uv = u[8 * h + 2 * i + j];
            const float g = j ? bf16_hi(gv[i]) : bf16_lo(gv[i]);
            const float sg = 1.0f / (1.0f + __expf(-av));
            da[j] = g * uv * sg * (1.0f + av * (1.0f - sg));
            du[j] = g * av * sg;
          }
          pa[i] = pack_bf16x2(da[0], da[1]);
          pu[i] = pack_bf16x2(du[0], du[1]);
        }
        *reinterpret_cast<uint4 *>(orow + col + 8 * h) = make_uint4(pa[0], pa[1], pa[2], pa[3]);
        *reinterpret_cast<uint4 *>(orow + args.n_out + col + 8 * h) = make_uint4(pu[0], pu[1], pu[2], pu[3]);
      }
    }
  } else {
    const uint16_t *grow = (MODE == kReLUBwd) ? args.dh + (size_t)(row_ok ? row : 0) * args.n_out : nullptr;
#pragma unroll 1
    for (int c = 0; c < 256; c += 32) {
      float v0[16], v1[16];
      tmem_ld16x2(taddr + c, taddr + c + 16, v0, v1);
      if (!row_ok) continue;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int col = n0 + c + 8 * q;
        if (col + 8 > args.n_out) continue;
        const float *v = q < 2 ? v0 + 8 * q : v1 + 8 * (q - 2);
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = (MODE == kReLU) ? fmaxf(v[i], 0.f) : v[i];
        if (MODE == kReLUBwd) {
          const uint4 gq = *reinterpret_cast<const uint4 *>(grow + col);
          const uint32_t gv[4] = {gq.x, gq.y, gq.z, gq.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            x[2 * i] = v[2 * i] > 0.f ? bf16_lo(gv[i]) : 0.f;
            x[2 * i + 1] = v[2 * i + 1] > 0.f ? bf16_hi(gv[i]) : 0.f;
          }
        }
        *reinterpret_cast<uint4 *>(orow + col) =
            make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]), pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
      }
    }
  }
}

// Epilogue of a swapped tile: this thread's TMEM lane is weight row f of the
// tile (f = quad * 32 + lane); D1 in columns [0, nt), D2 in [nt, 2 nt), one
// column per row of the group.  SwiGLU: out[row0 + j, n0 + f] = SiLU(D1) * D2;
// ReLU / plain: out[row0 + j, n0 + f] = act(D1), out[row0 + j, n0 + 128 + f] = act(D2).
template <int MODE>
__device__ __forceinline__ void epilogue_swapped(uint32_t taddr, const Args &args, int row0, int rows, int nt,
                                                 int n0, int f) {
  const int c1 = n0 + f, c2 = n0 + 128 + f;
  const bool ok1 = c1 < args.n_out;
  const bool ok2 = MODE != kSwiGLU && c2 < args.n_out;
#pragma unroll 1
  for (int c = 0; c < nt; c += 16) {
    float a[16], u[16];
    tmem_ld16x2(taddr + c, taddr + nt + c, a, u);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int j = c + i;
      if (j >= rows) break;
      uint16_t *orow = args.out + (size_t)(row0 + j) * args.out_stride;
      if (MODE == kSwiGLU) {
        if (ok1) orow[c1] = (uint16_t)(pack_bf16x2(silu(a[i]) * u[i], 0.f) & 0xFFFFu);
      } else {
        const float v1 = MODE == kReLU ? fmaxf(a[i], 0.f) : a[i];
        const float v2 = MODE == kReLU ? fmaxf(u[i], 0.f) : u[i];
        if (ok1) orow[c1] = (uint16_t)(pack_bf16x2(v1, 0.f) & 0xFFFFu);
        if (ok2) orow[c2] = (uint16_t)(pack_bf16x2(v2, 0.f) & 0xFFFFu);
      }
    }
  }
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                        const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                        const Args args) {
  constexpr int OUT_COLS = paired_b(MODE) ? 128 : 256;  // output columns per tile
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled operand tiles
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  int *tile_start = reinterpret_cast<int *>(smem + STAGES * STAGE_BYTES + 256);  // [G + 1]
  int *mtiles = tile_start + MAX_GROUPS + 1;                                     // [G]
  int *rowbeg = mtiles + MAX_GROUPS;                                             // [G]
  int *rowend = rowbeg + MAX_GROUPS;                                             // [G]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = args.G;
  const int n_tiles = (args.n_out + OUT_COLS - 1) / OUT_COLS;
  const int num_kb = args.num_kb;

  // gathered A: the A tensor map is a one-row-high map over x, read by TMA row
  // gathers (see the producer below)
  const bool gather = swappable(MODE) && args.gx != nullptr;
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
    int acc = 0;
    for (int g = 0; g < G; ++g) {
      int b = args.offsets ? args.offsets[g] : 0;
      int e = args.offsets ? args.offsets[g + 1] : args.M;
      if (b < 0 || e < b || e > args.a_rows) {  // malformed group: flag it, run nothing
        set_status(args.status, MOE_ERR_BOUNDS);
        b = e = 0;
      }
      rowbeg[g] = b;
      rowend[g] = e;
      const int mt = e > b ? (e - b + BM - 1) / BM : 0;
      mtiles[g] = mt;
      tile_start[g] = acc;
      acc += mt * n_tiles;
    }
    tile_start[G] = acc;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (paired_b(MODE) || MODE == kDualBT) tma_prefetch_desc(&tmB1);
    if (MODE == kDualBT) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[G];

  if (warp == 0 && gather) {
    // ------------------------------------------------------------ producer, gathered A
    // Lane 0 waits for the stage, sets its expected bytes (A and B, as for tiled
    // loads) and loads the B tile; then each of the 32 lanes loads rows 4 * lane ..
    // 4 * lane + 3 of the A tile with one TMA row gather: x's rows src[r] for the
    // tile's rows r, 64 columns each, into the 128-byte-swizzled tile.  Rows past
    // the group's end (not stored) and indices past x (flagged) read row 0 of x.
    int issued_parity[STAGES];
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    int stage = 0;
    uint32_t phase = 0;
    int g = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      while (tile >= tile_start[g + 1]) ++g;
      const int local = tile - tile_start[g];
      const int n_tile = local / mtiles[g];
      const int m_tile = local - n_tile * mtiles[g];
      const int a_row = rowbeg[g] + m_tile * BM;
      const int b_row = g * args.b_rows + n_tile * OUT_COLS;
      int t[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = a_row + 4 * lane + j;
        t[j] = 0;
        if (r < rowend[g]) {
          const int v = args.gsrc[r];
          if (v < 0 || v >= args.gx_rows)
            set_status(args.status, MOE_ERR_BOUNDS);
          else
            t[j] = v;
        }
      }
      for (int kb = 0; kb < num_kb; ++kb) {
        uint8_t *sa = smem + stage * STAGE_BYTES;
        uint8_t *sb = sa + A_BYTES;
        bool go = true;
        if (lane == 0) {
          go = mbar_wait(&empty[stage], phase ^ 1u, args.status);
          if (go) {
            mbar_arrive_expect_tx(&full[stage], STAGE_TX);
            tma_load_2d(sb, &tmB0, &full[stage], kb * BK, b_row);
            if (paired_b(MODE))
              tma_load_2d(sb + B_BYTES / 2, &tmB1, &full[stage], kb * BK, b_row);
            else
              tma_load_2d(sb + B_BYTES / 2, &tmB0, &full[stage], kb * BK, b_row + BN / 2);
            issued_parity[stage] = (int)phase;
          }
        }
        if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        tma_gather4(sa + lane * 512, &tmA, &full[stage], kb * BK, t[0], t[1], t[2], t[3]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // never leave the CTA with a bulk copy still writing its shared memory
    if (lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_parity[s], args.status);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
        while (tile >= tile_start[g + 1]) ++g;
        const int local = tile - tile_start[g];
        const int n_tile = local / mtiles[g];
        const int m_tile = local - n_tile * mtiles[g];
        const int a_row = rowbeg[g] + m_tile * BM;
        const int b_row = g * args.b_rows + n_tile * OUT_COLS;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + stage * STAGE_BYTES;
          uint8_t *sb = sa + A_BYTES;
          mbar_arrive_expect_tx(&full[stage], STAGE_TX);
          if (MODE == kPlainBT || MODE == kDualBT) {
            const bool second = MODE == kDualBT && kb >= args.kb1;
            const int k0 = (second ? kb - args.kb1 : kb) * BK;
            const CUtensorMap *mb = second ? &tmB1 : &tmB0;
            tma_load_2d(sa, second ? &tmA2 : &tmA, &full[stage], k0, a_row);
#pragma unroll
            for (int j = 0; j < BN / 64; ++j)
              tma_load_3d(sb + j * B_SLICE, mb, &full[stage], n_tile * OUT_COLS + 64 * j, k0, g);
          } else if (paired_b(MODE)) {
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, a_row);
            tma_load_2d(sb, &tmB0, &full[stage], kb * BK, b_row);
            tma_load_2d(sb + B_BYTES / 2, &tmB1, &full[stage], kb * BK, b_row);
          } else {
            tma_load_2d(sa, &tmA, &full[stage], kb * BK, a_row);
            tma_load_2d(sb, &tmB0, &full[stage], kb * BK, b_row);
            tma_load_2d(sb + B_BYTES / 2, &tmB0, &full[stage], kb * BK, b_row + BN / 2);
          }
          issued_parity[stage] = (int)phase;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // never leave the CTA with a bulk copy still writing its shared memory
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_parity[s], args.status);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      int g = 0;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
        while (tile >= tile_start[g + 1]) ++g;
        const int grows = rowend[g] - rowbeg[g];
        const bool swapped = swappable(MODE) && grows <= SWAP_ROWS;
        const int nt = (grows + 15) & ~15;  // N of the swapped MMAs
        const uint32_t idesc_sw = idesc_bf16_f32(BM, nt > 0 ? nt : 16);
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = smem_desc_sw128(sa);
          if (swappable(MODE) && swapped) {
            // weight halves as M (128 rows each), the group's rows as N
            const uint64_t w1 = smem_desc_sw128(sa + A_BYTES);
            const uint64_t w2 = smem_desc_sw128(sa + A_BYTES + B_BYTES / 2);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              tc_mma_bf16(d_tmem, w1 + 2ull * kk, adesc + 2ull * kk, idesc_sw, (kb | kk) != 0);
              tc_mma_bf16(d_tmem + (uint32_t)nt, w2 + 2ull * kk, adesc + 2ull * kk, idesc_sw, (kb | kk) != 0);
            }
          } else if (MODE == kPlainBT || MODE == kDualBT) {
            const uint64_t bdesc = smem_desc_sw128_mn(sa + A_BYTES, B_SLICE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)  // A: +32 B along K; B: +16 rows = +2048 B
              tc_mma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 128ull * kk, IDESC_BT, (kb | kk) != 0);
          } else {
            const uint64_t bdesc = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk) {
              // +32 bytes along K inside the 128-byte swizzle row = +2 in the address field
              tc_mma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, IDESC, (kb | kk) != 0);
            }
          }
          tc_commit(&empty[stage]);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit(&tfull[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int quad = warp & 3;  // TMEM lanes 32*quad .. 32*quad+31
    const int r = quad * 32 + lane;
    int g = 0;
    int it = 0;
    for (int tile = blockIdx.x; tile < total_tiles; tile += gridDim.x, ++it) {
      while (tile >= tile_start[g + 1]) ++g;
      const int local = tile - tile_start[g];
      const int n_tile = local / mtiles[g];
      const int m_tile = local - n_tile * mtiles[g];
      const int row0 = rowbeg[g] + m_tile * BM;
      const int rows_valid = min(BM, rowend[g] - row0);
      const int n0 = n_tile * OUT_COLS;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
      const int grows = rowend[g] - rowbeg[g];
      if (swappable(MODE) && grows <= SWAP_ROWS)
        epilogue_swapped<MODE>(taddr, args, row0, grows, (grows + 15) & ~15, n0, r);
      else
        epilogue_row<MODE>(taddr, args, row0 + r, r < rows_valid, n0);
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
// The same grouped GEMM on pairs of SMs (a cluster of two CTAs) with
// tcgen05.mma.cta_group::2: one pair computes a 256-row x 256-column tile.  Each
// CTA stages its own 128 rows of A and its half of the B tile (128 rows), so a
// CTA moves 32 KB per K block instead of 48 KB, which leaves room for six stages.
// CTA rank 0 (the leader) issues the MMAs; each CTA's tensor memory receives its
// 128 rows of the accumulator, which its own epilogue warps drain.
//   full[s]   in the leader: both CTAs' bulk copies complete on it; the leader
//             posts the expected bytes of both.
//   empty[s]  in each CTA: the leader's MMA commit arrives on both.
//   tfull[a]  in each CTA: the leader's commit after a tile arrives on both.
//   tempty[a] in the leader: all 8 epilogue warps of the pair arrive on it.
namespace pair {
constexpr int BM = 128;                          // rows per CTA; 256 per pair
constexpr int STAGES = 6;
constexpr int A_BYTES = BM * BK * 2;             // 16 KB
constexpr int BH_BYTES = 128 * BK * 2;           // 16 KB: this CTA's half of B
constexpr int STAGE_BYTES = A_BYTES + BH_BYTES;  // 32 KB
constexpr size_t SMEM_BYTES = 1024 + (size_t)STAGES * STAGE_BYTES + 256 + (size_t)(4 * MAX_GROUPS + 8) * 4;
constexpr uint32_t IDESC = idesc_bf16_f32(2 * BM, BN);
constexpr uint32_t IDESC_BT = idesc_bf16_f32_major(2 * BM, BN, false, true);
// Tile queue: the leader's producer takes the next tile from the counter and writes
// it to slot q of both CTAs (TQ slots), arriving on tq_full[q] of each; the leader's
// MMA thread, both CTAs' four epilogue warps and the peer's producer read it and
// arrive on the leader's tq_empty[q].
constexpr int TQ = 4;
constexpr uint32_t TQ_READERS = 1 + 4 + 1 + 4;
}  // namespace pair

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
                             const __grid_constant__ CUtensorMap tmB0, const __grid_constant__ CUtensorMap tmB1,
                             const Args args) {
  constexpr int STAGES = pair::STAGES, STAGE_BYTES = pair::STAGE_BYTES, A_BYTES = pair::A_BYTES;
  constexpr int BM = pair::BM;
  constexpr uint32_t IDESC = pair::IDESC;
  constexpr int OUT_COLS = paired_b(MODE) ? 128 : 256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + STAGES * STAGE_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *tq_full = tempty + 2;          // [TQ]
  uint64_t *tq_empty = tq_full + pair::TQ;  // [TQ], the leader's
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tq_empty + pair::TQ);
  volatile int *tq = reinterpret_cast<volatile int *>(tmem_slot + 2);  // [TQ] tile ids
  static_assert((2 * STAGES + 4 + 2 * pair::TQ) * 8 + 8 + 4 * pair::TQ <= 256, "barrier area");
  int *tile_start = reinterpret_cast<int *>(smem + STAGES * STAGE_BYTES + 256);
  int *mtiles = tile_start + MAX_GROUPS + 1;
  int *rowbeg = mtiles + MAX_GROUPS;
  int *rowend = rowbeg + MAX_GROUPS;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int G = args.G;
  const int n_tiles = (args.n_out + OUT_COLS - 1) / OUT_COLS;
  const int num_kb = args.num_kb;

  // gathered A: each CTA gathers its own 128 token rows by TMA (see the producer)
  const bool gather = swappable(MODE) && args.gx != nullptr;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 8);
    }
    for (int q = 0; q < pair::TQ; ++q) {
      mbar_init(&tq_full[q], 1);
      mbar_init(&tq_empty[q], pair::TQ_READERS);
    }
    fence_barrier_init();
    int acc = 0;
    for (int g = 0; g < G; ++g) {
      int b = args.offsets ? args.offsets[g] : 0;
      int e = args.offsets ? args.offsets[g + 1] : args.M;
      if (b < 0 || e < b || e > args.a_rows) {
        set_status(args.status, MOE_ERR_BOUNDS);
        b = e = 0;
      }
      rowbeg[g] = b;
      rowend[g] = e;
      const int mt = e > b ? (e - b + 2 * BM - 1) / (2 * BM) : 0;
      mtiles[g] = mt;
      tile_start[g] = acc;
      acc += mt * n_tiles;
    }
    tile_start[G] = acc;
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB0);
    if (paired_b(MODE) || MODE == kDualBT) tma_prefetch_desc(&tmB1);
    if (MODE == kDualBT) tma_prefetch_desc(&tmA2);
  }
  if (warp == 1) tmem_alloc_pair(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers are initialised before any cross-CTA use
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[G];
  const uint32_t full_lead = mapa_shared(smem_u32(&full[0]), 0);
  const uint32_t tempty_lead = mapa_shared(smem_u32(&tempty[0]), 0);
  const uint32_t tqe_lead = mapa_shared(smem_u32(&tq_empty[0]), 0);
  const uint32_t tqf_peer = mapa_shared(smem_u32(&tq_full[0]), 1);
  const uint32_t tq_peer = mapa_shared(smem_u32(const_cast<int *>(&tq[0])), 1);
  // The tile sequence, the same for every role of the pair: the leader's producer
  // publishes (publish = true), every other role reads.  One thread calls it; false
  // on a wait past its time limit.
  auto next_tile = [&](bool publish, int &q, uint32_t &qph, int &tile) -> bool {
    if (publish) {
      if (!mbar_wait_cluster(&tq_empty[q], qph ^ 1u, args.status)) return false;
      tile = atomicAdd(args.tile_counter, 1);
      if (tile >= total_tiles) tile = -1;
      tq[q] = tile;
      st_shared_cluster_u32(tq_peer + 4u * (uint32_t)q, (uint32_t)tile);
      mbar_arrive(&tq_full[q]);
      mbar_arrive_cluster(tqf_peer + 8u * (uint32_t)q);
    } else {
      if (!mbar_wait_cluster(&tq_full[q], qph, args.status)) return false;
      tile = tq[q];
      mbar_arrive_cluster(tqe_lead + 8u * (uint32_t)q);
    }
    if (++q == pair::TQ) {
      q = 0;
      qph ^= 1u;
    }
    return true;
  };

  if (warp == 0 && gather) {
    // ------------------------------------------------------------ producer, gathered A (both CTAs)
    // As in the single-CTA form: lane 0 waits for the stage and loads this CTA's
    // half of B (the leader also sets the pair's expected bytes); then the 32 lanes
    // gather this CTA's 128 token rows, 4 per lane, all counted on the leader's
    // full barrier.
    int issued_parity[STAGES];
    for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
    int stage = 0;
    uint32_t phase = 0;
    int g = 0;
    bool ok = true;
    const CUtensorMap *mb = (paired_b(MODE) && rank == 1) ? &tmB1 : &tmB0;
    int tq_q = 0;
    uint32_t tq_ph = 0;
    while (ok) {
      int tile = -1;
      bool got = true;
      if (lane == 0) got = next_tile(leader, tq_q, tq_ph, tile);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) break;
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0) break;
      while (tile >= tile_start[g + 1]) ++g;
      const int local = tile - tile_start[g];
      const int n_tile = local / mtiles[g];
      const int m_tile = local - n_tile * mtiles[g];
      const int a_row = rowbeg[g] + m_tile * 2 * BM + (int)rank * BM;
      const int b_row = paired_b(MODE) ? g * args.b_rows + n_tile * OUT_COLS
                                       : g * args.b_rows + n_tile * OUT_COLS + (int)rank * 128;
      int t[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int r = a_row + 4 * lane + j;
        t[j] = 0;
        if (r < rowend[g]) {
          const int v = args.gsrc[r];
          if (v < 0 || v >= args.gx_rows)
            set_status(args.status, MOE_ERR_BOUNDS);
          else
            t[j] = v;
        }
      }
      for (int kb = 0; kb < num_kb; ++kb) {
        uint8_t *sa = smem + stage * STAGE_BYTES;
        const uint32_t fb = full_lead + 8u * stage;
        bool go = true;
        if (lane == 0) {
          go = mbar_wait(&empty[stage], phase ^ 1u, args.status);
          if (go) {
            if (leader) mbar_arrive_expect_tx(&full[stage], 2u * STAGE_BYTES);
            tma_load_2d_pair(sa + A_BYTES, mb, fb, kb * BK, b_row);
            issued_parity[stage] = (int)phase;
          }
        }
        if (!__shfl_sync(0xffffffffu, go ? 1 : 0, 0)) {
          ok = false;
          break;
        }
        tma_gather4_pair(sa + lane * 512, &tmA, fb, kb * BK, t[0], t[1], t[2], t[3]);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // the leader's full barriers count both CTAs' copies: wait for the last ones
    if (leader && lane == 0)
      for (int s = 0; s < STAGES; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&full[s], (uint32_t)issued_parity[s], args.status);
  } else if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      int issued_parity[STAGES];
      for (int s = 0; s < STAGES; ++s) issued_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      int g = 0;
      bool ok = true;
      const CUtensorMap *mb = (paired_b(MODE) && rank == 1) ? &tmB1 : &tmB0;
      int tq_q = 0;
      uint32_t tq_ph = 0;
      while (ok) {
        int tile = -1;
        if (!next_tile(leader, tq_q, tq_ph, tile) || tile < 0) break;
        while (tile >= tile_start[g + 1]) ++g;
        const int local = tile - tile_start[g];
        const int n_tile = local / mtiles[g];
        const int m_tile = local - n_tile * mtiles[g];
        const int a_row = rowbeg[g] + m_tile * 2 * BM + (int)rank * BM;
        const int b_row = paired_b(MODE) ? g * args.b_rows + n_tile * OUT_COLS
                                         : g * args.b_rows + n_tile * OUT_COLS + (int)rank * 128;
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          uint8_t *sa = smem + stage * STAGE_BYTES;
          if (leader) mbar_arrive_expect_tx(&full[stage], 2u * STAGE_BYTES);
          const uint32_t fb = full_lead + 8u * stage;
          if (MODE == kPlainBT || MODE == kDualBT) {
            const bool second = MODE == kDualBT && kb >= args.kb1;
            const int k0 = (second ? kb - args.kb1 : kb) * BK;
            const CUtensorMap *mbt = second ? &tmB1 : &tmB0;
            tma_load_2d_pair(sa, second ? &tmA2 : &tmA, fb, k0, a_row);
            const int nb = n_tile * OUT_COLS + (int)rank * 128;  // this CTA's half of the tile's columns
#pragma unroll
            for (int j = 0; j < 2; ++j) tma_load_3d_pair(sa + A_BYTES + j * B_SLICE, mbt, fb, nb + 64 * j, k0, g);
          } else {
            tma_load_2d_pair(sa, &tmA, fb, kb * BK, a_row);
            tma_load_2d_pair(sa + A_BYTES, mb, fb, kb * BK, b_row);
          }
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
    // ------------------------------------------------------------ MMA issuer (leader only)
    if (leader && lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int it = 0;
      bool ok = true;
      int tq_q = 0;
      uint32_t tq_ph = 0;
      for (; ok; ++it) {
        int tile = -1;
        if (!next_tile(false, tq_q, tq_ph, tile) || tile < 0) break;
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait_cluster(&tempty[acc], (use & 1u) ^ 1u, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&full[stage], phase, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(smem + stage * STAGE_BYTES);
          const uint64_t adesc = smem_desc_sw128(sa);
          if (MODE == kPlainBT || MODE == kDualBT) {
            const uint64_t bdesc = smem_desc_sw128_mn(sa + A_BYTES, B_SLICE);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_bf16_pair(d_tmem, adesc + 2ull * kk, bdesc + 128ull * kk, pair::IDESC_BT, (kb | kk) != 0);
          } else {
            const uint64_t bdesc = smem_desc_sw128(sa + A_BYTES);
#pragma unroll
            for (int kk = 0; kk < BK / 16; ++kk)
              tc_mma_bf16_pair(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, IDESC, (kb | kk) != 0);
          }
          tc_commit_pair(&empty[stage], 0x3);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (ok) tc_commit_pair(&tfull[acc], 0x3);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int quad = warp & 3;
    const int r = quad * 32 + lane;
    int g = 0;
    int it = 0;
    int tq_q = 0;
    uint32_t tq_ph = 0;
    for (;; ++it) {
      // one tile id per warp: lane 0 reads the slot, frees it and passes the id on
      int tile = -1;
      bool got = true;
      if (lane == 0) got = next_tile(false, tq_q, tq_ph, tile);
      if (!__shfl_sync(0xffffffffu, got ? 1 : 0, 0)) break;
      tile = __shfl_sync(0xffffffffu, tile, 0);
      if (tile < 0) break;
      while (tile >= tile_start[g + 1]) ++g;
      const int local = tile - tile_start[g];
      const int n_tile = local / mtiles[g];
      const int m_tile = local - n_tile * mtiles[g];
      const int row0 = rowbeg[g] + m_tile * 2 * BM + (int)rank * BM;
      const int rows_valid = min(BM, rowend[g] - row0);
      const int n0 = n_tile * OUT_COLS;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
      epilogue_row<MODE>(taddr, args, row0 + r, r < rows_valid, n0);
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

// ---------------------------------------------------------------- host side
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

// 2-D bf16 map over a [rows, cols] row-major matrix (row stride `stride`
// elements, default cols), box 64 (cols) x box_rows (128 for tiles, 1 for row
// gathers), 128-byte swizzle; out-of-range elements read as zero.
static int make_map(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint64_t stride = 0,
                    uint32_t box_rows = BM) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if (!stride) stride = cols;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (stride * 2) % 16 || rows == 0 || cols == 0 || stride < cols)
    return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride * 2};
  cuuint32_t box[2] = {BK, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// 3-D bf16 map over G stacked [k, n] row-major matrices, box 64 (n) x 64 (k) x 1,
// 128-byte swizzle: one MN-major B slice.  Reads past k or n of a matrix are zero.
static int make_map_3d(CUtensorMap *m, const void *base, uint64_t G, uint64_t k, uint64_t n) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (n * 2) % 16 || G == 0 || k == 0 || n == 0) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[3] = {n, k, G};
  cuuint64_t strides[2] = {n * 2, n * k * 2};
  cuuint32_t box[3] = {64, BK, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? MOE_OK : MOE_ERR_CUDA;
}

// CTA pairs that can run at once (cluster occupancy), per device.
template <int MODE>
static int pair_grid(int device) {
  static std::mutex mu;
  static std::vector<int> cache;
  std::lock_guard<std::mutex> lk(mu);
  if ((int)cache.size() <= device) cache.resize(device + 1, 0);
  if (!cache[device]) {
    if (cudaFuncSetAttribute(grouped_gemm_pair_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)pair::SMEM_BYTES) != cudaSuccess)
      return -1;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * device_sm_count(device));
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = pair::SMEM_BYTES;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, grouped_gemm_pair_kernel<MODE>, &cfg) != cudaSuccess || clusters < 1)
      return -1;
    cache[device] = 2 * clusters;
  }
  return cache[device];
}

template <int MODE>
static int launch_pair(const CUtensorMap &ma, const CUtensorMap &ma2, const CUtensorMap &mb0, const CUtensorMap &mb1,
                       const Args &args, int device, cudaStream_t stream) {
  const int grid = pair_grid<MODE>(device);
  if (grid < 2) return MOE_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(THREADS);
  cfg.dynamicSmemBytes = pair::SMEM_BYTES;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  // the tile counter is the int after the workspace status word
  Args a = args;
  a.tile_counter = args.status + 1;
  if (cudaMemsetAsync(a.tile_counter, 0, sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<MODE>, ma, ma2, mb0, mb1, a) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

template <int MODE>
static int prepare_kernel(int device) {
  static std::mutex mu;
  static std::vector<int> done;
  std::lock_guard<std::mutex> lk(mu);
  if ((int)done.size() <= device) done.resize(device + 1, 0);
  if (!done[device]) {
    if (cudaFuncSetAttribute(grouped_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)SMEM_BYTES) != cudaSuccess)
      return MOE_ERR_CUDA;
    done[device] = 1;
  }
  return MOE_OK;
}

template <int MODE>
static int launch_single(const CUtensorMap &ma, const CUtensorMap &ma2, const CUtensorMap &mb0,
                         const CUtensorMap &mb1, const Args &args, int device, int sms, cudaStream_t stream) {
  int rc;
  if ((rc = prepare_kernel<MODE>(device))) return rc;
  grouped_gemm_kernel<MODE><<<dim3(sms), dim3(THREADS), SMEM_BYTES, stream>>>(ma, ma2, mb0, mb1, args);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

static int launch_mode(int mode, const CUtensorMap &ma, const CUtensorMap &ma2, const CUtensorMap &mb0,
                       const CUtensorMap &mb1, const Args &args, int device, int sms, bool pair_tiles,
                       cudaStream_t stream) {
  if (pair_tiles) {
    switch (mode) {
      case kSwiGLU: return launch_pair<kSwiGLU>(ma, ma2, mb0, mb1, args, device, stream);
      case kReLU: return launch_pair<kReLU>(ma, ma2, mb0, mb1, args, device, stream);
      case kPlain: return launch_pair<kPlain>(ma, ma2, mb0, mb1, args, device, stream);
      case kPlainBT: return launch_pair<kPlainBT>(ma, ma2, mb0, mb1, args, device, stream);
      case kDualBT: return launch_pair<kDualBT>(ma, ma2, mb0, mb1, args, device, stream);
      case kSwiGLUBwd: return launch_pair<kSwiGLUBwd>(ma, ma2, mb0, mb1, args, device, stream);
      default: return launch_pair<kReLUBwd>(ma, ma2, mb0, mb1, args, device, stream);
    }
  }
  switch (mode) {
    case kSwiGLU: return launch_single<kSwiGLU>(ma, ma2, mb0, mb1, args, device, sms, stream);
    case kReLU: return launch_single<kReLU>(ma, ma2, mb0, mb1, args, device, sms, stream);
    case kPlain: return launch_single<kPlain>(ma, ma2, mb0, mb1, args, device, sms, stream);
    case kPlainBT: return launch_single<kPlainBT>(ma, ma2, mb0, mb1, args, device, sms, stream);
    case kDualBT: return launch_single<kDualBT>(ma, ma2, mb0, mb1, args, device, sms, stream);
    case kSwiGLUBwd: return launch_single<kSwiGLUBwd>(ma, ma2, mb0, mb1, args, device, sms, stream);
    default: return launch_single<kReLUBwd>(ma, ma2, mb0, mb1, args, device, sms, stream);
  }
}

}  // namespace tc

int tc_grouped_gemm(int mode, const void *A, int64_t a_rows, int K, const void *B0, const void *B1,
                    int64_t b_rows_total, int b_rows_per_group, const int32_t *offsets, int G, int M, int n_out,
                    void *out, int *status, bool pair_tiles, cudaStream_t stream) {
  using namespace tc;
  if (G < 1 || G > MAX_GROUPS || K < 1 || n_out < 1 || a_rows < 1 || b_rows_total < 1) return MOE_ERR_INVALID_ARG;
  if (a_rows > INT32_MAX || n_out > b_rows_per_group || (int64_t)G * b_rows_per_group > b_rows_total)
    return MOE_ERR_INVALID_ARG;
  if (mode < kSwiGLU || mode > kPlain || (mode == kSwiGLU && !B1)) return MOE_ERR_INVALID_ARG;
  CUtensorMap ma, mb0, mb1;
  int rc;
  if ((rc = make_map(&ma, A, (uint64_t)a_rows, (uint64_t)K))) return rc;
  if ((rc = make_map(&mb0, B0, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  if (mode == kSwiGLU) {
    if ((rc = make_map(&mb1, B1, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  } else {
    mb1 = mb0;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  const int num_kb = (K + BK - 1) / BK;
  Args args{offsets, G, M, (int32_t)a_rows, n_out, K, b_rows_per_group, static_cast<uint16_t *>(out), status,
            num_kb, num_kb, n_out, nullptr};
  return launch_mode(mode, ma, ma, mb0, mb1, args, dev, sms, pair_tiles, stream);
}

int tc_grouped_gemm_gather(int mode, const void *x, int64_t x_rows, const int32_t *src_token, int64_t rows, int K,
                           const void *B0, const void *B1, int64_t b_rows_total, int b_rows_per_group,
                           const int32_t *offsets, int G, int n_out, void *out, int *status, bool pair_tiles,
                           cudaStream_t stream) {
  using namespace tc;
  if (G < 1 || G > MAX_GROUPS || K < 1 || n_out < 1 || rows < 1 || x_rows < 1 || b_rows_total < 1 || !src_token ||
      !offsets)
    return MOE_ERR_INVALID_ARG;
  if (rows > INT32_MAX || x_rows > INT32_MAX || n_out > b_rows_per_group ||
      (int64_t)G * b_rows_per_group > b_rows_total)
    return MOE_ERR_INVALID_ARG;
  if (mode < kSwiGLU || mode > kPlain || (mode == kSwiGLU && !B1)) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(x) & 15) || K % 8) return MOE_ERR_UNSUPPORTED;
  CUtensorMap ma, mb0, mb1;
  int rc;
  if ((rc = make_map(&ma, x, (uint64_t)x_rows, (uint64_t)K, 0, 1))) return rc;  // one-row boxes: row gathers
  if ((rc = make_map(&mb0, B0, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  if (mode == kSwiGLU) {
    if ((rc = make_map(&mb1, B1, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  } else {
    mb1 = mb0;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  const int num_kb = (K + BK - 1) / BK;
  Args args{offsets, G, 0, (int32_t)rows, n_out, K, b_rows_per_group, static_cast<uint16_t *>(out), status,
            num_kb, num_kb, n_out, nullptr, static_cast<const uint16_t *>(x), src_token, (int32_t)x_rows};
  return launch_mode(mode, ma, ma, mb0, mb1, args, dev, sms, pair_tiles, stream);
}

int tc_grouped_gemm_act_bwd(bool swiglu, const void *A, int64_t a_rows, int K, const void *W1, const void *W3,
                            int64_t b_rows_total, int F, const int32_t *offsets, int G, int M, const void *dh,
                            void *dA, int *status, bool pair_tiles, cudaStream_t stream) {
  using namespace tc;
  if (G < 1 || G > MAX_GROUPS || K < 1 || F < 1 || a_rows < 1 || a_rows > INT32_MAX || b_rows_total < 1)
    return MOE_ERR_INVALID_ARG;
  if ((int64_t)G * F > b_rows_total || !A || !W1 || (swiglu && !W3) || !dh || !dA) return MOE_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dh) | reinterpret_cast<uintptr_t>(dA)) & 15 || F % 8) return MOE_ERR_UNSUPPORTED;
  CUtensorMap ma, mb0, mb1;
  int rc;
  if ((rc = make_map(&ma, A, (uint64_t)a_rows, (uint64_t)K))) return rc;
  if ((rc = make_map(&mb0, W1, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  if (swiglu) {
    if ((rc = make_map(&mb1, W3, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  } else {
    mb1 = mb0;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  const int num_kb = (K + BK - 1) / BK;
  Args args{offsets, G, M, (int32_t)a_rows, F, K, F, static_cast<uint16_t *>(dA), status,
            num_kb, num_kb, swiglu ? 2 * F : F, static_cast<const uint16_t *>(dh)};
  return launch_mode(swiglu ? kSwiGLUBwd : kReLUBwd, ma, ma, mb0, mb1, args, dev, sms, pair_tiles, stream);
}

int tc_grouped_gemm_bt(const void *A, const void *A2, int64_t a_rows, int64_t a_stride, int K1, int K2,
                       const void *B0, const void *B1, int G, int n_out, const int32_t *offsets, int M, void *out,
                       int *status, bool pair_tiles, cudaStream_t stream) {
  using namespace tc;
  const bool dual = A2 != nullptr;
  if (G < 1 || G > MAX_GROUPS || K1 < 1 || n_out < 1 || a_rows < 1 || a_rows > INT32_MAX || !A || !B0 || !out)
    return MOE_ERR_INVALID_ARG;
  if (dual && (K2 < 1 || !B1)) return MOE_ERR_INVALID_ARG;
  if (a_stride < K1 || (dual && a_stride < K2)) return MOE_ERR_INVALID_ARG;
  CUtensorMap ma, ma2, mb0, mb1;
  int rc;
  if ((rc = make_map(&ma, A, (uint64_t)a_rows, (uint64_t)K1, (uint64_t)a_stride))) return rc;
  if ((rc = make_map_3d(&mb0, B0, (uint64_t)G, (uint64_t)K1, (uint64_t)n_out))) return rc;
  if (dual) {
    if ((rc = make_map(&ma2, A2, (uint64_t)a_rows, (uint64_t)K2, (uint64_t)a_stride))) return rc;
    if ((rc = make_map_3d(&mb1, B1, (uint64_t)G, (uint64_t)K2, (uint64_t)n_out))) return rc;
  } else {
    ma2 = ma;
    mb1 = mb0;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  const int kb1 = (K1 + BK - 1) / BK;
  const int num_kb = kb1 + (dual ? (K2 + BK - 1) / BK : 0);
  Args args{offsets, G, M, (int32_t)a_rows, n_out, K1, 0, static_cast<uint16_t *>(out), status, num_kb, kb1, n_out,
            nullptr};
  return launch_mode(dual ? kDualBT : kPlainBT, ma, ma2, mb0, mb1, args, dev, sms, pair_tiles, stream);
}

}  // namespace moe
