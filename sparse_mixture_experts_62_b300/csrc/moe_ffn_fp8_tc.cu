// Expert FFN with FP8 E4M3 weights (one float32 scale per output row) on the
// tcgen05 tensor cores.
//
// The pages leave the quantisation of experts open ("Stanford CS336 lecture 4",
// the section on compressing sparse MoEs: fewer bits per weight, paid for with
// scales and a dequantisation step); the reading taken is weight-only E4M3 with
// a float32 scale per output row: W[n, :] = s[n] * q[n, :].  Then
//   out[r, n] = EPI( s[n] * sum_k A[r, k] q[n, k] ),
// so the scale factors out of the K sum.  Every E4M3 value is a bf16 value, so the
// codes are turned into bf16 exactly and the product runs as the bf16 grouped
// GEMM; the epilogue multiplies each accumulator column by its row's scale.  The
// weights stream from HBM at one byte each: the memory-bound decode reads half the
// bytes of bf16 weights.
//
// Two kernels.  Groups of at most 64 rows (decode) take the second one below, which
// puts the weights on the M side of the MMA and their converted bf16 in tensor
// memory.  Larger groups take this first one, which tiles the tokens on M and the
// weight rows on N and converts the codes into a shared-memory B operand.
//
// Kernel shape (one CTA per SM, persistent over output tiles, 352 threads), three
// rings so that many weight bytes are in flight:
//   codes  6 x 16 KB  (E4M3, 256 rows x 64 bytes, no swizzle)   warp 0 loads (TMA)
//   A      2 x 16 KB  (bf16, 128 x 64, 128-byte swizzle)        warp 10 loads (TMA)
//   B      2 x 32 KB  (bf16, 256 x 64, K-major, 128-byte swizzle)
//   warps 6-9   convert a code tile into a B tile, fence it for the tensor core,
//               and signal it; the code buffer is released at once.
//   warp 1      MMA issuer: M=128, N=256, K=16 into one of two TMEM accumulators;
//               its commits release the A and B buffers.
//   warps 2-5   epilogue: scale, activation, bf16 stores masked to the group.
// Tiles run group by group as in the bf16 kernel.  Waits are bounded as there.
#include <cuda_fp8.h>

#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace f8 {

constexpr int BM = 128, BN = 256, BK = 64, THREADS = 352;
constexpr int NR = 6, NA = 2, NC = 2;                      // ring depths: codes, A, converted B
constexpr int A_BYTES = BM * BK * 2;                       // 16 KB
constexpr int R_BYTES = BN * BK;                           // 16 KB of E4M3 codes
constexpr int C_BYTES = BN * BK * 2;                       // 32 KB of converted bf16
constexpr int RING_BYTES = NR * R_BYTES + NA * A_BYTES + NC * C_BYTES;  // 192 KB
constexpr int MAX_GROUPS = 257;
constexpr uint32_t TMEM_COLS = 512;
constexpr size_t SMEM_BYTES = 1024 + (size_t)RING_BYTES + 256 + (size_t)(4 * MAX_GROUPS + 8) * 4;
constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN);

enum Mode { kSwiGLU = 0, kReLU = 1, kPlain = 2 };

struct Args {
  const int32_t *offsets;  // [G + 1] group row offsets, or nullptr: one group of M rows
  int32_t G;
  int32_t M;
  int32_t a_rows;
  int32_t n_out;
  int32_t b_rows;          // weight rows per group
  int32_t num_kb;
  const float *scale0;     // [G * b_rows] scales of the first weight (W1 or W2)
  const float *scale1;     // [G * b_rows] scales of W3 (kSwiGLU)
  uint16_t *out;           // [a_rows, n_out] bf16
  int *status;
};

__device__ __forceinline__ float silu(float a) { return __fdividef(a, 1.0f + __expf(-a)); }

// Two E4M3 codes -> two bf16 (exact) packed low/high.
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t two) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(two), __NV_E4M3);
  const float2 f = __half22float2(__half2(h));
  return pack_bf16x2(f.x, f.y);
}

template <int MODE>
__global__ void __launch_bounds__(THREADS, 1)
    grouped_gemm_fp8_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmQ0,
                            const __grid_constant__ CUtensorMap tmQ1, const Args args) {
  constexpr int OUT_COLS = (MODE == kSwiGLU) ? 128 : 256;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t *cbuf = smem;                                // NC x 32 KB (1024-aligned)
  uint8_t *abuf = cbuf + NC * C_BYTES;                 // NA x 16 KB
  uint8_t *rbuf = abuf + NA * A_BYTES;                 // NR x 16 KB
  uint64_t *r_full = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
  uint64_t *r_empty = r_full + NR;
  uint64_t *a_full = r_empty + NR;
  uint64_t *a_empty = a_full + NA;
  uint64_t *c_full = a_empty + NA;
  uint64_t *c_empty = c_full + NC;
  uint64_t *tfull = c_empty + NC;
  uint64_t *tempty = tfull + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tempty + 2);
  int *tile_start = reinterpret_cast<int *>(smem + RING_BYTES + 256);
  int *mtiles = tile_start + MAX_GROUPS + 1;
  int *rowbeg = mtiles + MAX_GROUPS;
  int *rowend = rowbeg + MAX_GROUPS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;
  const int n_tiles = (args.n_out + OUT_COLS - 1) / OUT_COLS;
  const int num_kb = args.num_kb;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NR; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 4);  // one arrival per converter warp
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&a_full[s], 1);
      mbar_init(&a_empty[s], 1);
    }
    for (int s = 0; s < NC; ++s) {
      mbar_init(&c_full[s], 4);
      mbar_init(&c_empty[s], 1);
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
      if (b < 0 || e < b || e > args.a_rows) {
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
    tma_prefetch_desc(&tmQ0);
    if (MODE == kSwiGLU) tma_prefetch_desc(&tmQ1);
  }
  if (warp == 10 && lane == 0) tma_prefetch_desc(&tmA);
  if (warp == 1) tmem_alloc(tmem_slot, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total_tiles = tile_start[G];

  if (warp == 0 || warp == 10) {
    // ------------------------------------------------------------ TMA producers: codes (warp 0), A (warp 10)
    if (lane == 0) {
      const bool codes = warp == 0;
      const int depth = codes ? NR : NA;
      uint64_t *fullb = codes ? r_full : a_full;
      uint64_t *emptyb = codes ? r_empty : a_empty;
      int issued_parity[NR];
      for (int s = 0; s < NR; ++s) issued_parity[s] = -1;
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
          if (!mbar_wait(&emptyb[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          if (codes) {
            uint8_t *sr = rbuf + stage * R_BYTES;
            mbar_arrive_expect_tx(&fullb[stage], R_BYTES);
            if (MODE == kSwiGLU) {
              tma_load_2d(sr, &tmQ0, &fullb[stage], kb * BK, b_row);
              tma_load_2d(sr + R_BYTES / 2, &tmQ1, &fullb[stage], kb * BK, b_row);
            } else {
              tma_load_2d(sr, &tmQ0, &fullb[stage], kb * BK, b_row);
              tma_load_2d(sr + R_BYTES / 2, &tmQ0, &fullb[stage], kb * BK, b_row + BN / 2);
            }
          } else {
            mbar_arrive_expect_tx(&fullb[stage], A_BYTES);
            tma_load_2d(abuf + stage * A_BYTES, &tmA, &fullb[stage], kb * BK, a_row);
          }
          issued_parity[stage] = (int)phase;
          if (++stage == depth) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // never leave the CTA with a bulk copy still writing its shared memory
      for (int s = 0; s < depth; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&fullb[s], (uint32_t)issued_parity[s], args.status);
    }
  } else if (warp >= 6) {
    // ------------------------------------------------------------ E4M3 -> bf16 converters (warps 6-9)
    const int tid = threadIdx.x - 192;  // 0..127: rows tid and tid + 128
    int rs = 0, cs = 0;
    uint32_t rph = 0, cph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < num_kb; ++kb) {
        if (!__all_sync(0xffffffffu, mbar_wait(&r_full[rs], rph, args.status)) ||
            !__all_sync(0xffffffffu, mbar_wait(&c_empty[cs], cph ^ 1u, args.status))) {
          ok = false;
          break;
        }
        const uint8_t *sr = rbuf + rs * R_BYTES;
        uint8_t *sc = cbuf + cs * C_BYTES;
#pragma unroll
        for (int q = 0; q < 2; ++q) {
          const int row = tid + 128 * q;
          const uint4 *src = reinterpret_cast<const uint4 *>(sr + row * BK);
#pragma unroll
          for (int h = 0; h < 4; ++h) {  // 16 codes -> two 16-byte chunks of bf16
            const uint4 v = src[h];
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t o[8];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              o[2 * i] = e4m3x2_to_bf16x2((uint16_t)(w[i] & 0xFFFFu));
              o[2 * i + 1] = e4m3x2_to_bf16x2((uint16_t)(w[i] >> 16));
            }
            const int c0 = 2 * h, c1 = 2 * h + 1;
            *reinterpret_cast<uint4 *>(sc + row * 128 + ((c0 ^ (row & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4 *>(sc + row * 128 + ((c1 ^ (row & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&r_empty[rs]);
          mbar_arrive(&c_full[cs]);
        }
        if (++rs == NR) {
          rs = 0;
          rph ^= 1u;
        }
        if (++cs == NC) {
          cs = 0;
          cph ^= 1u;
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int as = 0, cs = 0;
      uint32_t aph = 0, cph = 0;
      int it = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < total_tiles && ok; tile += gridDim.x, ++it) {
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, args.status)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!mbar_wait(&a_full[as], aph, args.status) || !mbar_wait(&c_full[cs], cph, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t adesc = smem_desc_sw128(smem_u32(abuf + as * A_BYTES));
          const uint64_t bdesc = smem_desc_sw128(smem_u32(cbuf + cs * C_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_bf16(d_tmem, adesc + 2ull * kk, bdesc + 2ull * kk, IDESC, (kb | kk) != 0);
          tc_commit(&a_empty[as]);
          tc_commit(&c_empty[cs]);
          if (++as == NA) {
            as = 0;
            aph ^= 1u;
          }
          if (++cs == NC) {
            cs = 0;
            cph ^= 1u;
          }
        }
        if (ok) tc_commit(&tfull[acc]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (warps 2-5)
    const int quad = warp & 3;
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
      const float *s0 = args.scale0 + (size_t)g * args.b_rows;
      const float *s1 = (MODE == kSwiGLU) ? args.scale1 + (size_t)g * args.b_rows : nullptr;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * BN) + ((uint32_t)(quad * 32) << 16);
      const bool row_ok = r < rows_valid;
      uint16_t *orow = args.out + (size_t)(row0 + (row_ok ? r : 0)) * args.n_out;
      if (MODE == kSwiGLU) {
#pragma unroll 1
        for (int c = 0; c < 128; c += 16) {
          float a[16], u[16];
          tmem_ld16x2(taddr + c, taddr + 128 + c, a, u);
          const int col = n0 + c;
          if (!row_ok || col >= args.n_out) continue;
          uint32_t p[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c2 = min(col + 2 * i, args.n_out - 2);  // columns past n_out are not stored
            const float a0 = a[2 * i] * s0[c2], a1 = a[2 * i + 1] * s0[c2 + 1];
            const float u0 = u[2 * i] * s1[c2], u1 = u[2 * i + 1] * s1[c2 + 1];
            p[i] = pack_bf16x2(silu(a0) * u0, silu(a1) * u1);
          }
          if (col + 8 <= args.n_out) *reinterpret_cast<uint4 *>(orow + col) = make_uint4(p[0], p[1], p[2], p[3]);
          if (col + 16 <= args.n_out) *reinterpret_cast<uint4 *>(orow + col + 8) = make_uint4(p[4], p[5], p[6], p[7]);
        }
      } else {
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
            for (int i = 0; i < 8; ++i) {
              x[i] = v[i] * s0[col + i];
              if (MODE == kReLU) x[i] = fmaxf(x[i], 0.f);
            }
            *reinterpret_cast<uint4 *>(orow + col) = make_uint4(pack_bf16x2(x[0], x[1]), pack_bf16x2(x[2], x[3]),
                                                                pack_bf16x2(x[4], x[5]), pack_bf16x2(x[6], x[7]));
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

}  // namespace f8

// ---------------------------------------------------------------------------
// The whole expert FFN for groups of at most a few dozen rows (decode), in one
// persistent launch.  The weights take the M side of the MMA and the group's
// tokens the N side,
//   D[n, t] = sum_k q[n, k] A[t, k]   (M = 128 weight rows, N = NT tokens),
// and the converted weights never touch shared memory: each converter thread
// turns its weight row's codes into bf16 in registers and writes them with
// tcgen05.st into tensor memory, where the MMA reads them as its A operand.
// Shared memory only holds the TMA-loaded codes (64-byte swizzle, so that the
// row-per-thread reads are free of bank conflicts) and the small token tiles,
// each in a ring of its own.
//   warps 0-3    epilogue (one TMEM lane quadrant each)
//   warps 4-11   converters, two sets of four taking alternate stages
//   warp 12      TMA producer of the codes of a stage
//   warp 13      TMEM owner and MMA issuer
//   warp 14      TMA producer of the stage's token tile
// A stage is four 128 x 64-byte boxes of codes: W1 and W3 over K = 128 for the
// SwiGLU gate/up product, else one weight over K = 256.
//
// Phase 0 (gate/up: h = act(x W1^T, x W3^T)) and phase 1 (down: y = h W2^T) run in
// one tile list, phase 0 first, dealt round-robin to the CTAs, so that the last,
// partial round of gate/up tiles overlaps down tiles instead of leaving SMs idle.
// A down tile of expert g reads rows of h written by all gate/up tiles of g: each
// gate/up epilogue warp counts its stores into dep[g] (fence, then an atomic add);
// the token producer of a down tile waits until dep[g] is complete (acquire load,
// bounded like every wait), then orders those writes before its TMA reads
// (fence.proxy.async.global).  The launch is cooperative: all CTAs are resident,
// and a CTA reaches its down tiles only after its own gate/up tiles, so the
// counters always complete.
namespace f8s {

using f8::kReLU;
using f8::kSwiGLU;

constexpr int BMW = 128, MAX_GROUPS = 257;
constexpr int W_TMA = 12, W_MMA = 13, W_TOK = 14, THREADS = 480;
constexpr int BOX_BYTES = BMW * 64;        // one 128 x 64 box of codes
constexpr int CODE_BYTES = 4 * BOX_BYTES;  // one stage of codes
constexpr int ACOLS = 128;                 // TMEM columns of one converted stage

template <int NT>
struct Shape {
  static constexpr int TOK_BYTES = 4 * NT * 128;  // up to four 64-wide token boxes
  // Codes and tokens have rings of their own: a code stage is free once converted,
  // a token stage once its MMAs are done.
  static constexpr int NTR = NT <= 32 ? 4 : 3;
  static constexpr int NR = (196608 - NTR * TOK_BYTES) / CODE_BYTES;
  static constexpr int RING = NR * CODE_BYTES + NTR * TOK_BYTES;
  static constexpr int DCOLS = 4 * NT;  // two accumulators of 2 x NT columns
  static constexpr int NA = (512 - DCOLS) / ACOLS;
  static constexpr size_t SMEM = 1024 + (size_t)RING + 512 + (size_t)(5 * MAX_GROUPS + 8) * 4;
  static_assert(TOK_BYTES % 1024 == 0 && NA >= 2 && NR >= 3, "stage layout");
};

struct Phase {
  int32_t n_out;   // output features
  int32_t b_rows;  // weight rows per group
  int32_t num_kb;  // stages
  int32_t nw;      // weights per stage: 2 (W1 and W3, K = 128) or 1 (K = 256)
  const float *s0;
  const float *s1;
  uint16_t *out;   // [a_rows, n_out] bf16
};

struct Args {
  const int32_t *offsets;  // [G + 1] group row offsets
  int32_t G;
  int32_t a_rows;
  int32_t act;             // kSwiGLU or kReLU (phase 0)
  Phase ph[2];
  int *dep;                // [G] gate/up epilogue-warp completions per group, zero at launch
  int *status;
};

// Four E4M3 codes (the bytes of w, lowest first) -> four bf16, two per word.
// Each code's sign, 4-bit exponent field and 3-bit mantissa are placed in a bf16
// with the same sign, the same exponent field and the mantissa at its top: that
// bf16 is the code's value times 2^-120 (bias 127 against 7; with a zero field
// both are subnormal with the same mantissa), so one multiplication by 2^120,
// exact in bf16, yields the value.  The two NaN codes come out as +-480, so
// they are not valid weights.
__device__ __forceinline__ uint32_t bf16x2_mul_exact(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ void e4m3x4_to_bf16(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t a = __byte_perm(w, 0u, 0x1404);  // code1 << 24 | code0 << 8
  const uint32_t b = __byte_perm(w, 0u, 0x3424);  // code3 << 24 | code2 << 8
  lo = bf16x2_mul_exact((a & 0x80008000u) | ((a >> 4) & 0x07F007F0u), 0x7B807B80u);  // x 2^120
  hi = bf16x2_mul_exact((b & 0x80008000u) | ((b >> 4) & 0x07F007F0u), 0x7B807B80u);
}
// The same bits by integer multiply-add, which runs on the FMA pipe instead of the
// integer-logic pipe: with x = code1 << 16 | code0, code << 4 puts exponent field
// and mantissa at bits 10-4 and the sign at bit 11, and adding 0x7800 for a set
// sign carries it to bit 15.  The decoders send one word in four this way: the
// logic pipe is the busiest one in the gate/up launch (three quarters of its
// cycles), and the multiply form's longer dependency chain costs more than it
// saves when used for half the words or more (measured).
__device__ __forceinline__ void e4m3x4_to_bf16_fma(uint32_t w, uint32_t &lo, uint32_t &hi) {
  const uint32_t a = __byte_perm(w, 0u, 0x4140);  // code1 << 16 | code0
  const uint32_t b = __byte_perm(w, 0u, 0x4342);  // code3 << 16 | code2
  lo = bf16x2_mul_exact(a * 16u + (a & 0x00800080u) * 240u, 0x7B807B80u);
  hi = bf16x2_mul_exact(b * 16u + (b & 0x00800080u) * 240u, 0x7B807B80u);
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t *v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]), "r"(v[17]),
      "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]), "r"(v[25]), "r"(v[26]),
      "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Each thread reads 16 consecutive 32-bit columns of its lane (load and wait in one statement).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *a) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) a[i] = __uint_as_float(r[i]);
}

// D[tmem] (+)= A[tmem] * B[smem]^T
__device__ __forceinline__ void tc_mma_bf16_ta(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(tmem_d),
      "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Wait until *counter >= target (acquire, GPU scope); false (and MOE_ERR_TIMEOUT)
// past the wait limit.
__device__ __forceinline__ bool wait_count(const int *counter, int target, int *status) {
  const uint64_t t0 = global_ns();
  for (;;) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
    if (v >= target) return true;
    if (global_ns() - t0 > kWaitLimitNs) {
      set_status(status, MOE_ERR_TIMEOUT);
      return false;
    }
    __nanosleep(200);
  }
}

// The tile list: phase-0 tiles of every group, then phase-1 tiles; within a phase
// and group, weight tile-major over token tiles.
struct Tiles {
  const int *start0, *start1, *ttiles;  // per-group first tile of each phase; token tiles per group
  int total0, total;
  int w_tiles[2];
  struct Tile {
    int phase, g, wt, tt;
  };
  // Resolves tile t; `g` is a cursor that only moves forward within a phase.
  __device__ Tile at(int t, int &g, int &phase_seen) const {
    Tile r;
    r.phase = t < total0 ? 0 : 1;
    if (r.phase != phase_seen) {
      phase_seen = r.phase;
      g = 0;
    }
    const int *st = r.phase ? start1 : start0;
    while (t >= st[g + 1]) ++g;
    const int local = t - st[g];
    r.g = g;
    r.wt = local / ttiles[g];
    r.tt = local - r.wt * ttiles[g];
    return r;
  }
};

template <int NT>
__global__ void __launch_bounds__(THREADS, 1)
    fp8_ffn_decode_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmH,
                          const __grid_constant__ CUtensorMap tmQ1, const __grid_constant__ CUtensorMap tmQ3,
                          const __grid_constant__ CUtensorMap tmQ2, const Args args) {
  using S = Shape<NT>;
  constexpr int NR = S::NR, NA = S::NA, NTR = S::NTR;
  constexpr uint32_t IDESC = idesc_bf16_f32(BMW, NT);
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024 - (raw_addr & 1023)) & 1023);
  uint8_t *tok_ring = smem + NR * CODE_BYTES;
  uint64_t *r_full = reinterpret_cast<uint64_t *>(smem + S::RING);
  uint64_t *r_empty = r_full + NR;
  uint64_t *k_full = r_empty + NR;
  uint64_t *k_empty = k_full + NTR;
  uint64_t *a_full = k_empty + NTR;
  uint64_t *a_empty = a_full + NA;
  uint64_t *tfull = a_empty + NA;
  uint64_t *tempty = tfull + 2;
  uint64_t *done = tempty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(done + 1);
  int *start0 = reinterpret_cast<int *>(smem + S::RING + 512);
  int *start1 = start0 + MAX_GROUPS + 1;
  int *ttiles = start1 + MAX_GROUPS + 1;
  int *rowbeg = ttiles + MAX_GROUPS;
  int *rowend = rowbeg + MAX_GROUPS;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = args.G;
  Tiles tl;
  tl.w_tiles[0] = (args.ph[0].n_out + BMW - 1) / BMW;
  tl.w_tiles[1] = (args.ph[1].n_out + BMW - 1) / BMW;

  if (threadIdx.x == 0) {
    for (int s = 0; s < NR; ++s) {
      mbar_init(&r_full[s], 1);
      mbar_init(&r_empty[s], 4);  // the four converter warps of a set
    }
    for (int s = 0; s < NTR; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);  // the MMA's commit
    }
    for (int s = 0; s < NA; ++s) {
      mbar_init(&a_full[s], 4);
      mbar_init(&a_empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(done, 1);
    fence_barrier_init();
    int acc0 = 0, acc1 = 0;
    for (int g = 0; g < G; ++g) {
      int b = args.offsets[g], e = args.offsets[g + 1];
      if (b < 0 || e < b || e > args.a_rows) {
        set_status(args.status, MOE_ERR_BOUNDS);
        b = e = 0;
      }
      rowbeg[g] = b;
      rowend[g] = e;
      const int tt = (e - b + NT - 1) / NT;
      ttiles[g] = tt;
      start0[g] = acc0;
      start1[g] = acc1;
      acc0 += tt * tl.w_tiles[0];
      acc1 += tt * tl.w_tiles[1];
    }
    start0[G] = acc0;
    start1[G] = acc1;
    for (int g = 0; g <= G; ++g) start1[g] += acc0;  // phase-1 tiles follow all phase-0 tiles
  }
  if (warp == W_TMA && lane == 0) {
    tma_prefetch_desc(&tmQ1);
    if (args.act == kSwiGLU) tma_prefetch_desc(&tmQ3);
    tma_prefetch_desc(&tmQ2);
  }
  if (warp == W_TOK && lane == 0) {
    tma_prefetch_desc(&tmX);
    tma_prefetch_desc(&tmH);
  }
  if (warp == W_MMA) tmem_alloc(tmem_slot, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  tl.start0 = start0;
  tl.start1 = start1;
  tl.ttiles = ttiles;
  tl.total0 = start0[G];
  tl.total = start1[G];

  if (warp == W_TMA || warp == W_TOK) {
    // ------------------------------------------------------------ TMA producers: codes (W_TMA), tokens (W_TOK)
    if (lane == 0) {
      const bool codes = warp == W_TMA;
      const int depth = codes ? NR : NTR;
      uint64_t *fullb = codes ? r_full : k_full;
      uint64_t *emptyb = codes ? r_empty : k_empty;
      int issued_parity[NR > NTR ? NR : NTR];
      for (int s = 0; s < depth; ++s) issued_parity[s] = -1;
      int stage = 0;
      uint32_t phase = 0;
      int g = 0, seen = -1;
      bool ok = true;
      for (int t = blockIdx.x; ok && t < tl.total; t += gridDim.x) {
        const Tiles::Tile tile = tl.at(t, g, seen);
        const Phase &P = args.ph[tile.phase];
        const int w_row = tile.g * P.b_rows + tile.wt * BMW;
        const int t_row = rowbeg[tile.g] + tile.tt * NT;
        const int ks = P.nw == 2 ? 128 : 256;  // K per stage
        if (!codes && tile.phase == 1) {  // the h rows of this group are written by gate/up tiles
          if (!wait_count(&args.dep[tile.g], 4 * tl.w_tiles[0] * ttiles[tile.g], args.status)) ok = false;
          asm volatile("fence.proxy.async.global;" ::: "memory");
        }
        for (int kb = 0; ok && kb < P.num_kb; ++kb) {
          if (!mbar_wait(&emptyb[stage], phase ^ 1u, args.status)) {
            ok = false;
            break;
          }
          if (codes) {
            uint8_t *st = smem + stage * CODE_BYTES;
            mbar_arrive_expect_tx(&fullb[stage], CODE_BYTES);
            if (P.nw == 2) {
              tma_load_2d(st, &tmQ1, &fullb[stage], kb * ks, w_row);
              tma_load_2d(st + BOX_BYTES, &tmQ1, &fullb[stage], kb * ks + 64, w_row);
              tma_load_2d(st + 2 * BOX_BYTES, &tmQ3, &fullb[stage], kb * ks, w_row);
              tma_load_2d(st + 3 * BOX_BYTES, &tmQ3, &fullb[stage], kb * ks + 64, w_row);
            } else {
              const CUtensorMap *q = tile.phase ? &tmQ2 : &tmQ1;
#pragma unroll
              for (int b = 0; b < 4; ++b) tma_load_2d(st + b * BOX_BYTES, q, &fullb[stage], kb * ks + 64 * b, w_row);
            }
          } else {
            uint8_t *st = tok_ring + stage * S::TOK_BYTES;
            const int nb = ks / 64;
            const CUtensorMap *m = tile.phase ? &tmH : &tmX;
            mbar_arrive_expect_tx(&fullb[stage], (uint32_t)(nb * NT * 128));
            for (int b = 0; b < nb; ++b) tma_load_2d(st + b * NT * 128, m, &fullb[stage], kb * ks + 64 * b, t_row);
          }
          issued_parity[stage] = (int)phase;
          if (++stage == depth) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      for (int s = 0; s < depth; ++s)
        if (issued_parity[s] >= 0) mbar_wait(&fullb[s], (uint32_t)issued_parity[s], args.status);
    }
  } else if (warp >= 4 && warp < 12) {
    // ------------------------------------------------------------ converters
    const int set = (warp - 4) >> 2;
    const int quad = warp & 3;
    const int r = quad * 32 + lane;  // weight row of this thread = TMEM lane
    const uint32_t lane_base = tmem_base + ((uint32_t)(quad * 32) << 16) + (uint32_t)S::DCOLS;
    const int swz = (r >> 1) & 3;
    int c = 0;  // stage counter of this CTA
    int g = 0, seen = -1;
    bool ok = true;
    for (int t = blockIdx.x; ok && t < tl.total; t += gridDim.x) {
      const Tiles::Tile tile = tl.at(t, g, seen);
      const int nkb = args.ph[tile.phase].num_kb;
      for (int kb = 0; kb < nkb; ++kb, ++c) {
        if ((c & 1) != set) continue;
        const int rs = c % NR, as = c % NA;
        const uint32_t rph = (uint32_t)(c / NR) & 1u, aph = (uint32_t)(c / NA) & 1u;
        if (!__all_sync(0xffffffffu, mbar_wait(&r_full[rs], rph, args.status)) ||
            !__all_sync(0xffffffffu, mbar_wait(&a_empty[as], aph ^ 1u, args.status))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint8_t *st = smem + rs * CODE_BYTES + r * 64;
#pragma unroll
        for (int b = 0; b < 4; ++b) {  // box b -> TMEM columns [32 b, 32 b + 32) of the slot
          uint32_t o[32];
#pragma unroll
          for (int ch = 0; ch < 4; ++ch) {
            const uint4 v = *reinterpret_cast<const uint4 *>(st + b * BOX_BYTES + ((ch ^ swz) << 4));
            e4m3x4_to_bf16(v.x, o[8 * ch + 0], o[8 * ch + 1]);
            e4m3x4_to_bf16(v.y, o[8 * ch + 2], o[8 * ch + 3]);
            e4m3x4_to_bf16(v.z, o[8 * ch + 4], o[8 * ch + 5]);
            e4m3x4_to_bf16_fma(v.w, o[8 * ch + 6], o[8 * ch + 7]);
          }
          tmem_st32(lane_base + (uint32_t)(as * ACOLS + b * 32), o);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&r_empty[rs]);
          mbar_arrive(&a_full[as]);
        }
      }
    }
  } else if (warp == W_MMA) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int ks = 0, as = 0;
      uint32_t kph = 0, aph = 0;
      int it = 0;
      int g = 0, seen = -1;
      bool ok = true, issued = false;
      for (int t = blockIdx.x; ok && t < tl.total; t += gridDim.x, ++it) {
        const Tiles::Tile tile = tl.at(t, g, seen);
        const Phase &P = args.ph[tile.phase];
        const int acc = it & 1;
        const uint32_t use = (uint32_t)(it >> 1);
        if (!mbar_wait(&tempty[acc], (use & 1u) ^ 1u, args.status)) break;
        tc_fence_after();
        const uint32_t d0 = tmem_base + (uint32_t)(acc * 2 * NT);
        for (int kb = 0; kb < P.num_kb; ++kb) {
          if (!mbar_wait(&k_full[ks], kph, args.status) || !mbar_wait(&a_full[as], aph, args.status)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = tmem_base + (uint32_t)(S::DCOLS + as * ACOLS);
          const uint32_t tok = smem_u32(tok_ring + ks * S::TOK_BYTES);
          if (P.nw == 2) {  // W1 in columns 0-63 and W3 in 64-127, K = 128
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
              const uint64_t bdesc = smem_desc_sw128(tok + (uint32_t)((kk >> 2) * NT * 128)) + 2ull * (kk & 3);
              const uint32_t accum = (kb | kk) != 0;
              tc_mma_bf16_ta(d0, a0 + 8u * kk, bdesc, IDESC, accum);
              tc_mma_bf16_ta(d0 + NT, a0 + 64u + 8u * kk, bdesc, IDESC, accum);
            }
          } else {  // one weight, K = 256
#pragma unroll
            for (int kk = 0; kk < 16; ++kk) {
              const uint64_t bdesc = smem_desc_sw128(tok + (uint32_t)((kk >> 2) * NT * 128)) + 2ull * (kk & 3);
              tc_mma_bf16_ta(d0, a0 + 8u * kk, bdesc, IDESC, (kb | kk) != 0);
            }
          }
          issued = true;
          tc_commit(&a_empty[as]);
          tc_commit(&k_empty[ks]);
          if (++ks == NTR) {
            ks = 0;
            kph ^= 1u;
          }
          if (++as == NA) {
            as = 0;
            aph ^= 1u;
          }
        }
        if (ok) tc_commit(&tfull[acc]);
      }
      if (issued) {  // every MMA has finished with tensor memory before it is freed
        tc_commit(done);
        mbar_wait(done, 0, args.status);
      }
    }
  } else if (warp < 4) {
    // ------------------------------------------------------------ epilogue (warps 0-3)
    const int quad = warp;
    int g = 0, seen = -1;
    int it = 0;
    for (int t = blockIdx.x; t < tl.total; t += gridDim.x, ++it) {
      const Tiles::Tile tile = tl.at(t, g, seen);
      const Phase &P = args.ph[tile.phase];
      const int t_row = rowbeg[tile.g] + tile.tt * NT;
      const int nvalid = min(NT, rowend[tile.g] - t_row);
      const int f = tile.wt * BMW + quad * 32 + lane;
      const bool f_ok = f < P.n_out;
      const bool glu = P.nw == 2;
      const bool relu = tile.phase == 0 && args.act == kReLU;
      const float s0 = f_ok ? P.s0[(size_t)tile.g * P.b_rows + f] : 0.f;
      const float s1 = (glu && f_ok) ? P.s1[(size_t)tile.g * P.b_rows + f] : 0.f;
      const int acc = it & 1;
      const uint32_t use = (uint32_t)(it >> 1);
      if (!mbar_wait(&tfull[acc], use & 1u, args.status)) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + (uint32_t)(acc * 2 * NT) + ((uint32_t)(quad * 32) << 16);
      uint16_t *ocol = P.out + (size_t)t_row * P.n_out + f;
#pragma unroll 1
      for (int c = 0; c < NT; c += 16) {
        float a[16], u[16];
        if (glu) {
          tmem_ld16x2(taddr + c, taddr + NT + c, a, u);
        } else {
          tmem_ld16(taddr + c, a);
        }
        if (!f_ok) continue;
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (c + j >= nvalid) break;
          float v;
          if (glu) {
            v = f8::silu(a[j] * s0) * (u[j] * s1);
          } else {
            v = a[j] * s0;
            if (relu) v = fmaxf(v, 0.f);
          }
          ocol[(size_t)(c + j) * P.n_out] = (uint16_t)(pack_bf16x2(v, 0.f) & 0xFFFFu);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (tile.phase == 0) {  // publish this warp's rows of h to the down tiles of the group
        __threadfence();
        __syncwarp();
        if (lane == 0) atomicAdd(&args.dep[tile.g], 1);
      }
    }
  }

  __syncthreads();
  if (warp == W_MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
}

}  // namespace f8s

namespace f8 {

// Per-row quantisation: one warp per row; s = max |w| / 448 (1 for a zero row),
// q = E4M3 (round to nearest even, saturating) of w / s.
__global__ void __launch_bounds__(256) quantize_rows_fp8_kernel(const uint16_t *__restrict__ w, int64_t rows, int cols,
                                                                uint8_t *__restrict__ q, float *__restrict__ scales) {
  const int lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (row >= rows) return;
  const uint16_t *wr = w + row * cols;
  float amax = 0.f;
  for (int c = lane; c < cols; c += 32) amax = fmaxf(amax, fabsf(__uint_as_float((uint32_t)wr[c] << 16)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  const float s = amax > 0.f ? amax / 448.0f : 1.0f;
  if (lane == 0) scales[row] = s;
  uint8_t *qr = q + row * cols;
  for (int c = lane; c < cols; c += 32) {
    const float v = __uint_as_float((uint32_t)wr[c] << 16) / s;
    qr[c] = (uint8_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
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

// bf16 [rows, cols], box 64 x 128, 128-byte swizzle (the A tile)
static int make_map_bf16(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16 || !rows || !cols) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {BK, BM};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// bf16 [rows, cols], box 64 x box_rows, 128-byte swizzle (the token tile of the decode kernel)
static int make_map_tokens(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (cols * 2) % 16 || !rows || !cols) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// E4M3 codes [rows, cols] bytes, box 64 x 128 with the 64-byte swizzle: the
// 16-byte chunk c of row r lands at chunk c ^ ((r >> 1) & 3) of its 64-byte row
// (the weight tile of the decode kernel)
static int make_map_u8_sw64(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || cols % 16 || !rows || !cols) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {64, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? MOE_OK
             : MOE_ERR_CUDA;
}

// E4M3 codes [rows, cols] bytes, box 64 x 128, no swizzle (the raw weight tile)
static int make_map_u8(CUtensorMap *m, const void *base, uint64_t rows, uint64_t cols) {
  EncodeTiledFn enc = get_encode();
  if (!enc) return MOE_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || cols % 16 || !rows || !cols) return MOE_ERR_UNSUPPORTED;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {BK, 128};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS
             ? MOE_OK
             : MOE_ERR_CUDA;
}

template <int MODE>
static int launch(const CUtensorMap &ma, const CUtensorMap &mq0, const CUtensorMap &mq1, const Args &args, int dev,
                  cudaStream_t stream) {
  static std::mutex mu;
  static std::vector<int> done;
  {
    std::lock_guard<std::mutex> lk(mu);
    if ((int)done.size() <= dev) done.resize(dev + 1, 0);
    if (!done[dev]) {
      if (cudaFuncSetAttribute(grouped_gemm_fp8_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)SMEM_BYTES) != cudaSuccess)
        return MOE_ERR_CUDA;
      done[dev] = 1;
    }
  }
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  grouped_gemm_fp8_kernel<MODE><<<sms, THREADS, SMEM_BYTES, stream>>>(ma, mq0, mq1, args);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

template <int NT>
static int launch_ffn_decode(const CUtensorMap &mx, const CUtensorMap &mh, const CUtensorMap &mq1,
                             const CUtensorMap &mq3, const CUtensorMap &mq2, const f8s::Args &args, int dev,
                             cudaStream_t stream) {
  static std::mutex mu;
  static std::vector<int> done;
  constexpr size_t smem = f8s::Shape<NT>::SMEM;
  {
    std::lock_guard<std::mutex> lk(mu);
    if ((int)done.size() <= dev) done.resize(dev + 1, 0);
    if (!done[dev]) {
      if (cudaFuncSetAttribute(f8s::fp8_ffn_decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess)
        return MOE_ERR_CUDA;
      done[dev] = 1;
    }
  }
  const int sms = device_sm_count(dev);
  if (sms <= 0) return MOE_ERR_CUDA;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f8s::fp8_ffn_decode_kernel<NT>, f8s::THREADS, smem) !=
          cudaSuccess ||
      per_sm < 1)
    return MOE_ERR_CUDA;
  // Cooperative: every CTA resident at once, since down tiles wait for gate/up tiles of other CTAs.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);
  cfg.blockDim = dim3(f8s::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, f8s::fp8_ffn_decode_kernel<NT>, mx, mh, mq1, mq3, mq2, args) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

template <int NT>
static int run_ffn_decode(int act, const void *x, const void *h, int64_t rows, int d, int F, const uint8_t *w1q,
                          const float *w1s, const uint8_t *w3q, const float *w3s, const uint8_t *w2q,
                          const float *w2s, const int32_t *offsets, int G, void *y, int *dep, int *status, int dev,
                          cudaStream_t stream) {
  CUtensorMap mx, mh, mq1, mq3, mq2;
  int rc;
  if ((rc = make_map_tokens(&mx, x, (uint64_t)rows, (uint64_t)d, NT))) return rc;
  if ((rc = make_map_tokens(&mh, h, (uint64_t)rows, (uint64_t)F, NT))) return rc;
  if ((rc = make_map_u8_sw64(&mq1, w1q, (uint64_t)G * F, (uint64_t)d))) return rc;
  if (act == kSwiGLU) {
    if ((rc = make_map_u8_sw64(&mq3, w3q, (uint64_t)G * F, (uint64_t)d))) return rc;
  } else {
    mq3 = mq1;
  }
  if ((rc = make_map_u8_sw64(&mq2, w2q, (uint64_t)G * d, (uint64_t)F))) return rc;
  const bool glu = act == kSwiGLU;
  f8s::Args args{};
  args.offsets = offsets;
  args.G = G;
  args.a_rows = (int32_t)rows;
  args.act = act;
  // phase 0: h = act(x W1^T [, x W3^T]); K = d in stages of 128 (two weights) or 256
  args.ph[0] = f8s::Phase{F, F, glu ? (d + 127) / 128 : (d + 255) / 256, glu ? 2 : 1, w1s, glu ? w3s : nullptr,
                          static_cast<uint16_t *>(const_cast<void *>(h))};
  // phase 1: y = h W2^T; K = F in stages of 256
  args.ph[1] = f8s::Phase{d, d, (F + 255) / 256, 1, w2s, nullptr, static_cast<uint16_t *>(y)};
  args.dep = dep;
  args.status = status;
  if (cudaMemsetAsync(dep, 0, (size_t)G * sizeof(int), stream) != cudaSuccess) return MOE_ERR_CUDA;
  return launch_ffn_decode<NT>(mx, mh, mq1, mq3, mq2, args, dev, stream);
}

}  // namespace f8

int tc_grouped_gemm_fp8(int mode, const void *A, int64_t a_rows, int K, const uint8_t *Q0, const float *S0,
                        const uint8_t *Q1, const float *S1, int64_t b_rows_total, int b_rows_per_group,
                        const int32_t *offsets, int G, int M, int n_out, void *out, int *status, cudaStream_t stream) {
  using namespace f8;
  if (G < 1 || G > MAX_GROUPS || K < 1 || n_out < 1 || a_rows < 1 || a_rows > INT32_MAX || b_rows_total < 1)
    return MOE_ERR_INVALID_ARG;
  if (mode < kSwiGLU || mode > kPlain || !Q0 || !S0 || (mode == kSwiGLU && (!Q1 || !S1)) ||
      n_out > b_rows_per_group || (int64_t)G * b_rows_per_group > b_rows_total || (n_out % 8))
    return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  CUtensorMap ma, mq0, mq1;
  int rc;
  if ((rc = make_map_bf16(&ma, A, (uint64_t)a_rows, (uint64_t)K))) return rc;
  if ((rc = make_map_u8(&mq0, Q0, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  if (mode == kSwiGLU) {
    if ((rc = make_map_u8(&mq1, Q1, (uint64_t)b_rows_total, (uint64_t)K))) return rc;
  } else {
    mq1 = mq0;
  }
  Args args{offsets, G, M, (int32_t)a_rows, n_out, b_rows_per_group, (K + BK - 1) / BK, S0, S1,
            static_cast<uint16_t *>(out), status};
  switch (mode) {
    case kSwiGLU: return launch<kSwiGLU>(ma, mq0, mq1, args, dev, stream);
    case kReLU: return launch<kReLU>(ma, mq0, mq1, args, dev, stream);
    default: return launch<kPlain>(ma, mq0, mq1, args, dev, stream);
  }
}

int tc_expert_ffn_fp8_decode(int act, const void *x_perm, void *h, int64_t rows, int d, int F, int max_group_rows,
                             const uint8_t *w1q, const float *w1s, const uint8_t *w3q, const float *w3s,
                             const uint8_t *w2q, const float *w2s, const int32_t *offsets, int G, void *y, int *dep,
                             int *status, cudaStream_t stream) {
  using namespace f8;
  if (G < 1 || G > f8s::MAX_GROUPS || rows < 1 || rows > INT32_MAX || d < 8 || F < 8 || (d % 8) || (F % 8) ||
      !offsets || !dep || !w1q || !w1s || !w2q || !w2s || (act == kSwiGLU && (!w3q || !w3s)) ||
      (act != kSwiGLU && act != kReLU))
    return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ERR_CUDA;
  switch (fp8_decode_tile_rows(max_group_rows)) {
    case 16:
      return run_ffn_decode<16>(act, x_perm, h, rows, d, F, w1q, w1s, w3q, w3s, w2q, w2s, offsets, G, y, dep, status,
                                dev, stream);
    case 32:
      return run_ffn_decode<32>(act, x_perm, h, rows, d, F, w1q, w1s, w3q, w3s, w2q, w2s, offsets, G, y, dep, status,
                                dev, stream);
    case 64:
      return run_ffn_decode<64>(act, x_perm, h, rows, d, F, w1q, w1s, w3q, w3s, w2q, w2s, offsets, G, y, dep, status,
                                dev, stream);
    default: return MOE_ERR_INVALID_ARG;
  }
}

int launch_quantize_fp8(const void *w, int64_t rows, int cols, uint8_t *q, float *scales, cudaStream_t s) {
  if (rows == 0) return MOE_OK;
  f8::quantize_rows_fp8_kernel<<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(static_cast<const uint16_t *>(w), rows,
                                                                           cols, q, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
