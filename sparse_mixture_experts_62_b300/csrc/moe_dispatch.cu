// Dispatch: group the (token, slot) assignments by expert, apply the capacity
// limit in token order, and gather the token rows into the permuted buffer.
//
// "Lecture29" (CS25 lecture 29 notes), section "Top-k routing semantics": tokens
// are rearranged by expert, run, and restored to their order; section
// "Inference load balance": an expert takes at most C = ceil(alpha T k / E)
// assignments, the rest are dropped.  "Chapter 19: MoE" 19.6.1 and CS336
// lecture 4 section 10: a dropped assignment contributes nothing; the residual
// path (owned by the caller) carries the token on.
//
// Deterministic without ordered atomics:
//   1. per 128-token chunk, a histogram of expert ids (shared-memory counts);
//   2. one CTA scans the histograms: per-expert totals, kept = min(total, C),
//      offsets = exclusive scan of kept, and each chunk's starting rank;
//   3. per chunk, each assignment's rank among the expert's assignments in
//      token order = chunk start + earlier warps + earlier lanes (bit masks);
//   4. a gather copies x[src_token[row]] into x_perm[row] with 16-byte vectors.
#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr int CH = kDispatchChunk;  // tokens per chunk = threads per CTA
constexpr int CH_WARPS = CH / 32;

// A token picks an expert at most once.  A top-k input that lists expert e in
// slot j and in an earlier slot keeps only the earlier one: the repeat is neither
// counted nor given a row (dest_row = -1), so every counted assignment has a row.
__device__ __forceinline__ bool repeats_earlier_slot(const int (&ex)[8], int j, int e) {
  bool rep = false;
#pragma unroll
  for (int i = 0; i < 7; ++i) rep |= (i < j) && (ex[i] == e);
  return rep;
}

__global__ void __launch_bounds__(CH) dispatch_hist_kernel(const int32_t *__restrict__ idx, int T, int k, int N,
                                                           int32_t *__restrict__ hist, int *status) {
  __shared__ int cnt[256];
  for (int e = threadIdx.x; e < N; e += CH) cnt[e] = 0;
  __syncthreads();
  const int t = blockIdx.x * CH + threadIdx.x;
  if (t < T) {
    int ex[8];
    for (int j = 0; j < k; ++j) {
      const int e = idx[(size_t)t * k + j];
      ex[j] = e;
      if (e < 0 || e >= N) {
        set_status(status, MOE_ERR_BOUNDS);
        continue;
      }
      if (repeats_earlier_slot(ex, j, e)) {  // counted once; the rank kernel drops the repeat
        set_status(status, MOE_ERR_INVALID_ARG);
        continue;
      }
      atomicAdd(&cnt[e], 1);
    }
  }
  __syncthreads();
  // expert-major ([N][nchunks]): the scan reads each expert's chunk counts contiguously
  for (int e = threadIdx.x; e < N; e += CH) hist[(size_t)e * gridDim.x + blockIdx.x] = cnt[e];
}

// One CTA of 1024 threads: G = 1024 / 256 = 4 (or, for N <= 128, 1024 / N rounded
// down to a power of two, at most 32) adjacent threads per expert.  hist and
// chunk_base are expert-major ([N][nchunks]); the expert's G threads take G
// adjacent chunks at a time (one 32-byte sector per expert and load), eight such
// rows of chunks in flight, and each row's exclusive scan (shuffles over the G
// threads) plus the running total of the rows before gives each chunk's starting
// rank.  Then the capacity and the exclusive scan of the kept counts over the
// experts (warp scans).
constexpr int SCAN_THREADS = 1024;
constexpr int SCAN_ROWS = 8;
__global__ void __launch_bounds__(SCAN_THREADS) dispatch_scan_kernel(const int32_t *__restrict__ hist, int nchunks,
                                                                     int N, int G, int capacity,
                                                                     int32_t *__restrict__ chunk_base,
                                                                     int32_t *__restrict__ counts_routed,
                                                                     int32_t *__restrict__ counts_kept,
                                                                     int32_t *__restrict__ offsets) {
  __shared__ int kept_s[256];
  __shared__ int warp_tot[8];
  const int e = threadIdx.x / G, g = threadIdx.x % G;
  const bool live = e < N;
  const int32_t *he = hist + (size_t)(live ? e : 0) * nchunks;
  int32_t *cb = chunk_base + (size_t)(live ? e : 0) * nchunks;
  int total = 0;  // the expert's assignments in the rows of chunks done so far
  for (int r0 = 0; r0 * G < nchunks; r0 += SCAN_ROWS) {
    int v[SCAN_ROWS];
#pragma unroll
    for (int i = 0; i < SCAN_ROWS; ++i) {
      const int c = (r0 + i) * G + g;
      v[i] = (live && c < nchunks) ? he[c] : 0;
    }
#pragma unroll
    for (int i = 0; i < SCAN_ROWS; ++i) {
      if ((r0 + i) * G >= nchunks) break;  // the same for every lane
      int incl = v[i];
      for (int off = 1; off < G; off <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, incl, off, G);
        if (g >= off) incl += u;
      }
      const int c = (r0 + i) * G + g;
      if (live && c < nchunks) cb[c] = total + incl - v[i];
      total += __shfl_sync(0xffffffffu, incl, G - 1, G);
    }
  }
  if (threadIdx.x < 256) kept_s[threadIdx.x] = 0;
  __syncthreads();
  if (e < N && g == 0) {
    counts_routed[e] = total;
    const int kept = capacity > 0 ? min(total, capacity) : total;
    counts_kept[e] = kept;
    kept_s[e] = kept;
  }
  __syncthreads();
  // exclusive scan of kept over the (at most 256) experts: a scan per warp of 32,
  // then the eight warp totals
  const int t = threadIdx.x, lane = t & 31, w = t >> 5;
  int mine = 0, inc = 0;
  if (t < 256) {
    mine = kept_s[t];
    inc = mine;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, inc, off);
      if (lane >= off) inc += v;
    }
    if (lane == 31) warp_tot[w] = inc;
  }
  __syncthreads();
  if (t < 256) {
    int before = 0;
    for (int i = 0; i < w; ++i) before += warp_tot[i];
    inc += before;
    if (t < N) offsets[t] = inc - mine;
    if (t == N - 1) offsets[N] = inc;
  }
}

__global__ void __launch_bounds__(CH) dispatch_rank_kernel(const int32_t *__restrict__ idx, int T, int k, int N,
                                                           int capacity, const int32_t *__restrict__ chunk_base,
                                                           const int32_t *__restrict__ offsets,
                                                           int32_t *__restrict__ dest_row,
                                                           int32_t *__restrict__ src_token) {
  __shared__ uint32_t lanes_with[CH_WARPS][256];  // which lanes of the warp picked expert e
  __shared__ int warp_before[CH_WARPS][256];      // assignments to e in earlier warps of the chunk
  __shared__ int base_s[256];                     // this chunk's starting rank per expert
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int v = threadIdx.x; v < CH_WARPS * 256; v += CH) (&lanes_with[0][0])[v] = 0u;
  for (int e = threadIdx.x; e < N; e += CH) base_s[e] = chunk_base[(size_t)e * gridDim.x + blockIdx.x];
  __syncthreads();
  const int t = blockIdx.x * CH + threadIdx.x;
  int ex[8];
  for (int j = 0; j < k; ++j) {
    ex[j] = -1;
    if (t < T) {
      const int e = idx[(size_t)t * k + j];
      if (e >= 0 && e < N && !repeats_earlier_slot(ex, j, e)) {
        ex[j] = e;
        atomicOr(&lanes_with[warp][e], 1u << lane);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < N; e += CH) {
    int run = 0;
    for (int w = 0; w < CH_WARPS; ++w) {
      warp_before[w][e] = run;
      run += __popc(lanes_with[w][e]);
    }
  }
  __syncthreads();
  if (t >= T) return;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = ex[j];
    int row = -1;
    if (e >= 0) {
      const int rank = base_s[e] + warp_before[warp][e] +
                       __popc(lanes_with[warp][e] & lt_mask);
      if (capacity <= 0 || rank < capacity) {
        row = offsets[e] + rank;
        src_token[row] = t;
      }
    }
    dest_row[(size_t)t * k + j] = row;
  }
}

// T <= 128 (one chunk, e.g. decode): histogram, capacity, offsets and ranks in
// one CTA, the three steps above without the launches between them.
__global__ void __launch_bounds__(CH) dispatch_one_chunk_kernel(const int32_t *__restrict__ idx, int T, int k, int N,
                                                                int capacity, int32_t *__restrict__ counts_routed,
                                                                int32_t *__restrict__ counts_kept,
                                                                int32_t *__restrict__ offsets,
                                                                int32_t *__restrict__ dest_row,
                                                                int32_t *__restrict__ src_token, int *status) {
  __shared__ uint32_t lanes_with[CH_WARPS][256];  // which lanes of the warp picked expert e
  __shared__ int warp_before[CH_WARPS][256];      // assignments to e in earlier warps
  __shared__ int kept_s[256];                     // kept counts, then their inclusive scan
  __shared__ int off_s[256];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int v = threadIdx.x; v < CH_WARPS * 256; v += CH) (&lanes_with[0][0])[v] = 0u;
  __syncthreads();
  const int t = threadIdx.x;
  int ex[8];
  for (int j = 0; j < k; ++j) {
    ex[j] = -1;
    if (t < T) {
      const int e = idx[(size_t)t * k + j];
      if (e < 0 || e >= N) {
        set_status(status, MOE_ERR_BOUNDS);
      } else if (repeats_earlier_slot(ex, j, e)) {
        set_status(status, MOE_ERR_INVALID_ARG);
      } else {
        ex[j] = e;
        atomicOr(&lanes_with[warp][e], 1u << lane);
      }
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < 256; e += CH) {
    int run = 0;
    if (e < N)
      for (int w = 0; w < CH_WARPS; ++w) {
        warp_before[w][e] = run;
        run += __popc(lanes_with[w][e]);
      }
    const int kept = (e < N) ? (capacity > 0 ? min(run, capacity) : run) : 0;
    if (e < N) {
      counts_routed[e] = run;
      counts_kept[e] = kept;
    }
    kept_s[e] = kept;
    off_s[e] = kept;
  }
  __syncthreads();
  // inclusive scan of the kept counts over 256 entries, two per thread
  for (int off = 1; off < 256; off <<= 1) {
    const int a = threadIdx.x, b = threadIdx.x + CH;
    const int va = a >= off ? kept_s[a - off] : 0;
    const int vb = b >= off ? kept_s[b - off] : 0;
    __syncthreads();
    kept_s[a] += va;
    kept_s[b] += vb;
    __syncthreads();
  }
  for (int e = threadIdx.x; e < N; e += CH) {
    off_s[e] = kept_s[e] - off_s[e];  // exclusive
    offsets[e] = off_s[e];
  }
  if (threadIdx.x == 0) offsets[N] = kept_s[N - 1];
  __syncthreads();
  if (t >= T) return;
  const uint32_t lt_mask = (1u << lane) - 1u;
  for (int j = 0; j < k; ++j) {
    const int e = ex[j];
    int row = -1;
    if (e >= 0) {
      const int rank = warp_before[warp][e] + __popc(lanes_with[warp][e] & lt_mask);
      if (capacity <= 0 || rank < capacity) {
        row = off_s[e] + rank;
        src_token[row] = t;
      }
    }
    dest_row[(size_t)t * k + j] = row;
  }
}

// x_perm[row] = x[src_token[row]] for row < offsets[N]; one warp per row.  Each
// lane issues four 16-byte loads before their stores, so that enough bytes are in
// flight per SM to cover the memory latency.
__global__ void __launch_bounds__(256) gather_rows_kernel(const uint8_t *__restrict__ x,
                                                          const int32_t *__restrict__ src_token,
                                                          const int32_t *__restrict__ offsets_end, int row_bytes,
                                                          uint8_t *__restrict__ x_perm) {
  const int rows = *offsets_end;
  const int nvec = row_bytes / 16;
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int row = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); row < rows; row += warps_total) {
    const int t = src_token[row];
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * row_bytes);
    uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)row * row_bytes);
    for (int v0 = lane; v0 < nvec; v0 += 128) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) buf[u] = __ldg(src + v0 + 32 * u);
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = buf[u];
    }
  }
}

// Token choice: x_perm[dest_row[t, j]] = x[t] for every kept slot j; one warp per
// token, which reads its row of x once and writes it to each of its rows of x_perm
// (a row gather would read x once per slot, from far-apart places once x no longer
// fits in L2 beside the x_perm being written).
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint8_t *__restrict__ x,
                                                           const int32_t *__restrict__ dest_row, int T, int k,
                                                           int row_bytes, uint8_t *__restrict__ x_perm) {
  const int nvec = row_bytes / 16;
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps_total) {
    const int my_row = lane < k ? dest_row[(size_t)t * k + lane] : -1;
    const uint4 *src = reinterpret_cast<const uint4 *>(x + (size_t)t * row_bytes);
    for (int v0 = lane; v0 < nvec; v0 += 128) {
      uint4 buf[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v0 + 32 * u < nvec) buf[u] = __ldg(src + v0 + 32 * u);
      for (int j = 0; j < k; ++j) {
        const int row = __shfl_sync(0xffffffffu, my_row, j);
        if (row < 0) continue;
        uint4 *dst = reinterpret_cast<uint4 *>(x_perm + (size_t)row * row_bytes);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (v0 + 32 * u < nvec) dst[v0 + 32 * u] = buf[u];
      }
    }
  }
}

}  // namespace

int launch_dispatch(const int32_t *idx, int T, int k, int N, int capacity, int32_t *hist, int32_t *chunk_base,
                    int32_t *counts_routed, int32_t *counts_kept, int32_t *offsets, int32_t *dest_row,
                    int32_t *src_token, int *status, cudaStream_t s) {
  const int nchunks = (T + CH - 1) / CH;
  if (nchunks == 1) {
    dispatch_one_chunk_kernel<<<1, CH, 0, s>>>(idx, T, k, N, capacity, counts_routed, counts_kept, offsets, dest_row,
                                               src_token, status);
    return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  if (nchunks > 0) dispatch_hist_kernel<<<nchunks, CH, 0, s>>>(idx, T, k, N, hist, status);
  int G = 4;  // threads per expert: a power of two, G * 256 <= 1024 for N <= 256
  while (G < 32 && 2 * G * N <= SCAN_THREADS) G *= 2;
  dispatch_scan_kernel<<<1, SCAN_THREADS, 0, s>>>(hist, nchunks, N, G, capacity, chunk_base, counts_routed,
                                                  counts_kept, offsets);
  if (nchunks > 0)
    dispatch_rank_kernel<<<nchunks, CH, 0, s>>>(idx, T, k, N, capacity, chunk_base, offsets, dest_row, src_token);
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_gather_rows(const void *x, const int32_t *src_token, const int32_t *offsets_end, int64_t max_rows,
                       int row_bytes, void *x_perm, cudaStream_t s) {
  if (max_rows <= 0) return MOE_OK;
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = device_sm_count(dev);
  int64_t blocks = (max_rows + 7) / 8;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  gather_rows_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(x), src_token, offsets_end, row_bytes,
                                                  static_cast<uint8_t *>(x_perm));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int launch_scatter_rows(const void *x, const int32_t *dest_row, int T, int k, int row_bytes, void *x_perm,
                        cudaStream_t s) {
  if (T <= 0) return MOE_OK;
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = device_sm_count(dev);
  int64_t blocks = ((int64_t)T + 7) / 8;
  const int64_t cap = (int64_t)(sms > 0 ? sms : 148) * 8;
  if (blocks > cap) blocks = cap;
  scatter_rows_kernel<<<(int)blocks, 256, 0, s>>>(static_cast<const uint8_t *>(x), dest_row, T, k, row_bytes,
                                                   static_cast<uint8_t *>(x_perm));
  return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
