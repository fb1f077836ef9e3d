// moe_dispatch_noalloc: the dispatch stage for callers that can neither allocate
// device memory nor hand the library a workspace.
//
// Who needs it: code that runs as a plug-in or custom operator inside a host
// program that owns the device memory -- for example an inference server that
// reserves the GPU's memory for its own pool when it starts -- and whose calling
// interface passes only the operator's input and output buffers.  Such code may
// not call cudaMalloc (the memory is already spoken for, and an allocation in the
// middle of serving can fail or stall), and it has no workspace to pass to
// moe_dispatch.  This entry point takes the same inputs and outputs as
// moe_dispatch and keeps its scratch (per-chunk expert histograms and their
// running sums) in a fixed array that is part of the library itself.
//
// The array lives in device memory from the moment the library's code is loaded
// on a GPU until the process exits, on every GPU that loads it: 1 MiB per GPU.
#include <mutex>
#include <vector>

#include "moe_common.cuh"
#include "moe_internal.h"

namespace moe {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;  // 1 MiB
// the scratch holds two int32 tables of ceil(T / 128) x N entries each
constexpr int64_t kNoAllocMaxEntries = (int64_t)(kNoAllocScratchBytes / (2 * sizeof(int32_t)));

static __device__ __align__(256) int32_t g_dispatch_scratch[kNoAllocScratchBytes / sizeof(int32_t)];

// Device address of g_dispatch_scratch on each device, looked up once per device.
// In host code the name g_dispatch_scratch is only a host-side stand-in; the
// kernels must be given this address instead.
int32_t *scratch_on_current_device(int *rc) {
  static std::mutex mu;
  static std::vector<int32_t *> addr;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *rc = MOE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(mu);
  if ((int)addr.size() <= dev) addr.resize(dev + 1, nullptr);
  if (!addr[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_dispatch_scratch) != cudaSuccess || !p) {
      *rc = MOE_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = static_cast<int32_t *>(p);
  }
  *rc = MOE_OK;
  return addr[dev];
}

}  // namespace
}  // namespace moe

extern "C" MOE_API int moe_dispatch_noalloc(const moe_config *cfg, const int32_t *topk_idx, const void *x,
                                            int32_t *counts_routed, int32_t *counts_kept, int32_t *offsets,
                                            int32_t *dest_row, int32_t *src_token, void *x_perm, int32_t *status,
                                            void *stream) {
  using namespace moe;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  // the same shape limits as every other entry point
  size_t ws_bytes = 0;
  const int rc0 = moe_workspace_size(cfg, &ws_bytes);
  if (rc0) return rc0;
  // expert choice routes and dispatches in moe_ec_route; moe_dispatch refuses it too
  if (cfg->routing == MOE_ROUTING_EXPERT_CHOICE) return MOE_ERR_INVALID_ARG;
  if (!counts_routed || !counts_kept || !offsets) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!topk_idx || !x || !dest_row || !src_token || !x_perm ||
                     (reinterpret_cast<uintptr_t>(x) & 15) || (reinterpret_cast<uintptr_t>(x_perm) & 15)))
    return MOE_ERR_INVALID_ARG;
  const int64_t nchunks = ((int64_t)cfg->T + kDispatchChunk - 1) / kDispatchChunk;
  if (nchunks * cfg->N > kNoAllocMaxEntries) return MOE_ERR_UNSUPPORTED;  // beyond the fixed scratch
  int rc = MOE_OK;
  int32_t *scratch = scratch_on_current_device(&rc);
  if (rc) return rc;
  int32_t *hist = scratch;
  int32_t *chunk_base = scratch + nchunks * cfg->N;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = launch_dispatch(topk_idx, cfg->T, cfg->k, cfg->N, cfg->capacity, hist, chunk_base, counts_routed, counts_kept,
                       offsets, dest_row, src_token, reinterpret_cast<int *>(status), s);
  if (rc || cfg->T == 0) return rc;
  const int es = cfg->dtype == MOE_BF16 ? 2 : 4;
  return launch_scatter_rows(x, dest_row, cfg->T, cfg->k, cfg->d * es, x_perm, s);
}
