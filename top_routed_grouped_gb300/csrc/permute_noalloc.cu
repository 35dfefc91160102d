// moe_permute_noalloc: the dispatch permutation for callers that cannot
// allocate device memory.
//
// Some callers of this library are handed only their input and output
// buffers: a custom operator or plugin hosted by another runtime that owns
// the whole device memory pool, or a latency-critical loop that must not call
// cudaMalloc because it can synchronise the device.  They cannot provide the
// workspace moe_permute needs.  This entry point runs the same permutation:
// as the one-launch cluster sort where that runs (it needs no scratch), else
// as the four-kernel sort with its scratch (the per-chunk expert histogram
// and the expert totals) in a fixed-size array in the library's own device
// memory.
//
// The array below is a file-scope __device__ object: every GPU that loads the
// library holds MOE_PERMUTE_NOALLOC_SCRATCH_BYTES of it until the process
// exits.  In host code its name is only a host-side stand-in; the device
// address is obtained once per device with cudaGetSymbolAddress (on the
// first call made with that device current) and cached.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

static __device__ __align__(256) int32_t g_permute_scratch[MOE_PERMUTE_NOALLOC_SCRATCH_BYTES / sizeof(int32_t)];

// Device address of g_permute_scratch on the current device (nullptr on a
// CUDA error).  First use per device does the lookup; later calls read the cache.
static int32_t *permute_scratch_device_ptr() {
  static std::mutex mu;
  static int32_t *cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    int32_t *ptr = nullptr;
    if (cudaGetSymbolAddress((void **)&ptr, g_permute_scratch) != cudaSuccess) return nullptr;
    cache[dev] = ptr;
  }
  return cache[dev];
}

}  // namespace moe

using namespace moe;

MOE_API int moe_permute_noalloc(const moe_dims_t *d, const int32_t *topk_ids, int32_t *expert_offsets,
                                int32_t *sorted_route, int32_t *route_pos, void *stream) {
  // The same argument checks as moe_permute (dims and buffers; there is no workspace).
  int st = permute_args_check(d, topk_ids, expert_offsets, sorted_route, route_pos);
  if (st != MOE_OK) return st;
  const int64_t R = (int64_t)d->T * d->k;
  if (permute_cluster_ok(R, d->E))  // the one-launch sort keeps its counts in shared memory: no scratch at all
    return launch_permute_cluster(R, d->E, topk_ids, expert_offsets, sorted_route, route_pos, device_status_ptr(),
                                  (cudaStream_t)stream) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  // The four-kernel sort over the fixed array: the default chunk where its
  // scratch fits, else the large chunk (same result); sizes that fit neither
  // are refused before any GPU work.
  int chunk = PERMUTE_CHUNK_SMALL;
  if (permute_scratch_bytes(R, d->E, chunk) > MOE_PERMUTE_NOALLOC_SCRATCH_BYTES) chunk = PERMUTE_CHUNK_LARGE;
  if (permute_scratch_bytes(R, d->E, chunk) > MOE_PERMUTE_NOALLOC_SCRATCH_BYTES) return MOE_ERR_UNSUPPORTED;
  int32_t *scratch = permute_scratch_device_ptr();
  if (!scratch) return MOE_ERR_CUDA;
  // Every scratch word the kernels read is written earlier by the same call,
  // so the previous call's contents never leak into this one.
  cudaError_t e = launch_permute(R, d->E, topk_ids, expert_offsets, sorted_route, route_pos, scratch,
                                 device_status_ptr(), (cudaStream_t)stream, chunk);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
