// Dispatch: stable counting sort of the routes by expert.
//
// RL-Kernel PR #557 "EP4 distributed logprob parity", section "What":
// dispatch is a local selection of the routes each expert owns; embedded
// #503 commit message, "Experts": every (token, route) row has one writer.
//
// Routes r = t*k + s are cut into chunks of CH consecutive routes (128, or
// 512 where the scratch must stay small), one warp per chunk.  (1) count: per-chunk expert histogram.  (2) scan_chunks:
// per expert, the exclusive prefix of the histogram over chunks, and the
// expert total.  (3) scan_experts: exclusive prefix of the totals = the
// segment offsets.  (4) scatter: each warp walks its chunk in ascending r;
// a route's position is offsets[e] + (routes of e in earlier chunks) +
// (routes of e earlier in this chunk), the last term from __match_any_sync
// and the lane order.  Integer arithmetic only, no atomics on positions: the
// result equals a sequential counting sort bit for bit, for any chunking.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int WARPS_PER_BLOCK = 4;
constexpr int PAST_END = -0x7fffffff - 1;  // lane past the last route (not an id)

size_t permute_scratch_bytes(int64_t R, int E, int chunk) {
  int64_t n_chunks = ceil_div(R, chunk);
  return (size_t)(n_chunks * E + E) * sizeof(int32_t);
}

template <int CH>
__global__ void __launch_bounds__(32 * WARPS_PER_BLOCK)
permute_count_kernel(int64_t R, int E, int n_chunks, const int32_t *__restrict__ ids, int32_t *__restrict__ counts,
                     int *status) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int32_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * WARPS_PER_BLOCK + warp;
  if (c >= n_chunks) return;
  constexpr int STEPS = CH / 32;  // 32 routes per step
  int32_t *hist = smem + warp * E;
  for (int i = lane; i < E; i += 32) hist[i] = 0;
  int eid[STEPS];  // all loads issued before the dependent match chain
#pragma unroll
  for (int step = 0; step < STEPS; ++step) {
    const int64_t r = (int64_t)c * CH + step * 32 + lane;
    eid[step] = r < R ? __ldg(ids + r) : PAST_END;
  }
  __syncwarp();
#pragma unroll
  for (int step = 0; step < STEPS; ++step) {
    int e = eid[step];
    if (e == PAST_END) {
      e = -1;
    } else if (e < 0 || e >= E) {
      record_status(status, STATUS_BAD_EXPERT_ID);
      e = -1;
    }
    unsigned peers = __match_any_sync(FULL_MASK, e);
    if (e >= 0 && lane == __ffs(peers) - 1) hist[e] += __popc(peers);
    __syncwarp();
  }
  int32_t *out = counts + (int64_t)c * E;
  for (int i = lane; i < E; i += 32) out[i] = hist[i];
}

// grid: ceil(E/32) blocks of 32 warps; lane = expert, warp = range of chunks.
__global__ void __launch_bounds__(1024)
permute_scan_chunks_kernel(int E, int n_chunks, int32_t *__restrict__ counts, int32_t *__restrict__ totals) {
  griddep_launch();
  griddep_wait();
  __shared__ int32_t part[32][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  const int cpw = (n_chunks + 31) / 32;
  const int c0 = warp * cpw, c1 = min(n_chunks, c0 + cpw);
  int32_t local = 0;
  if (e < E)
#pragma unroll 8
    for (int c = c0; c < c1; ++c) local += counts[(int64_t)c * E + e];
  part[warp][lane] = local;
  __syncthreads();
  if (warp == 0) {
    int32_t run = 0;
    for (int w = 0; w < 32; ++w) {
      int32_t v = part[w][lane];
      part[w][lane] = run;
      run += v;
    }
    if (e < E) totals[e] = run;
  }
  __syncthreads();
  if (e < E) {
    int32_t run = part[warp][lane];
#pragma unroll 8
    for (int c = c0; c < c1; ++c) {
      int32_t v = counts[(int64_t)c * E + e];
      counts[(int64_t)c * E + e] = run;
      run += v;
    }
  }
}

// One block of 1024 threads: offsets[e] = sum_{e' < e} totals[e'], offsets[E] = total.
__global__ void __launch_bounds__(1024)
permute_scan_experts_kernel(int E, const int32_t *__restrict__ totals, int32_t *__restrict__ offsets) {
  griddep_launch();
  griddep_wait();
  __shared__ int32_t buf[1024];
  const int i = threadIdx.x;
  int32_t v = i < E ? totals[i] : 0;
  buf[i] = v;
  __syncthreads();
  for (int d = 1; d < 1024; d <<= 1) {  // inclusive Hillis-Steele scan (integers: exact)
    int32_t add = i >= d ? buf[i - d] : 0;
    __syncthreads();
    buf[i] += add;
    __syncthreads();
  }
  if (i < E) offsets[i] = buf[i] - v;
  if (i == E - 1) offsets[E] = buf[i];
}

template <int CH>
__global__ void __launch_bounds__(32 * WARPS_PER_BLOCK)
permute_scatter_kernel(int64_t R, int E, int n_chunks, const int32_t *__restrict__ ids,
                       const int32_t *__restrict__ chunk_prefix, const int32_t *__restrict__ offsets,
                       int32_t *__restrict__ sorted_route, int32_t *__restrict__ route_pos) {
  griddep_launch();
  griddep_wait();
  extern __shared__ int32_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int c = blockIdx.x * WARPS_PER_BLOCK + warp;
  if (c >= n_chunks) return;
  int32_t *next = smem + warp * E;
  const int32_t *pre = chunk_prefix + (int64_t)c * E;
  for (int i = lane; i < E; i += 32) next[i] = offsets[i] + pre[i];
  __syncwarp();
  const unsigned lt = lanemask_lt();
  constexpr int STEPS = CH / 32;
  int eid[STEPS];
#pragma unroll
  for (int step = 0; step < STEPS; ++step) {
    const int64_t r = (int64_t)c * CH + step * 32 + lane;
    eid[step] = r < R ? __ldg(ids + r) : -1;
  }
#pragma unroll
  for (int step = 0; step < STEPS; ++step) {
    const int64_t r = (int64_t)c * CH + step * 32 + lane;
    int e = eid[step];
    if (e < 0 || e >= E) e = -1;
    unsigned peers = __match_any_sync(FULL_MASK, e);
    if (e >= 0) {
      int32_t pos = next[e] + __popc(peers & lt);
      sorted_route[pos] = (int32_t)r;
      route_pos[r] = pos;
    }
    __syncwarp();
    if (e >= 0 && lane == __ffs(peers) - 1) next[e] += __popc(peers);
    __syncwarp();
  }
}

template <int CH>
static cudaError_t run_permute(int64_t R, int E, const int32_t *ids, int32_t *offsets, int32_t *sorted_route,
                               int32_t *route_pos, void *scratch, int *status, cudaStream_t stream) {
  const int n_chunks = (int)ceil_div(R, CH);
  int32_t *counts = (int32_t *)scratch;
  int32_t *totals = counts + (int64_t)n_chunks * E;
  const size_t smem = (size_t)WARPS_PER_BLOCK * E * sizeof(int32_t);
  const unsigned blocks = (unsigned)ceil_div(n_chunks, WARPS_PER_BLOCK);
  cudaError_t err;
  if (n_chunks > 0) {
    err = launch_pdl(permute_count_kernel<CH>, dim3(blocks), dim3(32 * WARPS_PER_BLOCK), smem, stream, R, E, n_chunks,
                     ids, counts, status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(permute_scan_chunks_kernel, dim3((unsigned)ceil_div(E, 32)), dim3(1024), 0, stream, E, n_chunks,
                     counts, totals);
  } else {
    err = cudaMemsetAsync(totals, 0, sizeof(int32_t) * E, stream);
  }
  if (err != cudaSuccess) return err;
  err = launch_pdl(permute_scan_experts_kernel, dim3(1), dim3(1024), 0, stream, E, (const int32_t *)totals, offsets);
  if (err != cudaSuccess || n_chunks == 0) return err;
  return launch_pdl(permute_scatter_kernel<CH>, dim3(blocks), dim3(32 * WARPS_PER_BLOCK), smem, stream, R, E, n_chunks,
                    ids, (const int32_t *)counts, (const int32_t *)offsets, sorted_route, route_pos);
}

cudaError_t launch_permute(int64_t R, int E, const int32_t *ids, int32_t *offsets, int32_t *sorted_route,
                           int32_t *route_pos, void *scratch, int *status, cudaStream_t stream, int chunk) {
  if (chunk == PERMUTE_CHUNK_SMALL)
    return run_permute<PERMUTE_CHUNK_SMALL>(R, E, ids, offsets, sorted_route, route_pos, scratch, status, stream);
  if (chunk == PERMUTE_CHUNK_LARGE)
    return run_permute<PERMUTE_CHUNK_LARGE>(R, E, ids, offsets, sorted_route, route_pos, scratch, status, stream);
  return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Tile list of the grouped GEMMs: segment s in [0, E) holds the routes of
// expert s (offsets[s]..offsets[s+1]), segment E the T tokens of the shared
// expert.  tile_start[s] = sum_{s' < s} ceil(n_s' / bn), tile_start[E+1] =
// total, counting only the routed segments in [e_begin, e_end) and the
// shared one if `with_shared` (the others get no tiles).  One block; integer
// prefix, exact.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(1024)
build_tiles_kernel(int E, int T, int bn, const int32_t *__restrict__ offsets, int32_t *__restrict__ tile_start,
                   int e_begin, int e_end, int with_shared) {
  griddep_launch();
  griddep_wait();
  __shared__ int32_t buf[1024];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base <= E; base += 1024) {
    const int s = base + threadIdx.x;
    int32_t n = 0;
    if (s < E) n = (s >= e_begin && s < e_end) ? offsets[s + 1] - offsets[s] : 0;
    else if (s == E) n = with_shared ? T : 0;
    int32_t v = (n + bn - 1) / bn;
    buf[threadIdx.x] = v;
    __syncthreads();
    for (int d = 1; d < 1024; d <<= 1) {
      int32_t add = (int)threadIdx.x >= d ? buf[threadIdx.x - d] : 0;
      __syncthreads();
      buf[threadIdx.x] += add;
      __syncthreads();
    }
    if (s <= E) tile_start[s] = carry + buf[threadIdx.x] - v;
    if (s == E) tile_start[E + 1] = carry + buf[threadIdx.x];
    __syncthreads();
    if (threadIdx.x == 1023) carry += buf[1023];
    __syncthreads();
  }
}

cudaError_t launch_build_tiles(int E, int T, int bn, const int32_t *offsets, int32_t *tile_start,
                               cudaStream_t stream, int e_begin, int e_end, int with_shared) {
  if (e_end < 0) e_end = E;
  return launch_pdl(build_tiles_kernel, dim3(1), dim3(1024), 0, stream, E, T, bn, offsets, tile_start, e_begin, e_end,
                    with_shared);
}

}  // namespace moe
