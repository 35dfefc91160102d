// Dispatch in one launch: the stable counting sort of the routes by expert
// on one cluster of sixteen CTAs.
//
// RL-Kernel PR #557 "EP4 distributed logprob parity", section "What":
// dispatch is a local selection of the routes each expert owns; embedded
// #503 commit message, "Experts": every (token, route) row has one writer.
//
// Same result as the four-kernel counting sort of permute.cu, bit for bit:
// a route's position is offsets[e] + (routes of e before it in ascending
// route order).  Here the phases that need all routes are separated by
// cluster barriers instead of kernel boundaries, and the per-chunk counts
// live in shared memory instead of global scratch:
//   1. CTA c takes routes [c P, (c+1) P), warp w of it a contiguous 1/32 of
//      those; each warp counts its routes per expert (warp histogram, by
//      shared-memory atomic increments: a count does not depend on their
//      order).
//   2. Per expert: exclusive prefix of the warp histograms inside the CTA,
//      CTA totals; after a cluster barrier every CTA reads the sixteen CTAs'
//      totals through distributed shared memory, forms the segment sizes,
//      their exclusive scan (the offsets) and the routes of each expert in
//      the CTAs before it.
//   3. Each warp walks its routes again in ascending order and writes
//      sorted_route / route_pos; ties inside a step of 32 routes are ranked
//      by __match_any_sync and the lane order.
//   4. Optionally, the item tables of the two forward grouped GEMMs (the
//      same tables item_tables_kernel and item_expand_kernel build).
// Integer arithmetic only, no atomics on positions.  Ids outside [0, E) are
// skipped and recorded in the device status word (code 1), as in permute.cu.
// Sixteen is a non-portable cluster size: where the device does not allow it
// (or the cluster does not fit), callers take the four-kernel sort.  The
// routes of the SMs of one cluster are the limit: at 81,920 routes this
// launch takes 11.4 us against 15.2 us for the four kernels back to back,
// eight CTAs took 16.5 us, and counting with __match_any_sync (as the
// four-kernel sort does) instead of atomics took 27 us on eight CTAs.
#include "common.cuh"
#include "kernels.h"
#include "tc_host.h"
#include "umma.cuh"

namespace moe {

using namespace umma;

constexpr int PC_CTAS = 16, PC_THREADS = 1024, PC_WARPS = PC_THREADS / 32, PC_UNROLL = 8;
constexpr int PC_MAX_E = 1024;
constexpr int64_t PC_MAX_R = int64_t(1) << 20;
constexpr int PC_PAST_END = -0x7fffffff - 1;  // lane past the warp's last route (not an id)

static size_t pc_smem_bytes(int E) { return (size_t)(PC_WARPS + 4) * E * sizeof(int32_t); }

__device__ inline int32_t ld_cluster_s32(uint32_t addr) {
  int32_t v;
  asm volatile("ld.shared::cluster.s32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

// Exclusive scan of one value per thread over the 1024 threads of the block
// (integers: exact); *total = the sum.  `buf` holds 33 ints.
__device__ inline int32_t block_exclusive_scan(int32_t v, int32_t *buf, int32_t *total) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int32_t inc = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const int32_t u = __shfl_up_sync(FULL_MASK, inc, d);
    if (lane >= d) inc += u;
  }
  if (lane == 31) buf[warp] = inc;
  __syncthreads();
  if (warp == 0) {
    int32_t w = buf[lane], wi = w;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const int32_t u = __shfl_up_sync(FULL_MASK, wi, d);
      if (lane >= d) wi += u;
    }
    buf[lane] = wi - w;  // exclusive prefix of the warp sums
    if (lane == 31) buf[32] = wi;
  }
  __syncthreads();
  *total = buf[32];
  return buf[warp] + inc - v;
}

__global__ void __launch_bounds__(PC_THREADS, 1)
permute_cluster_kernel(int64_t R, int E, const int32_t *__restrict__ ids, int32_t *__restrict__ offsets,
                       int32_t *__restrict__ sorted_route, int32_t *__restrict__ route_pos, int *status,
                       PermuteItems itab) {
  extern __shared__ int32_t sm[];
  int32_t *hist = sm;            // [PC_WARPS][E]: warp histograms, then their exclusive prefixes
  int32_t *tot = hist + PC_WARPS * E;  // [E] this CTA's routes per expert (read by the other CTAs)
  int32_t *base = tot + E;       // [E] position of this CTA's first route of expert e
  int32_t *cnt = base + E;       // [E] routes of expert e (segment sizes)
  int32_t *off = cnt + E;        // [E] offsets[e]
  __shared__ int32_t scan_buf[33];
  griddep_launch();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  for (int i = threadIdx.x; i < PC_WARPS * E; i += PC_THREADS) hist[i] = 0;
  const int64_t per_cta = round_up(ceil_div(R, PC_CTAS), (int64_t)32 * PC_WARPS);
  const int64_t per_warp = per_cta / PC_WARPS;  // a multiple of 32
  const int64_t r0 = (int64_t)rank * per_cta + warp * per_warp;
  const int64_t r1 = min(R, r0 + per_warp);
  int32_t *h = hist + warp * E;
  griddep_wait();
  __syncthreads();

  // 1. warp histograms
  for (int64_t b = r0; b < r1; b += 32 * PC_UNROLL) {
    int eid[PC_UNROLL];  // all loads issued before the counts
#pragma unroll
    for (int u = 0; u < PC_UNROLL; ++u) {
      const int64_t r = b + 32 * u + lane;
      eid[u] = r < r1 ? __ldg(ids + r) : PC_PAST_END;
    }
#pragma unroll
    for (int u = 0; u < PC_UNROLL; ++u) {
      int e = eid[u];
      if (e == PC_PAST_END) {
        e = -1;
      } else if (e < 0 || e >= E) {
        record_status(status, STATUS_BAD_EXPERT_ID);
        e = -1;
      }
      if (e >= 0) atomicAdd(&h[e], 1);
    }
  }
  __syncthreads();

  // 2. prefixes over the warps of this CTA, over the CTAs, over the experts
  const int e = threadIdx.x;  // E <= PC_THREADS: one expert per thread
  if (e < E) {
    int32_t run = 0;
    for (int w = 0; w < PC_WARPS; ++w) {
      const int32_t v = hist[w * E + e];
      hist[w * E + e] = run;
      run += v;
    }
    tot[e] = run;
  }
  cluster_sync();  // every CTA's totals are complete and visible to the cluster
  int32_t before = 0, all = 0;
  if (e < E) {
    for (uint32_t c = 0; c < PC_CTAS; ++c) {
      const int32_t v = c == rank ? tot[e] : ld_cluster_s32(mapa_shared(tot + e, c));
      if (c < rank) before += v;
      all += v;
    }
  }
  int32_t total;
  const int32_t o = block_exclusive_scan(e < E ? all : 0, scan_buf, &total);
  if (e < E) {
    base[e] = o + before;
    cnt[e] = all;
    off[e] = o;
    if (rank == 0) offsets[e] = o;
  }
  if (rank == 0 && e == 0) offsets[E] = total;
  cluster_sync();  // no CTA reads another CTA's shared memory after this point

  // 3. stable scatter
  const unsigned lt = lanemask_lt();
  for (int64_t b = r0; b < r1; b += 32 * PC_UNROLL) {
    int eid[PC_UNROLL];
#pragma unroll
    for (int u = 0; u < PC_UNROLL; ++u) {
      const int64_t r = b + 32 * u + lane;
      eid[u] = r < r1 ? __ldg(ids + r) : -1;
    }
#pragma unroll
    for (int u = 0; u < PC_UNROLL; ++u) {
      const int64_t r = b + 32 * u + lane;
      int x = eid[u];
      if (x < 0 || x >= E) x = -1;
      const unsigned peers = __match_any_sync(FULL_MASK, x);
      if (x >= 0) {
        const int32_t pos = base[x] + h[x] + __popc(peers & lt);
        sorted_route[pos] = (int32_t)r;
        route_pos[r] = pos;
      }
      __syncwarp();
      if (x >= 0 && lane == __ffs(peers) - 1) h[x] += __popc(peers);
      __syncwarp();
    }
  }

  // 4. item tables of the grouped GEMMs: segment s < E has ceil(n_s / 256)
  // row tiles, the shared segment ceil(T / 256); table x gets nf_x_r items
  // per routed row tile and nf_x_s per shared one, in segment order.
  if (itab.start_a == nullptr) return;
  const int32_t v = e < E ? (cnt[e] + 255) / 256 : 0;
  int32_t vtot;
  const int32_t bt = block_exclusive_scan(v, scan_buf, &vtot);  // row tiles before segment e
  if (e < E) tot[e] = bt;  // tot is free again (step 2's cluster barrier)
  const int32_t v_sh = (itab.T + 255) / 256;
  if (rank == 0) {
    if (e < E) {
      itab.start_a[e] = bt * itab.nf_a_r;
      itab.start_b[e] = bt * itab.nf_b_r;
    }
    if (e == 0) {
      itab.start_a[E] = vtot * itab.nf_a_r;
      itab.start_b[E] = vtot * itab.nf_b_r;
      itab.start_a[E + 1] = vtot * itab.nf_a_r + v_sh * itab.nf_a_s;
      itab.start_b[E + 1] = vtot * itab.nf_b_r + v_sh * itab.nf_b_s;
    }
  }
  __syncthreads();
  // Expansion: one warp per segment, segments dealt round-robin over the
  // cluster's warps.
  for (int sg = (int)rank * PC_WARPS + warp; sg <= E; sg += PC_CTAS * PC_WARPS) {
    const int n_s = sg == E ? itab.T : cnt[sg];
    if (n_s == 0) continue;
    const int row0 = sg == E ? 0 : off[sg];
    const int ntile = (n_s + 255) >> 8;
    const int rpt = ((n_s + ntile - 1) / ntile + 15) & ~15;
    const int tb = sg == E ? vtot : tot[sg];
    const int a0 = tb * itab.nf_a_r, na = ntile * (sg == E ? itab.nf_a_s : itab.nf_a_r);
    const int b0 = tb * itab.nf_b_r, nb = ntile * (sg == E ? itab.nf_b_s : itab.nf_b_r);
    for (int local = lane; local < max(na, nb); local += 32) {
      const int nt = local % ntile;
      const int4 item = make_int4(sg, local / ntile, row0 + nt * rpt, min(rpt, n_s - nt * rpt));
      if (local < na && a0 + local < itab.max_a) itab.items_a[a0 + local] = item;
      if (local < nb && b0 + local < itab.max_b) itab.items_b[b0 + local] = item;
    }
  }
}

// Whether the one-launch sort can run for this size on the current device
// (a cluster of sixteen 1024-thread CTAs with their shared memory must fit).
bool permute_cluster_ok(int64_t R, int E) {
  if (R > PC_MAX_R || E < 1 || E > PC_MAX_E) return false;
  static std::mutex mu;
  static int cache[64] = {};  // 0 unknown, 1 yes, -1 no
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  std::lock_guard<std::mutex> lock(mu);
  int &c = cache[dev & 63];
  if (c == 0) {
    const size_t smem = pc_smem_bytes(PC_MAX_E);
    c = -1;
    if (cudaFuncSetAttribute((const void *)permute_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) == cudaSuccess &&
        cudaFuncSetAttribute((const void *)permute_cluster_kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
            cudaSuccess) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(PC_CTAS);
      cfg.blockDim = dim3(PC_THREADS);
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute at[1];
      at[0].id = cudaLaunchAttributeClusterDimension;
      at[0].val.clusterDim.x = PC_CTAS;
      at[0].val.clusterDim.y = 1;
      at[0].val.clusterDim.z = 1;
      cfg.attrs = at;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, (const void *)permute_cluster_kernel, &cfg) == cudaSuccess && n > 0)
        c = 1;
    }
    cudaGetLastError();
  }
  return c > 0;
}

cudaError_t launch_permute_cluster(int64_t R, int E, const int32_t *ids, int32_t *offsets, int32_t *sorted_route,
                                   int32_t *route_pos, int *status, cudaStream_t stream, const PermuteItems *items) {
  if (!permute_cluster_ok(R, E)) return cudaErrorInvalidConfiguration;
  PermuteItems it = {};
  if (items) it = *items;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(PC_CTAS);
  cfg.blockDim = dim3(PC_THREADS);
  cfg.dynamicSmemBytes = pc_smem_bytes(E);
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = PC_CTAS;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, permute_cluster_kernel, R, E, ids, offsets, sorted_route, route_pos, status, it);
}

}  // namespace moe
