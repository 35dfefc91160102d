// Tensor-core (tcgen05 / TMEM / TMA) GEMMs of the bf16 backward.
//
// RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503 commit
// message "Backward": the per-expert GEMMs write per-route input gradients
// into one dense buffer (summed per token in ascending expert order
// elsewhere) and produce per-expert weight gradients; "Results (4 x H100)",
// footnote 1: every reduction has a fixed order.  ROLL PR #502 "What this
// changes": one K partition, no atomic split-K accumulation.
//
// Input gradients (persistent kernel tc_dgrad_kernel, items = 256 weight
// features x up to 256 rows of one segment, like the forward):
//   DGRAD_DOWN     D[i, j] = sum_h Wdn[e][h, i] dYr[j, h]       (K = H)
//                  epilogue: the SwiGLU backward with the saved [g | u] of
//                  row j, dg = dh u silu'(g), du = dh silu(g) -> dGU[j] (bf16)
//   DGRAD_GATE_UP  D[h, j] = sum_f Wgu[e][f, h] dGU[j, f]       (K = 2I)
//                  epilogue: dXr[j, h] in FP32
// The weights are the M operand read MN-major straight from their storage
// layout (one 3-D TMA box per stage: 4 blocks of 64 features x 64 K rows);
// the gradient rows are the K-major N operand (TMA row boxes).
//
// Weight gradients (persistent kernel tc_wgrad_kernel, items = a 128 x 128
// output tile of one segment, K = the segment's rows in ascending order):
//   WGRAD_DOWN     dWdn[e][h, i] = sum_j dYr[j, h] h[j, i]
//   WGRAD_GATE_UP  dWgu[e][f, h] = sum_j dGU[j, f] x[tok(j), h]
// Both operands are MN-major (a row j of the activations is one K line);
// rows past the segment's end in its last K block are zeroed in shared
// memory before the MMAs read them.  Four TMEM accumulators rotate, so
// the epilogue of one tile overlaps the MMAs of the next ones; each epilogue warp
// copies its whole share of an accumulator into registers and releases it at
// once, then stages 32 x 32 FP32 sub-tiles in shared memory and writes them
// with TMA stores (L2 evict-first).  Empty segments get zero tiles (every
// output is written).
//
// Every output element is reduced over K in one fixed order (K blocks of
// 64, four K = 16 MMAs each); the tiling decides where a value is written,
// never the order of its sum.
#include <cuda.h>

#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "tc_host.h"
#include "umma.cuh"

namespace moe {

using namespace umma;

constexpr int DGRAD_DOWN = 1, DGRAD_GATE_UP = 2;
constexpr int WGRAD_DOWN = 1, WGRAD_GATE_UP = 2;

constexpr int GT_EPI_FIRST = 2;  // epilogue warps start at warp 2
constexpr uint32_t GT_TMEM_COLS = 512;

__device__ inline bool gt_warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(FULL_MASK, ok, 0) != 0;
}

// ===========================================================================
// Input gradients
// ===========================================================================
// MT = M tiles (128 weight features each) per item.  MT = 2: two
// accumulators of up to 256 columns fill TMEM (drained between items); MT = 1:
// two accumulator buffers alternate, so the epilogue of one item overlaps the
// mainloop of the next.
constexpr int DG_EPI_BYTES = 4096;
constexpr int DG_B_BYTES = 256 * 128;  // up to 256 rows x 64 K
template <int MT>
struct DgCfg {
  static constexpr int A_BYTES = MT * 2 * 8192;  // 2 MT blocks of 64 features x 64 K lines
  // The down dgrad's epilogue (the SwiGLU backward, with the saved g and u
  // loaded per 32 x 32 tile) paces it: 16 epilogue warps, one stage fewer.
  static constexpr int EPI_WARPS = MT == 1 ? 16 : 8;
  static constexpr int THREADS = 32 * (GT_EPI_FIRST + EPI_WARPS);
  static constexpr int STAGES = 3;
  static constexpr int NBUF = MT == 1 ? 2 : 1;
  static constexpr int SMEM = 1024 + STAGES * (A_BYTES + DG_B_BYTES) + EPI_WARPS * DG_EPI_BYTES + 256;
  static_assert(SMEM <= 232448, "dgrad shared memory");
  static_assert(NBUF * MT * 256 <= 512, "TMEM columns");
};

struct DgMaps {
  CUtensorMap a, a_sh;        // weights, MN-major boxes (64, 64, 4)
  CUtensorMap b[5], b_sh[5];  // gradient rows, box heights 256 .. 16
};

struct DgParams {
  int T, H, E, k, I, Is;
  int e0;  // first expert of the weight arrays (expert partition)
  const int32_t *item_start;
  const int4 *items;
  const __nv_bfloat16 *gu_routed, *gu_shared;  // DGRAD_DOWN: saved [g | u]
  __nv_bfloat16 *dgu_routed, *dgu_shared;      // DGRAD_DOWN: out [dg | du]
  float *dxr, *dxs;                            // DGRAD_GATE_UP: out
  int *status;
};

struct DgItem {
  int seg, f, rows, n, nk;
  int64_t row0;
};

// The shared segment's items (last in the table, the largest row tiles) first.
template <int MODE>
__device__ inline DgItem dg_item(int it, const DgParams &p) {
  const int routed = __ldg(p.item_start + p.E), total = __ldg(p.item_start + p.E + 1);
  const int n_sh = total - routed;
  const int4 d = __ldg(p.items + (it < n_sh ? routed + it : it - n_sh));
  DgItem r;
  r.seg = d.x;
  r.f = d.y;
  r.row0 = d.z;
  r.rows = d.w;
  r.n = (int)round_up(r.rows, 16);
  r.nk = (MODE == DGRAD_DOWN ? p.H : 2 * (r.seg == p.E ? p.Is : p.I)) / 64;
  return r;
}

template <int MODE, int MT>
__global__ void __launch_bounds__(DgCfg<MT>::THREADS, 1)
tc_dgrad_kernel(const __grid_constant__ DgMaps maps, const DgParams p) {
  constexpr int DG_STAGES = DgCfg<MT>::STAGES, DG_A_BYTES = DgCfg<MT>::A_BYTES, NBUF = DgCfg<MT>::NBUF;
  constexpr int DG_EPI_WARPS = DgCfg<MT>::EPI_WARPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sa = base;
  uint8_t *sb = sa + DG_STAGES * DG_A_BYTES;
  uint8_t *epi = sb + DG_STAGES * DG_B_BYTES;
  uint64_t *bars = (uint64_t *)(epi + DG_EPI_WARPS * DG_EPI_BYTES);
  uint64_t *full = bars, *empty = bars + DG_STAGES;
  uint64_t *tfull = bars + 2 * DG_STAGES, *tempty = tfull + NBUF, *mma_done = tempty + NBUF;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < DG_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * DG_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.a_sh);
  }
  if (warp == 1) tmem_alloc(tmem_slot, GT_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();
  griddep_wait();
  const int total = __ldg(p.item_start + p.E + 1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const DgItem im = dg_item<MODE>(it, p);
        const bool sh = im.seg == p.E;
        const uint32_t bytes = DG_A_BYTES + im.n * 128;
        // first weight row of this expert in the [E * rows, cols] view
        const int wrow = sh ? 0 : (im.seg - p.e0) * (MODE == DGRAD_DOWN ? p.H : 2 * p.I);
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_3d(sa + stage * DG_A_BYTES, sh ? &maps.a_sh : &maps.a, &full[stage], 0, wrow + kb * 64,
                      im.f * 2 * MT, pol_w);
          uint8_t *b_dst = sb + stage * DG_B_BYTES;
          const CUtensorMap *bm = sh ? maps.b_sh : maps.b;
          int r = 0;
#pragma unroll
          for (int h = 0; h < 5; ++h) {
            const int box = 256 >> h;
            while (im.n - r >= box) {
              tma_load_2d(b_dst + r * 128, &bm[h], &full[stage], kb * 64, (int)(im.row0 + r), pol_x);
              r += box;
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == DG_STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) {
        volatile int never = 0;
        for (int s = 0; s < DG_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, cnt = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const DgItem im = dg_item<MODE>(it, p);
        const int b = cnt % NBUF;
        if (!mbar_wait(&tempty[b], ((cnt / NBUF) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, im.n) | IDESC_A_MN;
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t bd = smem_desc_sw128(smem_u32(sb + stage * DG_B_BYTES));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint64_t ad = smem_desc_mn_sw128(smem_u32(sa + stage * DG_A_BYTES + mt * 16384), 8192);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 16: A +2048 bytes (MN-major), B +32 bytes (K-major)
              mma_bf16(tmem + (b * MT + mt) * 256, ad + 128 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          }
          mma_commit(&empty[stage]);
          if (++stage == DG_STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        mma_commit(&tfull[b]);
        ++cnt;
      }
      mma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter
    constexpr int CSTEP = 32 * (DG_EPI_WARPS / 4);
    const int cfirst = 32 * ((warp - GT_EPI_FIRST) >> 2);
    uint8_t *stg = epi + (warp - GT_EPI_FIRST) * DG_EPI_BYTES;
    uint32_t cnt = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
      const DgItem im = dg_item<MODE>(it, p);
      const bool sh = im.seg == p.E;
      const int b = cnt % NBUF;
      if (!gt_warp_wait(&tfull[b], (cnt / NBUF) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tq = tmem + b * MT * 256 + ((uint32_t)(q * 32) << 16);
      bool released = false;
      for (int c0 = cfirst; c0 < im.n; c0 += CSTEP) {
        float vt[MT][32];
        if (MT == 2) tmem_ld32x2(tq + c0, tq + 256 + c0, vt[0], vt[MT - 1]);
        else tmem_ld32(tq + c0, vt[0]);
        if (c0 + CSTEP >= im.n) {
          // The warp's last accumulator columns are in registers: the buffer
          // goes back to the MMA thread before the epilogue math.
          tc_fence_before();
          mbar_arrive(&tempty[b]);
          released = true;
        }
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
          const int f0 = im.f * 128 * MT + mt * 128 + q * 32;  // first feature of this warp's 32
          if (MODE == DGRAD_DOWN) {
            // Lane = feature i, column c = row j.  Stage the 32 x 32 tiles of g
            // and u of these rows (64 bytes per row each), compute dg, du in
            // place, write the rows back as [dg | du].
            const int Iseg = sh ? p.Is : p.I;
            const __nv_bfloat16 *gu = sh ? p.gu_shared : p.gu_routed;
            __nv_bfloat16 *dgu = sh ? p.dgu_shared : p.dgu_routed;
            __nv_bfloat16 *G = (__nv_bfloat16 *)stg, *U = G + 32 * 32;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = (lane >> 2) + 8 * i, ch = lane & 3;
              if (c0 + r < im.rows) {
                const __nv_bfloat16 *src = gu + (im.row0 + c0 + r) * 2 * Iseg + f0 + ch * 8;
                *(uint4 *)(G + r * 32 + ch * 8) = *(const uint4 *)src;
                *(uint4 *)(U + r * 32 + ch * 8) = *(const uint4 *)(src + Iseg);
              }
            }
            __syncwarp();
#pragma unroll
            for (int c = 0; c < 32; ++c) {
              const float g = __bfloat162float(G[c * 32 + lane]);
              const float u = __bfloat162float(U[c * 32 + lane]);
              const float s = sigmoid_f32(g);
              const float dh = vt[mt][c];
              G[c * 32 + lane] = __float2bfloat16_rn(dh * u * (s * (1.f + g * (1.f - s))));
              U[c * 32 + lane] = __float2bfloat16_rn(dh * (g * s));
            }
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int r = (lane >> 2) + 8 * i, ch = lane & 3;
              if (c0 + r < im.rows) {
                __nv_bfloat16 *dst = dgu + (im.row0 + c0 + r) * 2 * Iseg + f0 + ch * 8;
                *(uint4 *)dst = *(const uint4 *)(G + r * 32 + ch * 8);
                *(uint4 *)(dst + Iseg) = *(const uint4 *)(U + r * 32 + ch * 8);
              }
            }
            __syncwarp();
          } else {
            // Lane = hidden unit h, column c = row j: transpose through a
            // 32 x 32 FP32 tile, then 128-byte row segments of dXr.
            float *S = (float *)stg;
            float *out = sh ? p.dxs : p.dxr;
#pragma unroll
            for (int c = 0; c < 32; ++c) S[c * 32 + lane] = vt[mt][c];
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int r = (lane >> 3) + 4 * i, ch = lane & 7;
              if (c0 + r < im.rows)
                *(float4 *)(out + (im.row0 + c0 + r) * p.H + f0 + ch * 4) = *(const float4 *)(S + r * 32 + ch * 4);
            }
            __syncwarp();
          }
        }
      }
      if (!released) {
        tc_fence_before();
        mbar_arrive(&tempty[b]);
      }
      ++cnt;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, GT_TMEM_COLS);
}

// ===========================================================================
// Weight gradients
// ===========================================================================
// A stage holds one K block of both operands: A = 2 blocks (128 M) and B =
// WG_NBLK blocks (WG_N) of 64 MN elements, each block hb K lines of 128 bytes, where
// hb (64, 32 or 16) is the smallest box height that covers the rows left in
// the segment; the lines past the segment's end that the K = 16 MMAs read
// (at most 15 per block) are zeroed by a dedicated warp before the stage is
// released to the MMA thread.
// WG_EPI_WARPS epilogue warps (warps 2..), WG_EPI_WARPS / 4 per TMEM lane quarter, each
// draining WG_COLS of the WG_N accumulator columns through WG_NSTG staging tiles.
// WG_N output columns per tile (256 or 128): TMEM holds 512 / WG_N accumulators.
// 128 x 128 tiles with five operand stages: the gradient store stream paces
// these kernels and stalls whenever an accumulator waits for its operands,
// so the smaller stages let the loads run further ahead of it (T=4096
// backward 2.08 ms with 128 x 256 tiles and three stages, 2.02 with 128 x 128
// and four, 1.99 with five; more staging tiles per warp instead of stages,
// or sixteen epilogue warps, were slower).
constexpr int WG_N = 128, WG_STAGES = 5, WG_EPI_WARPS = 8, WG_NSTG = 2;
constexpr int WG_NBUF = 512 / WG_N, WG_NBLK = WG_N / 64;
constexpr int WG_COLS = 4 * WG_N / WG_EPI_WARPS;
constexpr int WG_A_BYTES = 2 * 8192;        // 128 M x 64 K lines, MN-major
constexpr int WG_B_BYTES = WG_NBLK * 8192;  // WG_N N x 64 K lines, MN-major
constexpr int WG_STG_BYTES = 4096;    // one 32 x 32 FP32 store tile
constexpr int WG_TAIL_WARP = GT_EPI_FIRST + WG_EPI_WARPS;  // zeroes segment tails, then releases the stage
// TMA tile store with an L2 cache policy (the weight gradients are written
// once and not read again by this layer: evict-first keeps the operand rows
// that the next tiles re-read in L2).
__device__ inline void tma_store_2d_hint(const CUtensorMap *m, const void *src, int c0, int c1, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%1, %2}], [%3], %4;" ::"l"(m),
               "r"(c0), "r"(c1), "r"(smem_u32(src)), "l"(pol)
               : "memory");
}
// Zero lines copied over a stage's segment tail (at most 15 lines of 128 bytes).
__device__ __align__(128) uint4 g_zero_lines[15 * 8];
constexpr int WG_THREADS = 32 * (WG_TAIL_WARP + 1);
constexpr int WG_SMEM = 1024 + WG_STAGES * (WG_A_BYTES + WG_B_BYTES) + WG_NSTG * WG_EPI_WARPS * WG_STG_BYTES + 256;
static_assert(WG_SMEM <= 232448, "wgrad shared memory");

struct WgMaps {
  CUtensorMap a[3], a_sh[3];  // A^T operand rows, boxes (64, hb, 2) for hb = 64, 32, 16
  CUtensorMap b[3], b_sh[3];  // B^T operand rows, boxes (64, hb, WG_NBLK)
  CUtensorMap out, out_sh;    // FP32 gradients, 32 x 32 boxes
};

struct WgParams {
  int T, H, E, k, I, Is;
  const int32_t *offsets;
  int tm_r, tn_r, tm_s, tn_s;  // output tiles per segment (M x N), routed and shared
  int e0;                      // first expert of the partition (its weight gradients start at index 0)
  int total;                   // tm_s * tn_s + (experts of the partition) * tm_r * tn_r
  int *status;
};

struct WgItem {
  int seg, mt, nt, rows, nk;
  int64_t r0;
};

// The shared segment's tiles come first (their K = T is the longest), then
// the routed segments in expert order; inside a segment, M tiles major.
__device__ inline WgItem wg_item(int it, const WgParams &p) {
  WgItem r;
  const int n_sh = p.tm_s * p.tn_s;
  int local;
  if (it < n_sh) {
    r.seg = p.E;
    local = it;
    r.mt = local / p.tn_s;
    r.nt = local % p.tn_s;
    r.r0 = 0;
    r.rows = p.T;
  } else {
    const int per = p.tm_r * p.tn_r;
    r.seg = p.e0 + (it - n_sh) / per;
    local = (it - n_sh) % per;
    r.mt = local / p.tn_r;
    r.nt = local % p.tn_r;
    r.r0 = __ldg(p.offsets + r.seg);
    r.rows = __ldg(p.offsets + r.seg + 1) - (int)r.r0;
  }
  r.nk = (int)ceil_div(r.rows, 64);
  return r;
}

// Box height index (0: 64, 1: 32, 2: 16 lines) for `valid` rows of a K block.
__device__ inline int wg_box(int valid) { return valid > 32 ? 0 : (valid > 16 ? 1 : 2); }

template <int MODE>
__global__ void __launch_bounds__(WG_THREADS, 1)
tc_wgrad_kernel(const __grid_constant__ WgMaps maps, const WgParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sa = base;
  uint8_t *sb = sa + WG_STAGES * WG_A_BYTES;
  uint8_t *stg_all = sb + WG_STAGES * WG_B_BYTES;
  uint64_t *bars = (uint64_t *)(stg_all + WG_NSTG * WG_EPI_WARPS * WG_STG_BYTES);
  uint64_t *full = bars, *empty = bars + WG_STAGES;
  uint64_t *tfull = bars + 2 * WG_STAGES, *tempty = tfull + WG_NBUF, *mma_done = tempty + WG_NBUF;
  uint64_t *ready = mma_done + 1;  // stage s landed and its tail lines are zero
  uint32_t *tmem_slot = (uint32_t *)(ready + WG_STAGES);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  fence_proxy_async_smem();
  if (threadIdx.x == 0) {
    for (int s = 0; s < WG_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&ready[s], 1);
    }
    for (int b = 0; b < WG_NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * WG_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a[0]);
    prefetch_tmap(&maps.b[0]);
    prefetch_tmap(&maps.out);
  }
  if (warp == 1) tmem_alloc(tmem_slot, GT_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();
  griddep_wait();

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // rows are read by every tile of their segment
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      WgItem nxt = wg_item(blockIdx.x, p);
      for (int it = blockIdx.x; it < p.total && ok; it += gridDim.x) {
        const WgItem im = nxt;
        if (it + (int)gridDim.x < p.total) nxt = wg_item(it + gridDim.x, p);  // loads overlap this item
        const bool sh = im.seg == p.E;
        for (int kb = 0; kb < im.nk; ++kb) {
          const int hi = wg_box(min(64, im.rows - kb * 64));
          const uint32_t bytes = (uint32_t)(WG_A_BYTES + WG_B_BYTES) >> hi;
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
          const int row = (int)im.r0 + kb * 64;
          tma_load_3d(sa + stage * WG_A_BYTES, sh ? &maps.a_sh[hi] : &maps.a[hi], &full[stage], 0, row, im.mt * 2, pol);
          tma_load_3d(sb + stage * WG_B_BYTES, sh ? &maps.b_sh[hi] : &maps.b[hi], &full[stage], 0, row, im.nt * WG_NBLK,
                      pol);
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == WG_STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) {
        volatile int never = 0;
        for (int s = 0; s < WG_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, cnt = 0;
      bool ok = true;
      const uint32_t idesc = idesc_bf16_f32(128, WG_N) | IDESC_A_MN | IDESC_B_MN;
      WgItem nxt = wg_item(blockIdx.x, p);
      for (int it = blockIdx.x; it < p.total && ok; it += gridDim.x) {
        const WgItem im = nxt;
        if (it + (int)gridDim.x < p.total) nxt = wg_item(it + gridDim.x, p);
        if (im.rows == 0) continue;
        const int b = cnt % WG_NBUF;
        if (!mbar_wait(&tempty[b], ((cnt / WG_NBUF) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&ready[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const int valid = min(64, im.rows - kb * 64);
          const uint32_t lbo = (uint32_t)(64 >> wg_box(valid)) * 128;  // stride between 64-element MN blocks
          const uint64_t ad = smem_desc_mn_sw128(smem_u32(sa + stage * WG_A_BYTES), lbo);
          const uint64_t bd = smem_desc_mn_sw128(smem_u32(sb + stage * WG_B_BYTES), lbo);
          const int nkk = (valid + 15) >> 4;
          for (int kk = 0; kk < nkk; ++kk)
            mma_bf16(tmem + b * WG_N, ad + 128 * kk, bd + 128 * kk, idesc, (kb | kk) != 0);
          mma_commit(&empty[stage]);
          if (++stage == WG_STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        mma_commit(&tfull[b]);
        ++cnt;
      }
      mma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else if (warp == WG_TAIL_WARP) {
    // ------------------------------------------------------------ stage tails
    // In a segment's last K block, lines [valid, 16 nkk) of each block hold
    // rows of the next segment (or TMA zero fill) and the K = 16 MMAs read
    // them: once the stage has landed, bulk copies from a zero buffer
    // overwrite them in both operands (6 blocks, at most 15 lines each; an
    // async-proxy write like the stage's own, so no proxy fence), completing
    // on ready[s]; other stages are released at once.
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;  // stages with zero copies in flight
      bool ok = true;
      WgItem nxt = wg_item(blockIdx.x, p);
      for (int it = blockIdx.x; it < p.total && ok; it += gridDim.x) {
        const WgItem im = nxt;
        if (it + (int)gridDim.x < p.total) nxt = wg_item(it + gridDim.x, p);
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          const int valid = min(64, im.rows - kb * 64);
          const int hb = 64 >> wg_box(valid);  // lines per block in this stage
          const uint32_t bytes = (uint32_t)(16 * ((valid + 15) >> 4) - valid) * 128;
          if (bytes) {
            mbar_arrive_expect_tx(&ready[stage], (2 + WG_NBLK) * bytes);
#pragma unroll
            for (int blk = 0; blk < 2 + WG_NBLK; ++blk) {
              uint8_t *blk_base = blk < 2 ? sa + stage * WG_A_BYTES + blk * hb * 128
                                          : sb + stage * WG_B_BYTES + (blk - 2) * hb * 128;
              bulk_load(blk_base + valid * 128, g_zero_lines, bytes, &ready[stage]);
            }
            issued |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          } else {
            mbar_arrive(&ready[stage]);
          }
          if (++stage == WG_STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) {
        // The zero copies in flight land before the CTA exits.
        volatile int never = 0;
        for (int s = 0; s < WG_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&ready[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp (q, part): TMEM lanes 32q.. (output rows), columns [WG_COLS part, +WG_COLS).
    const int q = warp & 3, half = (warp - GT_EPI_FIRST) >> 2;
    uint8_t *stg0 = stg_all + (warp - GT_EPI_FIRST) * WG_NSTG * WG_STG_BYTES;
    uint32_t cnt = 0, sbuf = 0;
    const int Mr = MODE == WGRAD_DOWN ? p.H : 2 * p.I;  // output rows per routed expert
    const uint64_t pol_out = policy_evict_first();  // gradient stores
    WgItem nxt = wg_item(blockIdx.x, p);
    for (int it = blockIdx.x; it < p.total; it += gridDim.x) {
      const WgItem im = nxt;
      if (it + (int)gridDim.x < p.total) nxt = wg_item(it + gridDim.x, p);
      const bool sh = im.seg == p.E;
      const CUtensorMap *om = sh ? &maps.out_sh : &maps.out;
      const int mrow = (sh ? 0 : (im.seg - p.e0) * Mr) + im.mt * 128 + q * 32;
      const int ncol = im.nt * WG_N + half * WG_COLS;
      constexpr int NCH = WG_COLS / 32;
      float v[NCH][32];
      if (im.rows == 0) {  // an empty segment's gradient tile is zero (no accumulator is used)
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc)
#pragma unroll
          for (int j = 0; j < 32; ++j) v[cc][j] = 0.f;
      } else {
        const int b = cnt % WG_NBUF;
        if (!gt_warp_wait(&tfull[b], (cnt / WG_NBUF) & 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t tb = tmem + b * WG_N + ((uint32_t)(q * 32) << 16) + half * WG_COLS;
        // The warp's whole share of the accumulator into registers, then the
        // buffer goes back to the MMA thread before any store is staged.
#pragma unroll
        for (int cc = 0; cc < NCH; cc += 2) tmem_ld32x2(tb + cc * 32, tb + (cc + 1) * 32, v[cc], v[cc + 1]);
        tc_fence_before();
        mbar_arrive(&tempty[b]);
        ++cnt;
      }
#pragma unroll
      for (int cc = 0; cc < NCH; ++cc) {
        uint8_t *stg = stg0 + sbuf * WG_STG_BYTES;
        if (lane == 0) bulk_wait_read<WG_NSTG - 1>();  // the last store from this buffer has read it
        __syncwarp();
        // Row `lane` of the 32 x 32 tile: 16-byte chunk j at (j ^ (lane % 8)), the 128-byte swizzle.
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *(float4 *)(stg + lane * 128 + ((j ^ (lane & 7)) << 4)) =
              make_float4(v[cc][4 * j], v[cc][4 * j + 1], v[cc][4 * j + 2], v[cc][4 * j + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          tma_store_2d_hint(om, stg, ncol + cc * 32, mrow, pol_out);
          bulk_commit();
        }
        if (++sbuf == WG_NSTG) sbuf = 0;
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, GT_TMEM_COLS);
}

// x rows in sorted (expert-segment) order: xs[j] = x[sorted_route[j] / k], one
// warp per row, 16 bytes per lane; only the rows of experts [e_begin, e_end).
__global__ void __launch_bounds__(256)
gather_sorted_rows_kernel(int64_t R, int H, int k, const int32_t *sorted_route, const int32_t *offsets, int e_begin,
                          int e_end, const __nv_bfloat16 *x, __nv_bfloat16 *xs) {
  griddep_launch();
  griddep_wait();
  const int64_t j = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (j >= R || j < __ldg(offsets + e_begin) || j >= __ldg(offsets + e_end)) return;
  const uint4 *src = (const uint4 *)(x + (int64_t)(__ldg(sorted_route + j) / k) * H);
  uint4 *dst = (uint4 *)(xs + j * H);
  for (int c = lane; c < H / 8; c += 32) dst[c] = __ldg(src + c);
}

// ===========================================================================
// Host side
// ===========================================================================
bool backward_tc_supported(int H, int I, int Is) { return H % 256 == 0 && I % 256 == 0 && Is % 256 == 0; }

// Down dgrad: items of one M tile (128 features of I); gate_up dgrad: items
// of two M tiles (256 hidden units).
size_t dgrad_tc_scratch_bytes(int T, int k, int E, int H, int I, int Is) {
  const size_t starts = (size_t)round_up((E + 2) * 4, 256);
  return 2 * starts + (size_t)round_up(tc_max_items(T, k, E, I / 128, Is / 128) * 16, 256) +
         (size_t)round_up(tc_max_items(T, k, E, H / 256, H / 256) * 16, 256);
}

template <int MODE, int MT>
static cudaError_t launch_dgrad(const DgMaps &m, const DgParams &p, int grid, cudaStream_t stream) {
  cudaError_t e = ensure_smem((const void *)tc_dgrad_kernel<MODE, MT>, DgCfg<MT>::SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(tc_dgrad_kernel<MODE, MT>, dim3(grid), dim3(DgCfg<MT>::THREADS), DgCfg<MT>::SMEM, stream, m, p);
}

cudaError_t launch_dgrad_tc(const BwArgs &a, void *scratch, int *status, cudaStream_t stream) {
  const size_t starts = (size_t)round_up((a.E + 2) * 4, 256);
  const int mi_dn = (int)tc_max_items(a.T, a.k, a.E, a.I / 128, a.Is / 128);
  const int mi_gu = (int)tc_max_items(a.T, a.k, a.E, a.H / 256, a.H / 256);
  uint8_t *w = (uint8_t *)scratch;
  int32_t *start_dn = (int32_t *)w;
  int32_t *start_gu = (int32_t *)(w + starts);
  int4 *items_dn = (int4 *)(w + 2 * starts);
  int4 *items_gu = (int4 *)(w + 2 * starts + round_up((int64_t)mi_dn * 16, 256));
  const int eb = a.e_begin, ee = a.e_end < 0 ? a.E : a.e_end;
  const int64_t nl = std::max(ee - eb, 1);  // expert rows of the weight maps (one when the partition is empty)
  cudaError_t e = launch_item_tables(a.E, a.T, a.I / 128, a.Is / 128, a.H / 256, a.H / 256, a.offsets, start_dn,
                                     start_gu, items_dn, items_gu, mi_dn, mi_gu, stream, eb, ee, 1);
  if (e != cudaSuccess) return e;
  const int64_t R = (int64_t)a.T * a.k;
  DgMaps md, mg;
  if (!map_col_blocks(&md.a, a.w_down, nl * a.H, a.I, 64, 2) ||
      !map_col_blocks(&md.a_sh, a.ws_down, a.H, a.Is, 64, 2) || !map_rows(md.b, a.dyr, R, a.H) ||
      !map_rows(md.b_sh, a.dys, a.T, a.H) ||
      !map_col_blocks(&mg.a, a.w_gate_up, nl * 2 * a.I, a.H, 64, 4) ||
      !map_col_blocks(&mg.a_sh, a.ws_gate_up, 2 * (int64_t)a.Is, a.H, 64, 4) ||
      !map_rows(mg.b, a.dgu_routed, R, 2 * (int64_t)a.I) || !map_rows(mg.b_sh, a.dgu_shared, a.T, 2 * (int64_t)a.Is))
    return cudaErrorInvalidValue;
  DgParams p = {};
  p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k; p.I = a.I; p.Is = a.Is;
  p.e0 = eb;
  p.gu_routed = (const __nv_bfloat16 *)a.gu_routed;
  p.gu_shared = (const __nv_bfloat16 *)a.gu_shared;
  p.dgu_routed = (__nv_bfloat16 *)a.dgu_routed;
  p.dgu_shared = (__nv_bfloat16 *)a.dgu_shared;
  p.dxr = a.dxr;
  p.dxs = a.dxs;
  p.status = status;
  const int grid = device_sms();
  p.item_start = start_dn;
  p.items = items_dn;
  if ((e = launch_dgrad<DGRAD_DOWN, 1>(md, p, grid, stream)) != cudaSuccess) return e;
  p.item_start = start_gu;
  p.items = items_gu;
  return launch_dgrad<DGRAD_GATE_UP, 2>(mg, p, grid, stream);
}

static bool wg_maps(CUtensorMap *m3, const void *ptr, int64_t rows, int64_t cols, uint32_t nblk) {
  for (int i = 0; i < 3; ++i)
    if (!map_col_blocks(&m3[i], ptr, rows, cols, 64u >> i, nblk)) return false;
  return true;
}

template <int MODE>
static cudaError_t launch_wgrad(const WgMaps &m, const WgParams &p, cudaStream_t stream) {
  cudaError_t e = ensure_smem((const void *)tc_wgrad_kernel<MODE>, WG_SMEM);
  if (e != cudaSuccess) return e;
  return launch_pdl(tc_wgrad_kernel<MODE>, dim3(std::min(p.total, device_sms())), dim3(WG_THREADS), WG_SMEM, stream, m,
                    p);
}

cudaError_t launch_wgrad_tc(const BwArgs &a, int *status, cudaStream_t stream) {
  const int64_t R = (int64_t)a.T * a.k;
  const int eb = a.e_begin, ee = a.e_end < 0 ? a.E : a.e_end;
  const int64_t nl = std::max(ee - eb, 1);  // expert rows of the output maps (one when the partition is empty)
  cudaError_t e0 = launch_pdl(gather_sorted_rows_kernel, dim3((unsigned)ceil_div(R, 8)), dim3(256), 0, stream, R, a.H,
                              a.k, a.sorted_route, a.offsets, eb, ee, (const __nv_bfloat16 *)a.x,
                              (__nv_bfloat16 *)a.x_sorted);
  if (e0 != cudaSuccess) return e0;
  WgMaps md, mg;
  if (!wg_maps(md.a, a.dyr, R, a.H, 2) || !wg_maps(md.a_sh, a.dys, a.T, a.H, 2) ||
      !wg_maps(md.b, a.h_routed, R, a.I, WG_NBLK) || !wg_maps(md.b_sh, a.h_shared, a.T, a.Is, WG_NBLK) ||
      !map_f32_tile(&md.out, a.dw_down, nl * a.H, a.I) || !map_f32_tile(&md.out_sh, a.dws_down, a.H, a.Is) ||
      !wg_maps(mg.a, a.dgu_routed, R, 2 * (int64_t)a.I, 2) || !wg_maps(mg.a_sh, a.dgu_shared, a.T, 2 * (int64_t)a.Is, 2) ||
      !wg_maps(mg.b, a.x_sorted, R, a.H, WG_NBLK) || !wg_maps(mg.b_sh, a.x, a.T, a.H, WG_NBLK) ||
      !map_f32_tile(&mg.out, a.dw_gate_up, nl * 2 * a.I, a.H) ||
      !map_f32_tile(&mg.out_sh, a.dws_gate_up, 2 * (int64_t)a.Is, a.H))
    return cudaErrorInvalidValue;
  WgParams p = {};
  p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k; p.I = a.I; p.Is = a.Is;
  p.offsets = a.offsets;
  p.status = status;
  p.e0 = eb;
  // down: M = H, N = I
  p.tm_r = a.H / 128; p.tn_r = a.I / WG_N; p.tm_s = a.H / 128; p.tn_s = a.Is / WG_N;
  p.total = p.tm_s * p.tn_s + (ee - eb) * p.tm_r * p.tn_r;
  cudaError_t e = launch_wgrad<WGRAD_DOWN>(md, p, stream);
  if (e != cudaSuccess) return e;
  // gate_up: M = 2I, N = H
  p.tm_r = 2 * a.I / 128; p.tn_r = a.H / WG_N; p.tm_s = 2 * a.Is / 128; p.tn_s = a.H / WG_N;
  p.total = p.tm_s * p.tn_s + (ee - eb) * p.tm_r * p.tn_r;
  return launch_wgrad<WGRAD_GATE_UP>(mg, p, stream);
}

}  // namespace moe
