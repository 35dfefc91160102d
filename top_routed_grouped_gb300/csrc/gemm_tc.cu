// Tensor-core (tcgen05 / TMEM / TMA) GEMMs of the bf16 path.
//
// RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503 commit
// message: "Routing" (FP32 router through a batch-invariant GEMM) and
// "Experts" (per-route gate_up and down projections through one
// fixed-configuration grouped GEMM, no routed-weight multiply, one writer per
// (token, route) row).  ROLL PR #502 "What this changes": a single K
// partition, no atomic split-K accumulation.
//
// One persistent kernel skeleton, three uses (MODE):
//   ROUTER   D[e, t] = sum_k Wr3[e, k] x[t, k mod H], k < 3H, where Wr3 holds
//            the exact three-way bf16 split of the FP32 router weight
//            (Wr = W1 + W2 + W3, every product exact).  The K range is cut
//            into four fixed chunks accumulated in separate TMEM columns and
//            summed in FP32 in chunk order (four times fewer accumulation
//            steps per accumulator); epilogue adds the bias, writes logits.
//   GATE_UP  D[f, j] = W_gu[e][f] . x[tok(j)] for the gate and up rows of 128
//            features (two M tiles of 64 gate + 64 up rows) and up to 256 rows
//            j of expert e's segment; the x rows are gathered by eight warps
//            with 16-byte cp.async into the swizzled operand layout; epilogue
//            h = silu(g) * u.
//   DOWN     D[o, j] = W_dn[e][o] . h[j] for 128 output features (one M
//            tile, two accumulator buffers); epilogue writes row j to
//            y_routed[sorted_route[j]] (or y_shared).
// GATE_UP and DOWN also run on CTA pairs (tc_pair_kernel below, the form
// used wherever the device and the shapes allow): the same items, one
// M = 256 MMA over two SMs.  So does the router (tc_router_pair_kernel, two
// 128-expert tiles per pair item, where E is a multiple of 256).
// The weights are the M operand (128-row tiles) and the tokens the N <= 256 operand,
// so a short expert segment costs at most 15 padded columns.  Every output
// element is accumulated over K in a fixed order (K blocks of 64, four
// K = 16 MMAs each, fixed chunking); tiling decides only where a column
// sits, never the order, so a token's values do not depend on T or on its
// segment.
//
// Roles: warp 0 issues TMA loads (one instruction per weight tile, at most a
// few power-of-two row boxes for a contiguous token tile) into a stage ring;
// warp 1 allocates the 512 TMEM columns and one thread issues the MMAs; the
// epilogue warps from warp 2 on drain the accumulators (each TMEM lane
// quarter shared by several warps taking column chunks in turn), staging rows
// in shared memory so that global stores write contiguous row segments;
// GATE_UP adds eight warps that gather the token rows.
#include <cuda.h>

#include <algorithm>
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "tc_host.h"
#include "umma.cuh"

namespace moe {

using namespace umma;

// Per-mode configuration.  GATE_UP and DOWN give each item two M tiles (256
// weight rows) that share one token tile, so every gathered / loaded token
// row feeds twice the tensor-core work; the two accumulators take the whole
// 512 TMEM columns (one accumulator set, drained between items).  ROUTER keeps
// one M tile and uses the 512 columns as four K-chunk accumulators.
template <int MODE>
struct TcCfg;
constexpr int TC_GATE_UP = 1, TC_DOWN = 2;
// EPI_WARPS epilogue warps (a multiple of 4: EPI_WARPS / 4 warps per TMEM
// lane quarter split the columns); EPI_BYTES of row staging per warp.
template <>
struct TcCfg<1> {
  static constexpr int NMAX = 256, MT = 2, STAGES = 3, EPI_WARPS = 8, EPI_BYTES = 2560;
};
template <>
struct TcCfg<2> {
  static constexpr int NMAX = 256, MT = 1, STAGES = 4, EPI_WARPS = 16, EPI_BYTES = 2048;
};
// MT = 1: two accumulator buffers of 256 columns alternate between items, so
// an item's epilogue overlaps the next item's mainloop.  MT = 2: the two M
// tiles' accumulators fill TMEM and are drained between items.
template <int MODE>
constexpr int tc_nbuf() {
  return TcCfg<MODE>::MT == 1 ? 2 : 1;
}

constexpr int TC_TILE_A_BYTES = 128 * 128;  // one M tile: 128 rows x 64 bf16
constexpr int TC_B_BYTES = 256 * 128;       // up to 256 token rows x 64 bf16
constexpr int TC_EPI_FIRST = 2;             // epilogue warps start at warp 2
constexpr int TC_GATHER_WARPS = 8;          // GATE_UP row gather, after the epilogue warps
constexpr int TC_TOK_INTS = 256;            // gathered-row token ids (8 warps x 32)
constexpr int TC_MAX_STAGES = 4;
constexpr int TC_EPI_MAX_BYTES = 32768;     // largest EPI_WARPS * EPI_BYTES
constexpr int TC_SMEM_BYTES = 1024 + 4 * (TC_TILE_A_BYTES + TC_B_BYTES) + TC_EPI_MAX_BYTES + TC_TOK_INTS * 4 +
                              256;  // the largest of the three layouts
static_assert(3 * (2 * TC_TILE_A_BYTES + TC_B_BYTES) <= 4 * (TC_TILE_A_BYTES + TC_B_BYTES), "stage ring");
constexpr uint32_t TC_TMEM_COLS = 512;
constexpr int GATHER_THREADS = 32 * TC_GATHER_WARPS;

template <int MODE>
constexpr int tc_gather_first() {
  return TC_EPI_FIRST + TcCfg<MODE>::EPI_WARPS;
}
template <int MODE>
constexpr int tc_threads() {
  return 32 * (tc_gather_first<MODE>() + (MODE == TC_GATE_UP ? TC_GATHER_WARPS : 0));
}

// Tensor maps.  b[h] / b_sh[h] are the token-tile maps with box height 256 >> h.
struct TcMaps {
  CUtensorMap a, a_sh;
  CUtensorMap b[5];
  CUtensorMap b_sh[5];
};

struct TcParams {
  int T, H, E, k, I, Is;
  int n_items;              // ROUTER: number of items (others: item_start[E+1])
  int rt_ntile, rt_rpt;     // ROUTER: token tiles and rows per tile
  int rt_splits;            // ROUTER: bf16 terms of the weight used (3: exact; 1: weight rounded to bf16)
  int rt_kparts;            // ROUTER (pair form): RT_CHUNKS = one item per K chunk, partials to rt_partial; else 1
  float *rt_partial;        // ROUTER: [RT_CHUNKS][T][E] per-chunk logit sums when rt_kparts == RT_CHUNKS
  int e0;                   // first expert of the weight arrays (expert partition)
  int y_sorted;             // DOWN: routed rows in sorted order
  int y_f32;                // DOWN: float rows, the accumulators unrounded
  const int32_t *offsets;
  const int32_t *sorted_route;
  const int32_t *item_start;  // [E+2] prefix of items per segment
  const int4 *items;          // per item: segment, M-tile pair, first row, rows
  const __nv_bfloat16 *x;
  const float *bias;
  float *logits;
  __nv_bfloat16 *h_routed, *h_shared;
  __nv_bfloat16 *gu_routed, *gu_shared;
  __nv_bfloat16 *y_routed, *y_shared;
  int *status;
};

struct Item {
  int seg;       // expert segment (E = shared); ROUTER: unused
  int f;         // ROUTER: expert tile; GATE_UP / DOWN: pair of M tiles
  int64_t row0;  // first row of the N tile (token for ROUTER / shared, sorted row otherwise)
  int rows;      // valid rows in the tile
  int n;         // MMA N = rows rounded up to 16
  int nk;        // K blocks of 64
};

// Item `it` of the persistent loop.  The shared segment's items (the last
// ones of the table; its row tiles are the largest) are taken first, so the
// heaviest items do not form the tail of the launch.
__device__ inline int item_slot(int it, const int32_t *item_start, int E) {
  const int routed = __ldg(item_start + E), total = __ldg(item_start + E + 1);
  const int n_sh = total - routed;
  return it < n_sh ? routed + it : it - n_sh;
}

template <int MODE>
__device__ inline Item decode_item(int it, const TcParams &p) {
  Item r;
  const int4 d = __ldg(p.items + item_slot(it, p.item_start, p.E));
  r.seg = d.x;
  r.f = d.y;
  r.row0 = d.z;
  r.rows = d.w;
  r.nk = (MODE == TC_GATE_UP ? p.H : (r.seg == p.E ? p.Is : p.I)) / 64;
  r.n = (int)round_up(r.rows, 16);
  return r;
}

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ inline bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(FULL_MASK, ok, 0) != 0;
}

// Gate_up epilogue of one 32-column chunk (columns c0..c0+31 = rows of the
// item) of one M tile: v holds this lane's 32 accumulator values; the warp's
// 32 TMEM lanes are 16 gate rows then the 16 up rows of features fcol..+15.
// Writes h (and, if guout, the [g | u] rows) through the warp's staging
// buffer `stg` (2560 bytes).
__device__ __forceinline__ void gate_up_epi_chunk(const float (&v)[32], int fcol, int c0, const Item &im, int Iseg,
                                                  __nv_bfloat16 *hout, __nv_bfloat16 *guout, uint8_t *stg, int lane) {
  // The h and the g/u staging share the warp's buffer, one after the other.
  uint32_t *stg_h = (uint32_t *)stg;              // [32 cols][12 words] (8 used: 16 bf16)
  __nv_bfloat16 *stg_gu = (__nv_bfloat16 *)stg;  // [32 cols][40] (32 used)
  const int fl = lane & 15;
  const int cbase = lane < 16 ? 0 : 16;
  const bool odd = lane & 1;
  // Lane i < 16 holds gate g of feature i, lane i + 16 the up value u of
  // the same feature, for columns c0..c0+31.  One exchange gives lane i
  // the u of columns 0-15 and lane i + 16 the g of columns 16-31, so
  // both halves compute h for 16 columns each.
  float hv[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float send = lane < 16 ? v[16 + j] : v[j];
    const float recv = __shfl_xor_sync(FULL_MASK, send, 16);
    const float g = lane < 16 ? v[j] : recv;
    const float u = lane < 16 ? recv : v[16 + j];
    hv[j] = __fdividef(g, 1.0f + __expf(-g)) * u;
  }
  // Pack features (2m, 2m+1) of a column into one bf16x2 word: for the
  // column pair (j, j+1) the even lane writes column j, the odd lane
  // column j+1, after swapping one value with its neighbour.
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const float x = __shfl_xor_sync(FULL_MASK, odd ? hv[j] : hv[j + 1], 1);
    const __nv_bfloat162 w2 = odd ? __floats2bfloat162_rn(x, hv[j + 1]) : __floats2bfloat162_rn(hv[j], x);
    stg_h[(cbase + j + (odd ? 1 : 0)) * 12 + (fl >> 1)] = *reinterpret_cast<const uint32_t *>(&w2);
  }
  __syncwarp();
  // Two lanes per column row: 16 rows x 32 contiguous bytes per store
  // instruction.  h and the saved g/u are read only by later launches (the
  // down GEMM, the backward), by which time they have left L2 anyway, so
  // they are stored evict-first (st.global.cs): L2 keeps the weight tiles
  // and x rows that the running pairs share (T = 8192 forward -5 µs,
  // T = 4096 -4.5 µs).
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = (lane >> 1) + 16 * i, cc = lane & 1;
    if (c0 + r < im.rows) {
      const int64_t row = im.row0 + c0 + r;
      __stcs((uint4 *)(hout + row * Iseg + fcol + cc * 8), *(const uint4 *)(stg_h + r * 12 + cc * 4));
    }
  }
  __syncwarp();
  if (guout) {
#pragma unroll
    for (int j = 0; j < 32; ++j) stg_gu[j * 40 + lane] = __float2bfloat16_rn(v[j]);
    __syncwarp();
    if (c0 + lane < im.rows) {
      const int64_t row = im.row0 + c0 + lane;
      const uint4 *sg = (const uint4 *)(stg_gu + lane * 40);
      uint4 *dg = (uint4 *)(guout + row * 2 * Iseg + fcol);
      uint4 *du = (uint4 *)(guout + row * 2 * Iseg + Iseg + fcol);
      __stcs(dg, sg[0]);
      __stcs(dg + 1, sg[1]);
      __stcs(du, sg[2]);
      __stcs(du + 1, sg[3]);
    }
    __syncwarp();
  }
}

// Down epilogue of one 32-column chunk (columns c0..c0+31 = rows of the
// item): v holds this lane's 32 accumulator values, lane = output feature
// ocol + lane; `dst` (lane j: the destination row of column c0 + j) comes
// from the caller.  Writes bf16 rows of yout [*, H] through the warp's
// staging buffer `stg` (2048 bytes).
__device__ __forceinline__ void down_epi_chunk(const float (&v)[32], int ocol, int c0, int dst, const Item &im,
                                               __nv_bfloat16 *yout, int H, uint8_t *stg, int lane) {
  // [32 cols][16 words]: two consecutive rows span all 32 banks, so the
  // pair writes and the quarter-warp 16-byte reads are conflict-free.
  uint32_t *stg_y = (uint32_t *)stg;
  const bool odd = lane & 1;
  // Pack features (2m, 2m+1) of a column into one bf16x2 word (see gate_up_epi_chunk).
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    const float x = __shfl_xor_sync(FULL_MASK, odd ? v[j] : v[j + 1], 1);
    const __nv_bfloat162 w2 = odd ? __floats2bfloat162_rn(x, v[j + 1]) : __floats2bfloat162_rn(v[j], x);
    stg_y[(j + (odd ? 1 : 0)) * 16 + (lane >> 1)] = *reinterpret_cast<const uint32_t *>(&w2);
  }
  __syncwarp();
  // Four lanes per column row: 8 rows x 64 contiguous bytes per store instruction.
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = (lane >> 2) + 8 * i, cc = lane & 3;
    const int drow = __shfl_sync(FULL_MASK, dst, r);
    if (c0 + r < im.rows)
      *(uint4 *)(yout + (int64_t)drow * H + ocol + cc * 8) = *(const uint4 *)(stg_y + r * 16 + cc * 4);
  }
  __syncwarp();
}

// The same chunk written as float rows without rounding: lane = output
// feature, so each of the 32 stores (one per column) is one 128-byte row segment.
__device__ __forceinline__ void down_epi_chunk_f32(const float (&v)[32], int ocol, int c0, int dst, const Item &im,
                                                   float *yout, int H, int lane) {
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    const int drow = __shfl_sync(FULL_MASK, dst, j);
    if (c0 + j < im.rows) yout[(int64_t)drow * H + ocol + lane] = v[j];
  }
}

template <int MODE>
__global__ void __launch_bounds__(tc_threads<MODE>(), 1)
tc_gemm_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  constexpr int NMAX = TcCfg<MODE>::NMAX, MT = TcCfg<MODE>::MT, STAGES = TcCfg<MODE>::STAGES;
  constexpr int A_BYTES = MT * TC_TILE_A_BYTES;
  constexpr int EPI_WARPS = TcCfg<MODE>::EPI_WARPS, EPI_BYTES = TcCfg<MODE>::EPI_BYTES;
  constexpr int GATHER_FIRST = tc_gather_first<MODE>();
  static_assert(EPI_WARPS * EPI_BYTES <= TC_EPI_MAX_BYTES && EPI_WARPS % 4 == 0, "epilogue layout");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sa = base;
  uint8_t *sb = sa + STAGES * A_BYTES;
  uint8_t *epi = sb + STAGES * TC_B_BYTES;
  int32_t *tok_all = (int32_t *)(epi + TC_EPI_MAX_BYTES);
  uint64_t *bars = (uint64_t *)(tok_all + TC_TOK_INTS);
  uint64_t *full = bars, *empty = bars + TC_MAX_STAGES;
  constexpr int NBUF = tc_nbuf<MODE>();
  uint64_t *tfull = bars + 2 * TC_MAX_STAGES, *tempty = tfull + NBUF, *mma_done = tempty + NBUF;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(&full[s], 1 + (MODE == TC_GATE_UP ? GATHER_THREADS : 0));
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < NBUF; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.a_sh);
  }
  if (warp == 1) tmem_alloc(tmem_slot, TC_TMEM_COLS);
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
      // Weights stream through L2 once; activations are read by several CTAs.
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      int stage = 0;
      uint32_t phase = 0;
      uint32_t issued = 0, issued_phase = 0;  // per-stage bits, for draining after an abort
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const Item im = decode_item<MODE>(it, p);
        const bool sh = im.seg == p.E;
        const uint32_t bytes = A_BYTES + (MODE == TC_GATE_UP ? 0 : im.n * 128);
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
          uint8_t *a_dst = sa + stage * A_BYTES;
          uint8_t *b_dst = sb + stage * TC_B_BYTES;
          if (MODE == TC_GATE_UP) {
            // One 5-D box: for 8 groups of 16 features (two M tiles), 16 gate rows then 16 up rows.
            tma_load_5d(a_dst, sh ? &maps.a_sh : &maps.a, &full[stage], kb * 64, 0, 0, im.f * 4 * MT, sh ? 0 : im.seg - p.e0,
                        pol_w);
          } else {
            tma_load_2d(a_dst, sh ? &maps.a_sh : &maps.a, &full[stage], kb * 64,
                        (sh ? 0 : (im.seg - p.e0) * p.H) + im.f * 128 * MT, pol_w);
          }
          if (MODE != TC_GATE_UP) {
            // Token rows [row0, row0 + n) as power-of-two boxes (n is a multiple of 16).
            const int kx = kb * 64;
            const CUtensorMap *bm = sh ? maps.b_sh : maps.b;
            int r = 0;
#pragma unroll
            for (int h = 0; h < 5; ++h) {
              const int box = 256 >> h;
              if (box > NMAX) continue;
              while (im.n - r >= box) {
                tma_load_2d(b_dst + r * 128, &bm[h], &full[stage], kx, (int)(im.row0 + r), pol_x);
                r += box;
              }
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) {
        // Let the copies already in flight land before the CTA exits.
        volatile int never = 0;
        for (int s = 0; s < STAGES; ++s)
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
        const Item im = decode_item<MODE>(it, p);
        const int b = cnt % NBUF;
        if (!mbar_wait(&tempty[b], ((cnt / NBUF) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t idesc = idesc_bf16_f32(128, im.n);
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          if (MODE == TC_GATE_UP) fence_proxy_async_smem();  // the gathered rows: generic -> async proxy
          tc_fence_after();
          const uint64_t bd = smem_desc_sw128(smem_u32(sb + stage * TC_B_BYTES));
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const uint32_t d = tmem + (b * MT + mt) * 256;
            const uint32_t accumulate = kb != 0;
            const uint64_t ad = smem_desc_sw128(smem_u32(sa + stage * A_BYTES + mt * TC_TILE_A_BYTES));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes = +2 in the descriptor address field
              mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (accumulate | kk) != 0);
          }
          mma_commit(&empty[stage]);
          if (++stage == STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        mma_commit(&tfull[b]);
        ++cnt;
      }
      // Every MMA this thread issued has finished before TMEM is released.
      mma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else if (warp < GATHER_FIRST) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    // The EPI_WARPS / 4 warps of a quarter take 32-column chunks in turn.
    constexpr int CSTEP = 32 * (EPI_WARPS / 4);
    const int cfirst = 32 * ((warp - TC_EPI_FIRST) >> 2);
    uint8_t *stg = epi + (warp - TC_EPI_FIRST) * EPI_BYTES;
    uint32_t cnt = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
      const Item im = decode_item<MODE>(it, p);
      const int b = cnt % NBUF;
      if (!warp_wait(&tfull[b], (cnt / NBUF) & 1, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tq = tmem + b * MT * 256 + ((uint32_t)(q * 32) << 16);
      if (MODE == TC_GATE_UP) {
        const bool sh = im.seg == p.E;
        const int Iseg = sh ? p.Is : p.I;
        __nv_bfloat16 *hout = sh ? p.h_shared : p.h_routed;
        __nv_bfloat16 *guout = sh ? p.gu_shared : p.gu_routed;
        for (int c0 = cfirst; c0 < im.n; c0 += CSTEP) {
          float vt[MT][32];
          if (MT == 2) tmem_ld32x2(tq + c0, tq + 256 + c0, vt[0], vt[MT - 1]);
          else tmem_ld32(tq + c0, vt[0]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt)
            gate_up_epi_chunk(vt[mt], (im.f * MT + mt) * 64 + 16 * q, c0, im, Iseg, hout, guout, stg, lane);
        }
      } else {
        const bool sh = im.seg == p.E;
        __nv_bfloat16 *yout = sh ? p.y_shared : p.y_routed;
        for (int c0 = cfirst; c0 < im.n; c0 += CSTEP) {
          // Destination row of column c0 + lane, fetched before the accumulator loads.
          int dst = 0;
          if (c0 + lane < im.rows)
            dst = (sh || p.y_sorted) ? (int)(im.row0 + c0 + lane) : __ldg(p.sorted_route + im.row0 + c0 + lane);
          float vt[MT][32];
          if (MT == 2) tmem_ld32x2(tq + c0, tq + 256 + c0, vt[0], vt[MT - 1]);
          else tmem_ld32(tq + c0, vt[0]);
#pragma unroll
          for (int mt = 0; mt < MT; ++mt) {
            const int ocol = (im.f * MT + mt) * 128 + q * 32;
            if (p.y_f32) down_epi_chunk_f32(vt[mt], ocol, c0, dst, im, (float *)(void *)yout, p.H, lane);
            else down_epi_chunk(vt[mt], ocol, c0, dst, im, yout, p.H, stg, lane);
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[b]);
      ++cnt;
    }
  } else if (MODE == TC_GATE_UP) {
    // ------------------------------------------------------------ row gather
    // Warp g copies the rows r = 8 i + g; lane = 8 * (i mod 4) + 16-byte chunk
    // qc, written at the 128-byte swizzled position (qc ^ g) of row r.  Each
    // thread's copies into a stage arrive on the stage's `full` barrier when
    // they land, so the warps run ahead as far as free stages allow; the MMA
    // thread fences them into the async proxy after its wait (pad rows past the
    // segment are left as they are: their accumulator columns are never read).
    const int g = warp - GATHER_FIRST;
    const int sub = lane >> 3, qc = lane & 7;
    int32_t *tok = tok_all + g * 32;
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
      const Item im = decode_item<MODE>(it, p);
      const bool sh = im.seg == p.E;
      const int ni = (im.rows - g + 7) / 8;  // rows of this warp: i < ni  (<= 32)
      __syncwarp();
      if (lane < ni) {
        const int64_t row = im.row0 + 8 * lane + g;
        tok[lane] = sh ? (int)row : __ldg(p.sorted_route + row) / p.k;
      }
      __syncwarp();
      for (int kb = 0; kb < im.nk; ++kb) {
        if (!warp_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
        const uint32_t bsm = smem_u32(sb + stage * TC_B_BYTES) + g * 128 + ((qc ^ g) << 4);
        const __nv_bfloat16 *src = p.x + kb * 64 + qc * 8;
        for (int i = sub; i < ni; i += 4) cp_async_16(bsm + i * 1024, src + (int64_t)tok[i] * p.H);
        cp_async_mbar_arrive(&full[stage]);
        if (++stage == STAGES) stage = 0, phase ^= 1;
      }
    }
    cp_async_wait<0>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TC_TMEM_COLS);
}

// ---------------------------------------------------------------------------
// The grouped GEMMs on CTA pairs (cta_group::2).
//
// An item is two M tiles (gate_up: 64 gate + 64 up rows each, i.e. 128
// features; down: 128 outputs each) x up to 256 rows of one segment.  The
// two CTAs of a cluster run it as one M = 256 MMA: CTA r holds M tile 2f + r
// of the weights and rows [r n/2, (r + 1) n/2) of the item's rows (gate_up:
// x rows gathered by TMA gather4; down: consecutive h rows by tile boxes),
// so each row is fetched once per item and each CTA's accumulator is 128
// lanes x n columns.  That leaves room for two accumulator buffers, so an
// item's epilogue overlaps the next item's mainloop.  A stage holds PR_KSUB
// K blocks of 64: per block 16 KB of weights + 16 KB of rows per CTA (fewer,
// larger stages: one handshake per 128 K for the single MMA thread that
// drives both SMs).
//
// Synchronisation: the even CTA's MMA thread waits on its full[s]: one
// arrival by the even CTA's producer, which expects the bytes of both CTAs'
// weight tiles and rows; every copy of both CTAs is a TMA load completing on
// that barrier.  MMA completion is committed to empty[s] / tfull[b] /
// mma_done in both CTAs at once; the epilogue warps of both CTAs arrive on
// the even CTA's tempty[b].
// ---------------------------------------------------------------------------
constexpr int PR_KSUB = 2;    // K blocks of 64 per stage
constexpr int PR_STAGES = 3;  // stage ring depth
constexpr int PR_A_BYTES = TC_TILE_A_BYTES, PR_B_BYTES = 128 * 128;  // one K block
constexpr int PR_STAGE_BYTES = PR_KSUB * (PR_A_BYTES + PR_B_BYTES);
// Per mode: epilogue warps and staging bytes per warp; rows of an item are
// padded to a multiple of NROUND (each CTA's half a multiple of 8 for the
// gate_up gather4 quads, of 16 for the down tile boxes).
template <int MODE>
struct PrCfg;
template <>
struct PrCfg<TC_GATE_UP> {
  static constexpr int EPI_WARPS = 8, EPI_BYTES = 2560, NROUND = 16, GATHER_WARPS = TC_GATHER_WARPS;
};
template <>
struct PrCfg<TC_DOWN> {
  static constexpr int EPI_WARPS = 16, EPI_BYTES = 2048, NROUND = 32, GATHER_WARPS = 0;
};
template <int MODE>
constexpr int pr_threads() {
  return 32 * (TC_EPI_FIRST + PrCfg<MODE>::EPI_WARPS + PrCfg<MODE>::GATHER_WARPS);
}
template <int MODE>
constexpr int pr_smem_bytes() {
  return 1024 + PR_STAGES * PR_STAGE_BYTES + PrCfg<MODE>::EPI_WARPS * PrCfg<MODE>::EPI_BYTES + 512;
}
static_assert(pr_smem_bytes<TC_GATE_UP>() <= 232448 && pr_smem_bytes<TC_DOWN>() <= 232448, "pair shared memory");

template <int MODE>
__global__ void __launch_bounds__(pr_threads<MODE>(), 1)
tc_pair_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  constexpr int EPI_WARPS = PrCfg<MODE>::EPI_WARPS, EPI_BYTES = PrCfg<MODE>::EPI_BYTES;
  constexpr int NROUND = PrCfg<MODE>::NROUND;
  constexpr int GATHER_FIRST = TC_EPI_FIRST + EPI_WARPS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  // Stage s: K block j's weight tile at sa(s, j), its rows at sb(s, j).
  auto sa = [&](int s, int j) { return base + s * PR_STAGE_BYTES + j * PR_A_BYTES; };
  auto sb = [&](int s, int j) { return base + s * PR_STAGE_BYTES + PR_KSUB * PR_A_BYTES + j * PR_B_BYTES; };
  uint8_t *epi = base + PR_STAGES * PR_STAGE_BYTES;
  uint64_t *bars = (uint64_t *)(epi + EPI_WARPS * EPI_BYTES);
  uint64_t *full = bars, *empty = full + PR_STAGES;
  uint64_t *tfull = empty + PR_STAGES, *tempty = tfull + 2, *mma_done = tempty + 2;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  // The item with its rows padded for the pair (each CTA takes n / 2 of them).
  auto item = [&](int it) {
    Item im = decode_item<MODE>(it, p);
    im.n = (int)round_up(im.rows, NROUND);
    return im;
  };
  if (threadIdx.x == 0) {
    for (int s = 0; s < PR_STAGES; ++s) {
      mbar_init(&full[s], 1);  // used in the even CTA
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.a);
    prefetch_tmap(&maps.a_sh);
  }
  cluster_sync();  // both CTAs' barriers exist before either touches the other's
  if (warp == 1) tmem_alloc_pair(tmem_slot, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();
  griddep_wait();
  const int total = __ldg(p.item_start + p.E + 1);

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    // Weights (both modes) and, for DOWN, this CTA's half of the item's h
    // rows (consecutive in sorted order) as power-of-two boxes.
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first(), pol_x = policy_evict_last();
      const uint32_t full0 = mapa_shared(&full[0], 0);
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int it = cid; it < total && ok; it += ncl) {
        const Item im = item(it);
        const bool sh = im.seg == p.E;
        const int mtile = im.f * 2 + (int)rank;  // this CTA's M tile (64 gate/up features or 128 outputs)
        const CUtensorMap *am = sh ? &maps.a_sh : &maps.a;
        const int half = im.n >> 1;
        for (int ks = 0; ks < im.nk / PR_KSUB; ++ks) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          // Both CTAs' weight tiles and rows (n / 2 each) complete on the even CTA's barrier.
          if (leader) mbar_arrive_expect_tx(&full[stage], PR_KSUB * (2 * PR_A_BYTES + (uint32_t)im.n * 128));
          const uint32_t bar = full0 + (uint32_t)(stage * sizeof(uint64_t));
#pragma unroll
          for (int j = 0; j < PR_KSUB; ++j) {
            const int kx = (ks * PR_KSUB + j) * 64;
            if (MODE == TC_GATE_UP) {
              // 4 groups of 16 features: 16 gate rows then 16 up rows each.
              tma_load_5d_pair(sa(stage, j), am, bar, kx, 0, 0, mtile * 4, sh ? 0 : im.seg - p.e0, pol_w);
            } else {
              tma_load_2d_pair(sa(stage, j), am, bar, kx, (sh ? 0 : (im.seg - p.e0) * p.H) + mtile * 128, pol_w);
              const CUtensorMap *bm = sh ? maps.b_sh : maps.b;
              const int r0 = (int)im.row0 + (int)rank * half;
              int r = 0;
#pragma unroll
              for (int h = 1; h < 5; ++h) {  // boxes of 128 .. 16 rows
                const int box = 256 >> h;
                while (half - r >= box) {
                  tma_load_2d_pair(sb(stage, j) + r * 128, &bm[h], bar, kx, r0 + r, pol_x);
                  r += box;
                }
              }
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == PR_STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok && leader) {
        // The stages in flight (both CTAs' copies complete here) land before the pair exits.
        volatile int never = 0;
        for (int s = 0; s < PR_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // -------------------------------------------------------- MMA issuer (both CTAs' tensor memory)
        int stage = 0;
        uint32_t phase = 0, cnt = 0;
        bool ok = true;
        for (int it = cid; it < total && ok; it += ncl) {
          const Item im = item(it);
          const int b = cnt & 1;
          if (!mbar_wait(&tempty[b], ((cnt >> 1) & 1) ^ 1, abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t idesc = idesc_bf16_f32(256, im.n);
          for (int ks = 0; ks < im.nk / PR_KSUB; ++ks) {
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int j = 0; j < PR_KSUB; ++j) {
              const uint64_t ad = smem_desc_sw128(smem_u32(sa(stage, j)));
              const uint64_t bd = smem_desc_sw128(smem_u32(sb(stage, j)));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes = +2 in the descriptor address field
                mma_bf16_pair(tmem + b * 256, ad + 2 * kk, bd + 2 * kk, idesc, (ks | j | kk) != 0);
            }
            mma_commit_pair(&empty[stage]);
            if (++stage == PR_STAGES) stage = 0, phase ^= 1;
          }
          if (!ok) break;
          mma_commit_pair(&tfull[b]);
          ++cnt;
        }
        mma_commit_pair(mma_done);
      }
      // Every pair MMA has finished (it wrote both CTAs' tensor memory) before TMEM is released.
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else if (warp < GATHER_FIRST) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;
    constexpr int CSTEP = 32 * (EPI_WARPS / 4);
    const int cfirst = 32 * ((warp - TC_EPI_FIRST) >> 2);
    uint8_t *stg = epi + (warp - TC_EPI_FIRST) * EPI_BYTES;
    const uint32_t tempty_leader0 = mapa_shared(&tempty[0], 0);
    uint32_t cnt = 0;
    for (int it = cid; it < total; it += ncl) {
      const Item im = item(it);
      const int b = cnt & 1;
      int ok = 0;
      if (lane == 0) ok = mbar_wait(&tfull[b], (cnt >> 1) & 1, abort_flag, p.status) ? 1 : 0;
      if (!__shfl_sync(FULL_MASK, ok, 0)) break;
      tc_fence_after();
      const bool sh = im.seg == p.E;
      const uint32_t tq = tmem + b * 256 + ((uint32_t)(q * 32) << 16);
      const int mtile = im.f * 2 + (int)rank;
      if (MODE == TC_GATE_UP) {
        const int Iseg = sh ? p.Is : p.I;
        __nv_bfloat16 *hout = sh ? p.h_shared : p.h_routed;
        __nv_bfloat16 *guout = sh ? p.gu_shared : p.gu_routed;
        for (int c0 = cfirst; c0 < im.n; c0 += CSTEP) {
          float v[32];
          tmem_ld32(tq + c0, v);
          gate_up_epi_chunk(v, mtile * 64 + 16 * q, c0, im, Iseg, hout, guout, stg, lane);
        }
      } else {
        __nv_bfloat16 *yout = sh ? p.y_shared : p.y_routed;
        for (int c0 = cfirst; c0 < im.n; c0 += CSTEP) {
          int dst = 0;
          if (c0 + lane < im.rows)
            dst = (sh || p.y_sorted) ? (int)(im.row0 + c0 + lane) : __ldg(p.sorted_route + im.row0 + c0 + lane);
          float v[32];
          tmem_ld32(tq + c0, v);
          if (p.y_f32) down_epi_chunk_f32(v, mtile * 128 + q * 32, c0, dst, im, (float *)(void *)yout, p.H, lane);
          else down_epi_chunk(v, mtile * 128 + q * 32, c0, dst, im, yout, p.H, stg, lane);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader) mbar_arrive(&tempty[b]);
        else mbar_arrive_remote(tempty_leader0 + (uint32_t)(b * sizeof(uint64_t)));
      }
      ++cnt;
    }
  } else if (MODE == TC_GATE_UP) {
    // ------------------------------------------------------------ row gather (TMA gather4)
    // This CTA's rows of the item: [rank n/2, rank n/2 + n/2) ∩ [0, rows),
    // row i at line i of a K block's B tile (the 128-byte swizzle), four rows
    // per copy; quad qd = g + 8 lane (lanes 0-3) of warp g.  The bytes of
    // both CTAs complete on the even CTA's full[s].  Lines past the item's
    // rows read token 0: their accumulator columns are never read.  The
    // shared expert's rows are consecutive tokens: lane 0 of warp 0 copies
    // the largest multiple of 16 of them as boxes of 128 .. 16 rows
    // (maps.b_sh; lines past the last token are zero-filled), and the quads
    // after it (at most one 8-row remainder) take gather4 copies as above.
    const int g = warp - GATHER_FIRST;
    const uint64_t pol_x = policy_evict_last();
    const uint32_t full0 = mapa_shared(&full[0], 0);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    for (int it = cid; it < total && ok; it += ncl) {
      const Item im = item(it);
      const bool sh = im.seg == p.E;
      const int half = im.n >> 1, hbase = (int)rank * half;
      const int hrows = max(0, min(half, im.rows - hbase));
      const int qd = g + 8 * lane;
      const int hbox = sh ? (half & ~15) : 0;  // rows copied as boxes
      const bool mine = lane < 4 && 4 * qd >= hbox && 4 * qd < half;
      const bool boxes = hbox > 0 && g == 0 && lane == 0;
      int t4[4] = {0, 0, 0, 0};
      if (mine) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * qd + j;
          if (r < hrows) {
            const int64_t row = im.row0 + hbase + r;
            t4[j] = sh ? (int)row : __ldg(p.sorted_route + row) / p.k;
          }
        }
      }
      for (int ks = 0; ks < im.nk / PR_KSUB; ++ks) {
        int w = 0;
        if (lane == 0) w = mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status) ? 1 : 0;
        if (!__shfl_sync(FULL_MASK, w, 0)) { ok = false; break; }
        if (mine) {
          const uint32_t bar = full0 + (uint32_t)(stage * sizeof(uint64_t));
#pragma unroll
          for (int j = 0; j < PR_KSUB; ++j)
            tma_gather4_pair(sb(stage, j) + qd * 512, &maps.b[0], bar, (ks * PR_KSUB + j) * 64, t4[0], t4[1], t4[2],
                             t4[3], pol_x);
        }
        if (boxes) {
          const uint32_t bar = full0 + (uint32_t)(stage * sizeof(uint64_t));
          const int r0 = (int)im.row0 + hbase;
#pragma unroll
          for (int j = 0; j < PR_KSUB; ++j) {
            const int kx = (ks * PR_KSUB + j) * 64;
            int r = 0;
#pragma unroll
            for (int h = 1; h < 5; ++h) {  // boxes of 128 .. 16 rows
              const int box = 256 >> h;
              while (hbox - r >= box) {
                tma_load_2d_pair(sb(stage, j) + r * 128, &maps.b_sh[h], bar, kx, r0 + r, pol_x);
                r += box;
              }
            }
          }
        }
        if (++stage == PR_STAGES) stage = 0, phase ^= 1;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrival, copy or commit targets this CTA any more
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, TC_TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Router logits on the tensor cores.
//
// An item is 128 experts x up to 256 tokens.  A stage holds, for one K block
// j of 64 hidden units, the x tile once and the three split-weight tiles
// W1, W2, W3 of the same columns; the three MMA groups read the same x tile.
// The K range is cut into four fixed chunks of K blocks (chunk c = blocks
// [c nkh / 4, (c + 1) nkh / 4)); a chunk accumulates in one of two TMEM
// buffers while the epilogue adds the previous chunk into FP32 registers, so
// logit = ((chunk0 + chunk1) + chunk2) + chunk3 (+ bias), the same order for
// every token and every T.
// ---------------------------------------------------------------------------
constexpr int RT_NMAX = 256, RT_STAGES = 2, RT_CHUNKS = 4, RT_EPI_WARPS = 8;
constexpr int RT_A_BYTES = 3 * TC_TILE_A_BYTES;
constexpr int RT_THREADS = 32 * (TC_EPI_FIRST + RT_EPI_WARPS);
static_assert(RT_STAGES * (RT_A_BYTES + TC_B_BYTES) + 256 + 1024 <= TC_SMEM_BYTES, "router smem");

struct RtItem {
  int f;         // expert tile (128 experts; the pair form: 256)
  int64_t row0;  // first token
  int rows, n;
  int kc;        // the pair form with split K: the one K chunk of the item
};

// Token tiles of rt_rpt rows (a multiple of 16, at most 256); the host picks
// the tile count so that the items fill the SMs.  A logit's K order does not
// depend on the tile its token falls in.
__device__ inline RtItem rt_item(int it, const TcParams &p) {
  const int nt = it % p.rt_ntile;
  RtItem r;
  r.f = it / p.rt_ntile;
  r.row0 = (int64_t)nt * p.rt_rpt;
  r.rows = min(p.rt_rpt, p.T - nt * p.rt_rpt);
  r.n = (int)round_up(r.rows, 16);
  return r;
}

__global__ void __launch_bounds__(RT_THREADS, 1)
tc_router_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sa = base;
  uint8_t *sb = sa + RT_STAGES * RT_A_BYTES;
  uint64_t *bars = (uint64_t *)(sb + RT_STAGES * TC_B_BYTES);
  uint64_t *full = bars, *empty = bars + RT_STAGES;
  uint64_t *tfull = bars + 2 * RT_STAGES, *tempty = tfull + 2, *mma_done = tempty + 2;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RT_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 32 * RT_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&maps.a);
  if (warp == 1) tmem_alloc(tmem_slot, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();
  griddep_wait();
  const int total = p.n_items, nkh = p.H / 64;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // split weights and x are read by many CTAs
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const RtItem im = rt_item(it, p);
        const uint32_t bytes = p.rt_splits * TC_TILE_A_BYTES + im.n * 128;
        for (int j = 0; j < nkh; ++j) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[stage], bytes);
          uint8_t *a_dst = sa + stage * RT_A_BYTES;
          uint8_t *b_dst = sb + stage * TC_B_BYTES;
#pragma unroll
          for (int sp = 0; sp < p.rt_splits; ++sp)
            tma_load_2d(a_dst + sp * TC_TILE_A_BYTES, &maps.a, &full[stage], sp * p.H + j * 64, im.f * 128, pol);
          int r = 0;
#pragma unroll
          for (int h = 0; h < 5; ++h) {
            const int box = 256 >> h;
            while (im.n - r >= box) {
              tma_load_2d(b_dst + r * 128, &maps.b[h], &full[stage], j * 64, (int)(im.row0 + r), pol);
              r += box;
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == RT_STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok) {
        volatile int never = 0;
        for (int s = 0; s < RT_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, uses = 0;  // uses: bit b = parity of the uses of TMEM buffer b
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const RtItem im = rt_item(it, p);
        const uint32_t idesc = idesc_bf16_f32(128, im.n);
        for (int c = 0; c < RT_CHUNKS && ok; ++c) {
          const int b = c & 1;
          if (!mbar_wait(&tempty[b], ((uses >> b) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint32_t d = tmem + b * 256;
          const int j0 = c * nkh / RT_CHUNKS, j1 = (c + 1) * nkh / RT_CHUNKS;
          for (int j = j0; j < j1; ++j) {
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint64_t bd = smem_desc_sw128(smem_u32(sb + stage * TC_B_BYTES));
#pragma unroll
            for (int sp = 0; sp < p.rt_splits; ++sp) {
              const uint64_t ad = smem_desc_sw128(smem_u32(sa + stage * RT_A_BYTES + sp * TC_TILE_A_BYTES));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (j != j0 || sp != 0 || kk != 0) ? 1u : 0u);
            }
            mma_commit(&empty[stage]);
            if (++stage == RT_STAGES) stage = 0, phase ^= 1;
          }
          if (!ok) break;
          mma_commit(&tfull[b]);
          uses ^= 1u << b;
        }
      }
      mma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp (q, hq): TMEM lane quarter q (experts), columns [128 hq, 128 hq + 128).
    const int q = warp & 3, hq = (warp - TC_EPI_FIRST) >> 2;
    uint32_t uses = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
      const RtItem im = rt_item(it, p);
      float acc[128];
#pragma unroll
      for (int c = 0; c < RT_CHUNKS; ++c) {
        const int b = c & 1;
        if (!warp_wait(&tfull[b], (uses >> b) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + b * 256 + ((uint32_t)(q * 32) << 16) + hq * 128;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          if (hq * 128 + cc * 32 < im.n) {
            float v[32];
            tmem_ld32(tb + cc * 32, v);
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) acc[cc * 32 + jj] = c == 0 ? v[jj] : acc[cc * 32 + jj] + v[jj];
          }
        }
        tc_fence_before();
        mbar_arrive(&tempty[b]);
        uses ^= 1u << b;
      }
      if (!ok) break;
      const int e = im.f * 128 + q * 32 + lane;
      const float bias = (p.bias && e < p.E) ? __ldg(p.bias + e) : 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int jj = 0; jj < 32; ++jj) {
          const int col = hq * 128 + cc * 32 + jj;
          if (col < im.rows && e < p.E)
            p.logits[(im.row0 + col) * p.E + e] = p.bias ? acc[cc * 32 + jj] + bias : acc[cc * 32 + jj];
        }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TC_TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Router logits on CTA pairs (tcgen05.mma.cta_group::2, M = 256): a pair
// item is 256 experts (128 per CTA: its M tile of each split weight) x up to
// 256 tokens (each CTA loads half of the token rows; the even CTA's one MMA
// thread drives both tensor cores).  A stage holds one K block of 64 hidden
// units: per CTA the three split-weight tiles (48 KB) and its half of the x
// rows (up to 16 KB), so three stages fit where the single-SM router holds
// two.  The K chunks, their order and the FP32 sums of the epilogue are the
// single-SM router's, so every logit is the same MMA chain and the same sum:
// the two kernels give equal logits bit for bit.  Small batches run with
// split K: each item computes one chunk and writes its sum to a partial
// plane, which router_chunk_sum_kernel adds in the same order.
// ---------------------------------------------------------------------------
constexpr int RP_STAGES = 3, RP_NROUND = 32;
// Sixteen epilogue warps, 64 accumulator columns each: a warp keeps the
// running chunk sums of its columns in registers (64 per thread) without
// spilling them.  With eight warps (128 sums per thread, 168 registers at
// three warps per SM sub-partition) part of the sums spilled to local
// memory, which the small L1 left by 198 KB of shared memory serves from L2,
// or from memory when L2 holds other data.
constexpr int RP_EPI_WARPS = 16, RP_COLS = 4 * RT_NMAX / RP_EPI_WARPS;
constexpr int RP_THREADS = 32 * (TC_EPI_FIRST + RP_EPI_WARPS);
constexpr int RP_B_BYTES = 128 * 128;  // this CTA's half of up to 256 token rows x 64 bf16
constexpr int RP_STAGE_BYTES = RT_A_BYTES + RP_B_BYTES;
constexpr int RP_SMEM = 1024 + RP_STAGES * RP_STAGE_BYTES + 512;
static_assert(RP_SMEM <= 232448, "pair router shared memory");

__global__ void __launch_bounds__(RP_THREADS, 1)
tc_router_pair_kernel(const __grid_constant__ TcMaps maps, const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  auto sa = [&](int s) { return base + s * RP_STAGE_BYTES; };
  auto sb = [&](int s) { return base + s * RP_STAGE_BYTES + RT_A_BYTES; };
  uint64_t *bars = (uint64_t *)(base + RP_STAGES * RP_STAGE_BYTES);
  uint64_t *full = bars, *empty = full + RP_STAGES;
  uint64_t *tfull = empty + RP_STAGES, *tempty = tfull + 2, *mma_done = tempty + 2;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cid = blockIdx.x >> 1, ncl = gridDim.x >> 1;
  if (threadIdx.x == 0) {
    for (int s = 0; s < RP_STAGES; ++s) {
      mbar_init(&full[s], 1);  // used in the even CTA
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 2 * RP_EPI_WARPS);  // used in the even CTA: one arrival per epilogue warp of the pair
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tmap(&maps.a);
  cluster_sync();  // both CTAs' barriers exist before either touches the other's
  if (warp == 1) tmem_alloc_pair(tmem_slot, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();
  griddep_wait();
  const int total = p.n_items, nkh = p.H / 64;
  // Item it, with q = it / kparts: experts [256 f, +256) for f = q / rt_ntile (this CTA's
  // 128 from 256 f + 128 rank), tokens [rt_rpt (q % rt_ntile), +rt_rpt), rows padded to
  // RP_NROUND (each CTA loads n / 2); with split K (kparts = RT_CHUNKS) only K chunk
  // it % kparts, else all RT_CHUNKS chunks.
  const int kparts = p.rt_kparts > 1 ? p.rt_kparts : 1;
  auto item = [&](int it) {
    const int rest = it / kparts;
    const int nt = rest % p.rt_ntile;
    RtItem r;
    r.kc = it % kparts;
    r.f = rest / p.rt_ntile;
    r.row0 = (int64_t)nt * p.rt_rpt;
    r.rows = min(p.rt_rpt, p.T - nt * p.rt_rpt);
    r.n = (int)round_up(r.rows, RP_NROUND);
    return r;
  };
  // The chunks [c_begin, c_end) of an item.
  auto c_begin = [&](const RtItem &im) { return kparts == 1 ? 0 : im.kc; };
  auto c_end = [&](const RtItem &im) { return kparts == 1 ? RT_CHUNKS : im.kc + 1; };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (both CTAs)
    if (lane == 0) {
      const uint64_t pol = policy_evict_last();  // split weights and x are read by many CTAs
      const uint32_t full0 = mapa_shared(&full[0], 0);
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int it = cid; it < total && ok; it += ncl) {
        const RtItem im = item(it);
        const int erow = im.f * 256 + (int)rank * 128;
        const int half = im.n >> 1;
        const int64_t r0 = im.row0 + (int64_t)rank * half;
        for (int j = c_begin(im) * nkh / RT_CHUNKS; j < c_end(im) * nkh / RT_CHUNKS; ++j) {
          if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
          // Both CTAs' weight tiles and rows complete on the even CTA's barrier.
          if (leader) mbar_arrive_expect_tx(&full[stage], 2 * p.rt_splits * TC_TILE_A_BYTES + (uint32_t)im.n * 128);
          const uint32_t bar = full0 + (uint32_t)(stage * sizeof(uint64_t));
          for (int sp = 0; sp < p.rt_splits; ++sp)
            tma_load_2d_pair(sa(stage) + sp * TC_TILE_A_BYTES, &maps.a, bar, sp * p.H + j * 64, erow, pol);
          int r = 0;
#pragma unroll
          for (int h = 1; h < 5; ++h) {  // boxes of 128 .. 16 rows
            const int box = 256 >> h;
            while (half - r >= box) {
              tma_load_2d_pair(sb(stage) + r * 128, &maps.b[h], bar, j * 64, (int)(r0 + r), pol);
              r += box;
            }
          }
          issued |= 1u << stage;
          issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == RP_STAGES) stage = 0, phase ^= 1;
        }
      }
      if (!ok && leader) {
        // The stages in flight (both CTAs' copies complete here) land before the pair exits.
        volatile int never = 0;
        for (int s = 0; s < RP_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      if (leader) {
        // -------------------------------------------------------- MMA issuer (both CTAs' tensor memory)
        int stage = 0;
        uint32_t phase = 0, uses = 0;  // uses: bit b = parity of the uses of TMEM buffer b
        bool ok = true;
        for (int it = cid; it < total && ok; it += ncl) {
          const RtItem im = item(it);
          const uint32_t idesc = idesc_bf16_f32(256, im.n);
          for (int c = c_begin(im); c < c_end(im) && ok; ++c) {
            const int b = c & 1;
            if (!mbar_wait(&tempty[b], ((uses >> b) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
            const uint32_t d = tmem + b * 256;
            const int j0 = c * nkh / RT_CHUNKS, j1 = (c + 1) * nkh / RT_CHUNKS;
            for (int j = j0; j < j1; ++j) {
              if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
              tc_fence_after();
              const uint64_t bd = smem_desc_sw128(smem_u32(sb(stage)));
              for (int sp = 0; sp < p.rt_splits; ++sp) {
                const uint64_t ad = smem_desc_sw128(smem_u32(sa(stage) + sp * TC_TILE_A_BYTES));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16_pair(d, ad + 2 * kk, bd + 2 * kk, idesc, (j != j0 || sp != 0 || kk != 0) ? 1u : 0u);
              }
              mma_commit_pair(&empty[stage]);
              if (++stage == RP_STAGES) stage = 0, phase ^= 1;
            }
            if (!ok) break;
            mma_commit_pair(&tfull[b]);
            uses ^= 1u << b;
          }
        }
        mma_commit_pair(mma_done);
      }
      // Every pair MMA has finished (it wrote both CTAs' tensor memory) before TMEM is released.
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // Warp (q, part): TMEM lane quarter q (experts), columns [RP_COLS part, RP_COLS part + RP_COLS).
    const int q = warp & 3, part = (warp - TC_EPI_FIRST) >> 2;
    constexpr int NCC = RP_COLS / 32;  // 32-column pieces of the stores (TMEM is read 16 columns at a time)
    const uint32_t tempty_leader0 = mapa_shared(&tempty[0], 0);
    uint32_t uses = 0;
    bool ok = true;
    for (int it = cid; it < total && ok; it += ncl) {
      const RtItem im = item(it);
      const int cb = c_begin(im), ce = c_end(im);
      float acc[RP_COLS];
#pragma unroll
      for (int c = 0; c < RT_CHUNKS; ++c) {
        if (c < cb || c >= ce) continue;
        const int b = c & 1;
        if (!warp_wait(&tfull[b], (uses >> b) & 1, abort_flag, p.status)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tb = tmem + b * 256 + ((uint32_t)(q * 32) << 16) + part * RP_COLS;
#pragma unroll
        for (int cc = 0; cc < RP_COLS / 16; ++cc) {
          if (part * RP_COLS + cc * 16 < im.n) {
            float v[16];
            tmem_ld16(tb + cc * 16, v);
#pragma unroll
            for (int jj = 0; jj < 16; ++jj) acc[cc * 16 + jj] = c == cb ? v[jj] : acc[cc * 16 + jj] + v[jj];
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (leader) mbar_arrive(&tempty[b]);
          else mbar_arrive_remote(tempty_leader0 + (uint32_t)(b * sizeof(uint64_t)));
        }
        uses ^= 1u << b;
      }
      if (!ok) break;
      const int e = im.f * 256 + (int)rank * 128 + q * 32 + lane;
      if (kparts == 1) {
        const float bias = (p.bias && e < p.E) ? __ldg(p.bias + e) : 0.f;
#pragma unroll
        for (int cc = 0; cc < NCC; ++cc)
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int col = part * RP_COLS + cc * 32 + jj;
            if (col < im.rows && e < p.E)
              p.logits[(im.row0 + col) * p.E + e] = p.bias ? acc[cc * 32 + jj] + bias : acc[cc * 32 + jj];
          }
      } else {
        // This item's chunk sum, summed with the other chunks (in chunk order) by router_chunk_sum_kernel.
        float *plane = p.rt_partial + (size_t)im.kc * p.T * p.E;
#pragma unroll
        for (int cc = 0; cc < NCC; ++cc)
#pragma unroll
          for (int jj = 0; jj < 32; ++jj) {
            const int col = part * RP_COLS + cc * 32 + jj;
            if (col < im.rows && e < p.E) plane[(im.row0 + col) * p.E + e] = acc[cc * 32 + jj];
          }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no remote arrival, copy or commit targets this CTA any more
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, TC_TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Router with split K (small batches): the pair router wrote the four chunk
// sums of every logit separately; logit = ((part0 + part1) + part2) + part3
// (+ bias), the additions and order of the epilogue that sums all four
// chunks of an item itself, so a token's logits do not depend on which
// form ran (that is, on T).  Four consecutive logits per thread (E % 256 == 0).
__global__ void __launch_bounds__(256)
router_chunk_sum_kernel(int64_t n, int E, const float *__restrict__ part, const float *__restrict__ bias,
                        float *__restrict__ logits) {
  griddep_launch();
  griddep_wait();
  const int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * 4;
  if (i >= n) return;
  float4 a = __ldg((const float4 *)(part + i));
#pragma unroll
  for (int c = 1; c < RT_CHUNKS; ++c) {
    const float4 b = __ldg((const float4 *)(part + c * n + i));
    a.x = a.x + b.x;
    a.y = a.y + b.y;
    a.z = a.z + b.z;
    a.w = a.w + b.w;
  }
  if (bias) {
    const float4 g = __ldg((const float4 *)(bias + i % E));
    a.x = a.x + g.x;
    a.y = a.y + g.y;
    a.z = a.z + g.z;
    a.w = a.w + g.w;
  }
  *(float4 *)(logits + i) = a;
}

// ---------------------------------------------------------------------------
// Exact three-way bf16 split of the FP32 router weight: Wr3[e] = [W1 | W2 | W3]
// with W1 = rn(w), W2 = rn(w - W1), W3 = rn(w - W1 - W2).  Each residual is
// exact in FP32 and holds at most 16 then 8 significant bits, so W3 captures
// the rest and W1 + W2 + W3 = w exactly.
// ---------------------------------------------------------------------------
__global__ void split_router_weight_kernel(int64_t n4, int H, const float4 *__restrict__ wr,
                                           __nv_bfloat16 *__restrict__ wr3) {
  griddep_launch();
  griddep_wait();
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;  // four consecutive weights
  if (i >= n4) return;
  const int64_t e = (i * 4) / H, h = (i * 4) % H;  // H % 4 == 0: the four share a row
  const float4 w4 = __ldg(wr + i);
  const float w[4] = {w4.x, w4.y, w4.z, w4.w};
  __nv_bfloat162 p1[2], p2[2], p3[2];
#pragma unroll
  for (int j = 0; j < 2; ++j) {
    __nv_bfloat16 a[2], b[2], c[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      const float v = w[2 * j + q];
      a[q] = __float2bfloat16_rn(v);
      const float r1 = v - __bfloat162float(a[q]);
      b[q] = __float2bfloat16_rn(r1);
      const float r2 = r1 - __bfloat162float(b[q]);
      c[q] = __float2bfloat16_rn(r2);
    }
    p1[j] = __halves2bfloat162(a[0], a[1]);
    p2[j] = __halves2bfloat162(b[0], b[1]);
    p3[j] = __halves2bfloat162(c[0], c[1]);
  }
  __nv_bfloat16 *row = wr3 + e * 3 * H + h;
  *(uint2 *)row = *(const uint2 *)p1;
  *(uint2 *)(row + H) = *(const uint2 *)p2;
  *(uint2 *)(row + 2 * H) = *(const uint2 *)p3;
}

// Item tables of two grouped GEMMs over the same segments, one block of 1024
// threads.  start_x[s] = sum_{s' < s} ceil(n_s' / tile) * nf_s' (nf_*_r for
// the routed segments, nf_*_s for the shared segment n_E = T; tile = 256 rows
// for the grouped GEMMs); items[it] = (segment, M-tile pair, first row, rows):
// the rows of a segment are cut into ceil(n / tile) tiles of equal size
// rounded up to 16, a cut that depends only on the segment's own length.  One block forms the prefixes; the expansion
// runs one warp per segment.
constexpr int IT_MAX_E = 1024;

__global__ void __launch_bounds__(1024)
item_tables_kernel(int E, int T, int nf_a_r, int nf_a_s, int nf_b_r, int nf_b_s, const int32_t *__restrict__ offsets,
                   int32_t *__restrict__ start_a, int32_t *__restrict__ start_b, int e_begin, int e_end,
                   int with_shared, int tile) {
  griddep_launch();
  griddep_wait();
  __shared__ int32_t s_off[IT_MAX_E + 1], s_a[IT_MAX_E + 2], s_b[IT_MAX_E + 2];
  __shared__ int32_t buf[1024];
  __shared__ int32_t carry;
  // An empty expert range (the shared expert alone) reads no offsets: they
  // may not exist yet when that table is built.
  for (int i = threadIdx.x; i <= E; i += 1024) s_off[i] = e_begin < e_end ? offsets[i] : 0;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base <= E; base += 1024) {
    const int s = base + threadIdx.x;
    int32_t v = 0;
    if (s < E) v = (s >= e_begin && s < e_end) ? (int32_t)ceil_div(s_off[s + 1] - s_off[s], tile) : 0;
    else if (s == E) v = with_shared ? (int32_t)ceil_div(T, tile) : 0;
    buf[threadIdx.x] = v;
    __syncthreads();
    for (int d = 1; d < 1024; d <<= 1) {
      const int32_t add = (int)threadIdx.x >= d ? buf[threadIdx.x - d] : 0;
      __syncthreads();
      buf[threadIdx.x] += add;
      __syncthreads();
    }
    const int32_t before = carry + buf[threadIdx.x] - v;  // row tiles before segment s
    if (s <= E) {
      s_a[s] = before * nf_a_r;
      s_b[s] = before * nf_b_r;
    }
    if (s == E) {
      s_a[E + 1] = before * nf_a_r + v * nf_a_s;
      s_b[E + 1] = before * nf_b_r + v * nf_b_s;
    }
    __syncthreads();
    if (threadIdx.x == 1023) carry += buf[1023];
    __syncthreads();
  }
  for (int i = threadIdx.x; i <= E + 1; i += 1024) {
    start_a[i] = s_a[i];
    start_b[i] = s_b[i];
  }
}

// Expansion: one warp per segment writes that segment's items of both tables.
__global__ void __launch_bounds__(256)
item_expand_kernel(int E, int T, const int32_t *__restrict__ offsets, const int32_t *__restrict__ start_a,
                   const int32_t *__restrict__ start_b, int4 *__restrict__ items_a, int4 *__restrict__ items_b,
                   int max_a, int max_b, int tile) {
  griddep_launch();
  griddep_wait();
  const int sg = (int)((blockIdx.x * blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (sg > E) return;
  if (__ldg(start_a + sg + 1) == __ldg(start_a + sg) && __ldg(start_b + sg + 1) == __ldg(start_b + sg))
    return;  // empty, or outside the expert range (its offsets are not read)
  const int base = sg == E ? 0 : __ldg(offsets + sg);
  const int n_s = sg == E ? T : __ldg(offsets + sg + 1) - base;
  if (n_s == 0) return;
  const int ntile = (n_s + tile - 1) / tile;
  const int rpt = ((n_s + ntile - 1) / ntile + 15) & ~15;
  const int a0 = __ldg(start_a + sg), na = __ldg(start_a + sg + 1) - a0;
  const int b0 = __ldg(start_b + sg), nb = __ldg(start_b + sg + 1) - b0;
  for (int local = lane; local < max(na, nb); local += 32) {
    const int nt = local % ntile;
    const int4 v = make_int4(sg, local / ntile, base + nt * rpt, min(rpt, n_s - nt * rpt));
    if (local < na && a0 + local < max_a) items_a[a0 + local] = v;
    if (local < nb && b0 + local < max_b) items_b[b0 + local] = v;
  }
}

// ---------------------------------------------------------------- host side
template <int MODE>
static cudaError_t launch_tc(const TcMaps &maps, const TcParams &p, int grid, cudaStream_t stream) {
  cudaError_t e = ensure_smem((const void *)tc_gemm_kernel<MODE>, TC_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  return launch_pdl(tc_gemm_kernel<MODE>, dim3(grid), dim3(tc_threads<MODE>()), TC_SMEM_BYTES, stream, maps, p);
}

// Clusters of two pair CTAs of `MODE` that fit on the device at once (0:
// the pair kernel cannot run here).  Queried once per device.
template <int MODE>
static int pair_clusters() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const int sms = device_sms();
  if (ensure_smem((const void *)tc_pair_kernel<MODE>, pr_smem_bytes<MODE>()) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  int &c = cache[dev & 63];
  if (c == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * sms);
    cfg.blockDim = dim3(pr_threads<MODE>());
    cfg.dynamicSmemBytes = pr_smem_bytes<MODE>();
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void *)tc_pair_kernel<MODE>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

// MOE_TC_PAIR, a diagnostic switch for comparing the CTA-pair and single-SM
// forms, read once per process at the first launch: "0" no pair form (router
// and both grouped GEMMs on single SMs), "1" the gate_up pair only, "2" the
// down pair only; unset (-1): every pair form wherever the shapes and the
// device allow.
static int pair_override() {
  static const int mode = [] {
    const char *e = getenv("MOE_TC_PAIR");
    return (e && e[0] >= '0' && e[0] <= '2') ? e[0] - '0' : -1;
  }();
  return mode;
}

// Whether the grouped GEMM of `MODE` runs on CTA pairs.
template <int MODE>
static bool use_pair(const FfnArgs &a) {
  const int m = pair_override();
  if (m == 0 || (m == 1 && MODE != TC_GATE_UP) || (m == 2 && MODE != TC_DOWN)) return false;
  const bool shapes = MODE == TC_GATE_UP ? a.H % (64 * PR_KSUB) == 0
                                         : a.H % 256 == 0 && a.I % (64 * PR_KSUB) == 0 && a.Is % (64 * PR_KSUB) == 0;
  return shapes && pair_clusters<MODE>() > 0;
}

template <int MODE>
static cudaError_t launch_pair(const TcMaps &maps, const TcParams &p, cudaStream_t stream) {
  const int nc = pair_clusters<MODE>();
  if (nc <= 0) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * nc);
  cfg.blockDim = dim3(pr_threads<MODE>());
  cfg.dynamicSmemBytes = pr_smem_bytes<MODE>();
  cfg.stream = stream;
  cudaLaunchAttribute at[2];
  at[0].id = cudaLaunchAttributeClusterDimension;
  at[0].val.clusterDim.x = 2;
  at[0].val.clusterDim.y = 1;
  at[0].val.clusterDim.z = 1;
  at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  at[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = at;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, tc_pair_kernel<MODE>, maps, p);
}

// Split K for the pair router: a small batch (T * E / 256 <= 4096 token-tiles' worth)
// has too few tokens per weight tile to use the tensor cores well, so each
// of its items takes one K chunk; a rule on the shapes alone, so that the
// workspace size does not depend on the device.
bool router_split_k(int T, int E) { return T > 0 && E % 256 == 0 && (int64_t)T * (E / 256) <= 4096; }

size_t router_tc_scratch_bytes(int T, int E, int H) {
  const size_t wr3 = (size_t)round_up((int64_t)E * 3 * H * 2, 256);
  return wr3 + (router_split_k(T, E) ? (size_t)RT_CHUNKS * T * E * sizeof(float) : 0);
}

// Clusters of two pair-router CTAs that fit on the device at once (0: the
// pair form cannot run here).  Queried once per device.
static int router_pair_clusters() {
  static std::mutex mu;
  static int cache[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (ensure_smem((const void *)tc_router_pair_kernel, RP_SMEM) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mu);
  int &c = cache[dev & 63];
  if (c == 0) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * device_sms());
    cfg.blockDim = dim3(RP_THREADS);
    cfg.dynamicSmemBytes = RP_SMEM;
    cudaLaunchAttribute at[1];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    cfg.attrs = at;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, (const void *)tc_router_pair_kernel, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    c = n > 0 ? n : -1;
  }
  return c > 0 ? c : 0;
}

cudaError_t launch_router_logits_tc(int T, int H, int E, const void *x, const float *wr, const float *bias,
                                    float *logits, void *scratch, int *status, cudaStream_t stream, int splits) {
  if (splits != 1 && splits != 3) return cudaErrorInvalidValue;
  if (T == 0) return cudaSuccess;
  __nv_bfloat16 *wr3 = (__nv_bfloat16 *)scratch;
  const int64_t n4 = (int64_t)E * H / 4;
  cudaError_t e = launch_pdl(split_router_weight_kernel, dim3((unsigned)ceil_div(n4, 256)), dim3(256), 0, stream, n4, H,
                             (const float4 *)wr, wr3);
  if (e != cudaSuccess) return e;
  TcMaps m;
  if (!map_2d(&m.a, wr3, E, 3 * (int64_t)H, 128) || !map_rows(m.b, x, T, H)) return cudaErrorInvalidValue;
  m.a_sh = m.a;
  for (int h = 0; h < 5; ++h) m.b_sh[h] = m.b[h];
  TcParams p = {};
  p.T = T; p.H = H; p.E = E;
  p.rt_splits = splits;
  p.bias = bias;
  p.logits = logits;
  p.status = status;
  // The pair form (two 128-expert tiles per pair item) wherever E is a multiple
  // of 256 and the device runs it; MOE_TC_PAIR=0 (the diagnostic switch of the
  // grouped GEMMs) selects the single-SM form for comparison.
  const int npc = (E % 256 == 0 && pair_override() != 0) ? router_pair_clusters() : 0;
  if (npc > 0) {
    const int ptiles = E / 256;
    const bool split = router_split_k(T, E);
    p.rt_kparts = split ? RT_CHUNKS : 1;
    p.rt_partial = split ? (float *)((uint8_t *)scratch + round_up((int64_t)E * 3 * H * 2, 256)) : nullptr;
    const int per_tile = ptiles * p.rt_kparts;  // items per token tile
    const int want = std::max<int>((int)ceil_div(T, RT_NMAX),
                                   std::min<int>(std::max(npc / per_tile, 1), (int)ceil_div(T, RP_NROUND)));
    p.rt_rpt = (int)round_up(ceil_div(T, want), RP_NROUND);
    p.rt_ntile = (int)ceil_div(T, p.rt_rpt);
    p.n_items = per_tile * p.rt_ntile;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * std::min(p.n_items, npc));
    cfg.blockDim = dim3(RP_THREADS);
    cfg.dynamicSmemBytes = RP_SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute at[2];
    at[0].id = cudaLaunchAttributeClusterDimension;
    at[0].val.clusterDim.x = 2;
    at[0].val.clusterDim.y = 1;
    at[0].val.clusterDim.z = 1;
    at[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = at;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, tc_router_pair_kernel, m, p);
    if (e != cudaSuccess || !split) return e;
    const int64_t n = (int64_t)T * E;
    return launch_pdl(router_chunk_sum_kernel, dim3((unsigned)ceil_div(n / 4, 256)), dim3(256), 0, stream, n, E,
                      (const float *)p.rt_partial, bias, logits);
  }
  const int etiles = (int)ceil_div(E, 128), sms = device_sms();
  const int want = std::max<int>((int)ceil_div(T, RT_NMAX), std::min<int>(sms / etiles, (int)ceil_div(T, 16)));
  p.rt_rpt = (int)round_up(ceil_div(T, want), 16);
  p.rt_ntile = (int)ceil_div(T, p.rt_rpt);
  p.n_items = etiles * p.rt_ntile;
  e = ensure_smem((const void *)tc_router_kernel, TC_SMEM_BYTES);
  if (e != cudaSuccess) return e;
  const int grid = std::min(p.n_items, sms);
  return launch_pdl(tc_router_kernel, dim3(grid), dim3(RT_THREADS), TC_SMEM_BYTES, stream, m, p);
}

// Upper bound on the items of a grouped GEMM: sum_s ceil(n_s / 256) <=
// ceil(R / 256) + E over the routed segments, ceil(T / 256) for the shared one.
int64_t tc_max_items(int T, int k, int E, int nf_routed, int nf_shared) {
  return (ceil_div((int64_t)T * k, 256) + E) * nf_routed + ceil_div(T, 256) * nf_shared;
}
static int64_t max_items(int T, int k, int E, int nf_routed, int nf_shared) {
  return tc_max_items(T, k, E, nf_routed, nf_shared);
}

cudaError_t launch_item_tables(int E, int T, int nf_a_r, int nf_a_s, int nf_b_r, int nf_b_s, const int32_t *offsets,
                               int32_t *start_a, int32_t *start_b, int4 *items_a, int4 *items_b, int max_a,
                               int max_b, cudaStream_t stream, int e_begin, int e_end, int with_shared, int tile) {
  if (E > IT_MAX_E || tile < 16 || tile > 256 || tile % 16) return cudaErrorInvalidValue;
  if (e_end < 0) e_end = E;
  cudaError_t e = launch_pdl(item_tables_kernel, dim3(1), dim3(1024), 0, stream, E, T, nf_a_r, nf_a_s, nf_b_r, nf_b_s,
                             offsets, start_a, start_b, e_begin, e_end, with_shared, tile);
  if (e != cudaSuccess) return e;
  return launch_pdl(item_expand_kernel, dim3((unsigned)ceil_div((int64_t)(E + 1) * 32, 256)), dim3(256), 0, stream, E,
                    T, offsets, (const int32_t *)start_a, (const int32_t *)start_b, items_a, items_b, max_a, max_b,
                    tile);
}

static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

size_t ffn_tc_scratch_bytes(int T, int k, int E, int H, int I, int Is) {
  const size_t starts = round256((size_t)(E + 2) * 4);
  constexpr int DN_ROWS = 128 * TcCfg<TC_DOWN>::MT;  // output features per down item
  constexpr int GU_FEAT = 64 * TcCfg<TC_GATE_UP>::MT;  // features (gate + up row pairs) per gate_up item
  return 2 * starts + round256((size_t)max_items(T, k, E, I / GU_FEAT, Is / GU_FEAT) * 16) +
         round256((size_t)max_items(T, k, E, H / DN_ROWS, H / DN_ROWS) * 16);
}

// Where launch_ffn_tc keeps its item tables in `scratch` and how many items
// each row tile of a segment gives (none for the shared segment without
// with_shared; false: the call needs tables that the one-launch sort does not
// build, i.e. an expert range).
bool ffn_tc_item_tables(const FfnArgs &a, void *scratch, PermuteItems *it) {
  if (a.e_begin != 0 || (a.e_end >= 0 && a.e_end != a.E)) return false;
  const size_t starts = round256((size_t)(a.E + 2) * 4);
  constexpr int GU_FEAT = 64 * TcCfg<TC_GATE_UP>::MT;
  constexpr int DN_ROWS = 128 * TcCfg<TC_DOWN>::MT;
  const int mi_gu = (int)max_items(a.T, a.k, a.E, a.I / GU_FEAT, a.Is / GU_FEAT);
  const int mi_dn = (int)max_items(a.T, a.k, a.E, a.H / DN_ROWS, a.H / DN_ROWS);
  const int dn_rows = use_pair<TC_DOWN>(a) ? 256 : DN_ROWS;
  uint8_t *w = (uint8_t *)scratch;
  it->T = a.T;
  it->nf_a_r = a.I / GU_FEAT;
  it->nf_a_s = a.with_shared ? a.Is / GU_FEAT : 0;
  it->nf_b_r = a.H / dn_rows;
  it->nf_b_s = a.with_shared ? a.H / dn_rows : 0;
  it->max_a = mi_gu;
  it->max_b = mi_dn;
  it->start_a = (int32_t *)w;
  it->start_b = (int32_t *)(w + starts);
  it->items_a = (int4 *)(w + 2 * starts);
  it->items_b = (int4 *)(w + 2 * starts + round256((size_t)mi_gu * 16));
  return true;
}

cudaError_t launch_ffn_tc(const FfnArgs &a, void *scratch, int *status, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  const size_t starts = round256((size_t)(a.E + 2) * 4);
  constexpr int GU_FEAT = 64 * TcCfg<TC_GATE_UP>::MT;
  const int mi_gu = (int)max_items(a.T, a.k, a.E, a.I / GU_FEAT, a.Is / GU_FEAT);
  constexpr int DN_ROWS = 128 * TcCfg<TC_DOWN>::MT;
  const int mi_dn = (int)max_items(a.T, a.k, a.E, a.H / DN_ROWS, a.H / DN_ROWS);
  uint8_t *w = (uint8_t *)scratch;
  int32_t *start_gu = (int32_t *)w;
  int32_t *start_dn = (int32_t *)(w + starts);
  int4 *items_gu = (int4 *)(w + 2 * starts);
  int4 *items_dn = (int4 *)(w + 2 * starts + round256((size_t)mi_gu * 16));
  const int eb = a.e_begin, ee = a.e_end < 0 ? a.E : a.e_end, n_local = ee - eb;
  const bool gu_pair = use_pair<TC_GATE_UP>(a), dn_pair = use_pair<TC_DOWN>(a);
  const int dn_rows = dn_pair ? 256 : DN_ROWS;  // outputs per down item (a pair item is two M tiles)
  if (!a.items_ready) {
    cudaError_t e0 = launch_item_tables(a.E, a.T, a.I / GU_FEAT, a.Is / GU_FEAT, a.H / dn_rows, a.H / dn_rows,
                                        a.offsets, start_gu, start_dn, items_gu, items_dn, mi_gu, mi_dn, stream, eb, ee,
                                        a.with_shared);
    if (e0 != cudaSuccess) return e0;
  }
  const int64_t R = (int64_t)a.T * a.k;
  TcMaps mg, md;
  if (!map_gate_up(&mg.a, a.w_gate_up, std::max(n_local, 1), a.I, a.H, 4 * TcCfg<TC_GATE_UP>::MT) ||
      !map_gate_up(&mg.a_sh, a.ws_gate_up, 1, a.Is, a.H, 4 * TcCfg<TC_GATE_UP>::MT) ||
      !map_2d(&md.a, a.w_down, (int64_t)std::max(n_local, 1) * a.H, a.I, DN_ROWS) || !map_2d(&md.a_sh, a.ws_down, a.H, a.Is, DN_ROWS) ||
      !map_rows(md.b, a.h_routed, R, a.I) || !map_rows(md.b_sh, a.h_shared, a.T, a.Is))
    return cudaErrorInvalidValue;
  for (int h = 0; h < 5; ++h) mg.b[h] = mg.b_sh[h] = mg.a;  // gate_up gathers its token rows with cp.async
  TcParams p = {};
  p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k; p.I = a.I; p.Is = a.Is;
  p.offsets = a.offsets;
  p.sorted_route = a.sorted_route;
  p.x = (const __nv_bfloat16 *)a.x;
  p.h_routed = (__nv_bfloat16 *)a.h_routed;
  p.h_shared = (__nv_bfloat16 *)a.h_shared;
  p.gu_routed = (__nv_bfloat16 *)a.gu_routed;
  p.gu_shared = (__nv_bfloat16 *)a.gu_shared;
  p.y_routed = (__nv_bfloat16 *)a.y_routed;
  p.y_shared = (__nv_bfloat16 *)a.y_shared;
  p.e0 = eb;
  p.y_sorted = a.y_sorted;
  p.y_f32 = a.y_f32;
  p.status = status;
  const int grid = device_sms();
  p.item_start = start_gu;
  p.items = items_gu;
  cudaError_t e;
  if (gu_pair) {
    // One M tile (4 groups of 16 features) per CTA of the pair; x rows for
    // the gather4 copies through a one-row box.
    if (!map_gate_up(&mg.a, a.w_gate_up, std::max(n_local, 1), a.I, a.H, 4) ||
        !map_gate_up(&mg.a_sh, a.ws_gate_up, 1, a.Is, a.H, 4) || !map_2d(&mg.b[0], a.x, a.T, a.H, 1) ||
        (a.with_shared && !map_rows(mg.b_sh, a.x, a.T, a.H)))  // the shared expert's row boxes
      return cudaErrorInvalidValue;
    e = launch_pair<TC_GATE_UP>(mg, p, stream);
  } else {
    e = launch_tc<TC_GATE_UP>(mg, p, grid, stream);
  }
  if (e != cudaSuccess) return e;
  p.item_start = start_dn;
  p.items = items_dn;
  return dn_pair ? launch_pair<TC_DOWN>(md, p, stream) : launch_tc<TC_DOWN>(md, p, grid, stream);
}

}  // namespace moe
