// Expert-tensor-parallel slice with gate_up and down fused: h stays on chip.
//
// RL-Kernel PR #557 "What", bullet "Fail closed" (EP 1 = every expert
// expert-tensor-parallel over 4 ranks) and the embedded #503 commit message,
// bullets "Experts" and "TP4 block": a rank holds a slice of the intermediate
// dimension of every expert and computes, for every route, the FP32 partial
// sum of the down projection over its slice.  moe_grouped_ffn_etp does that
// with the two grouped GEMMs and the intermediate h [rows, slice] going
// through HBM between them; this kernel keeps h in shared memory instead.
//
// One 128-feature slice (the ETP tile of the bf16 kernels: I = 512 over four
// ranks), one SM per item, items = up to 128 rows of one segment:
//   phase 1  G[f, j] = W_gu[e][f] . x[tok(j)] for the slice's 128 gate and
//            128 up rows (two M tiles, 64 gate + 64 up rows each, interleaved
//            per 16 features), K = H; epilogue h = silu(g) * u rounded to
//            bf16, written into shared memory as the K-major, 128-byte
//            swizzled B operand of phase 2 (two K blocks of 64 features);
//   phase 2  D[o, j] = W_dn[e][o] . h[j] for H / 128 output tiles of 128,
//            K = 128; epilogue writes the FP32 accumulators unrounded to the
//            partial row (route order, or token order for the shared expert).
// The same arithmetic as the two-kernel path step for step (h rounded once
// with the same formula; every output one MMA chain over K in ascending
// order), so the partial rows equal moe_grouped_ffn_etp's bit for bit.
//
// Schedule: one sequence of stages per CTA, shared by the producer, the row
// gather and the MMA thread.  For the CTA's items i_0 .. i_{n-1}, round c
// (0 <= c <= n) runs, for each output tile t of H / 128: phase-1 K blocks
// 2t and 2t+1 of item i_c (c < n), then phase-2 tile t of item i_{c-1}
// (c >= 1).  So the tensor cores accumulate the next item's gate/up while
// the epilogue drains the current item's FP32 tiles.  The phase-1 accumulator of round c is committed after the
// round's last phase-2 MMA, so when the epilogue sees it, no MMA reads the
// previous item's h any more and it can be overwritten.
//
// TMEM: phase 1 at columns [0, 256) (M tile m at 128 m, N <= 128 rows),
// phase 2 alternates between [256, 384) and [384, 512).
// Roles: warp 0 TMA producer (weight tiles), warp 1 TMEM allocator + MMA
// issuer, EF_EPI_WARPS epilogue warps from warp 2 (EF_WPQ per TMEM lane
// quarter, EF_CPW columns each), then one warp that gathers the token rows of
// phase 1 with TMA gather4; the weight tile of a stage completes on full[s]
// (armed by the producer), its gathered rows on rows[s] (armed by the gather
// warp), so each issuing warp can wait for its own copies.  Every wait is
// bounded (2 s), records the device status word, and on a timeout each role
// waits for its own copies in flight before the CTA releases TMEM and exits.
// Measured slower than the two-kernel path (the bench's etp_slice entry):
// one SM per 128-row item fetches the slice's gate/up rows twice as often as
// the CTA-pair kernels, and the tensor pipe idles while phase 1's
// accumulator is turned into h.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"
#include "tc_host.h"
#include "umma.cuh"

namespace moe {

using namespace umma;

constexpr int EF_ROWS = 128;                     // rows per item (N of both GEMMs)
constexpr int EF_SLICE = 128;                    // features of the slice (I and Is)
constexpr int EF_STAGES = 4;
constexpr int EF_A_BYTES = 2 * 16384;            // phase 1: 256 gate/up rows x 64 K; phase 2: 128 outputs x 128 K
constexpr int EF_B_BYTES = EF_ROWS * 128;        // phase 1: 128 gathered rows x 64 K
constexpr int EF_STAGE_BYTES = EF_A_BYTES + EF_B_BYTES;
constexpr int EF_H_BYTES = 2 * EF_ROWS * 128;    // h: two K blocks of 128 rows x 64 features
// One gather warp issues the token rows of phase 1 as TMA gather4 copies
// (lane = a quad of four rows, 32 quads = 128 rows).
constexpr int EF_EPI_FIRST = 2, EF_EPI_WARPS = 16, EF_GATHER_WARPS = 1;
constexpr int EF_WPQ = EF_EPI_WARPS / 4;  // epilogue warps per TMEM lane quarter
constexpr int EF_CPW = EF_ROWS / EF_WPQ;  // accumulator columns (rows of the item) per epilogue warp
static_assert(EF_CPW == 64 || EF_CPW == 32, "one or two 32-column chunks per epilogue warp");
constexpr int EF_GATHER_FIRST = EF_EPI_FIRST + EF_EPI_WARPS;
constexpr int EF_THREADS = 32 * (EF_GATHER_FIRST + EF_GATHER_WARPS);
constexpr int EF_SMEM = 1024 + EF_STAGES * EF_STAGE_BYTES + EF_H_BYTES + 256;
static_assert(EF_SMEM <= 232448, "fused ETP shared memory");
constexpr uint32_t EF_TMEM_COLS = 512;

struct EfMaps {
  CUtensorMap gu, gu_sh;  // gate/up slices, 5-D boxes of 8 groups of 16 features (256 rows x 64 K)
  CUtensorMap dn, dn_sh;  // down slices [rows = outputs, 128 features], boxes 128 x 64
  CUtensorMap x;          // token rows, one-row boxes of 64 features (gather4)
};

struct EfParams {
  int T, H, E, k;
  const int32_t *sorted_route;
  const int32_t *item_start;  // [E+2] prefix of items per segment (shared last)
  const int4 *items;          // per item: segment, 0, first row, rows
  const __nv_bfloat16 *x;
  float *yr, *ys;             // FP32 partial rows [T k, H] (route order) and [T, H]
  int *status;
};

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ inline bool warp_wait_ef(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(FULL_MASK, ok, 0) != 0;
}

struct EfItem {
  int seg, rows, n;
  int64_t row0;
};

// Item `it` of this CTA's sequence: the shared segment's items first.
__device__ inline EfItem ef_item(int it, const EfParams &p) {
  const int routed = __ldg(p.item_start + p.E), total = __ldg(p.item_start + p.E + 1);
  const int n_sh = total - routed;
  const int4 d = __ldg(p.items + (it < n_sh ? routed + it : it - n_sh));
  EfItem r;
  r.seg = d.x;
  r.row0 = d.z;
  r.rows = d.w;
  r.n = (int)round_up(r.rows, 16);
  return r;
}

// h of one 32-column chunk of one phase-1 M tile into the shared h block:
// lanes 0-15 hold the gate values of features 16 q + lane, lanes 16-31 the
// up values of the same features, for columns (rows) c0 .. c0 + 31.  h =
// silu(g) * u, rounded to bf16; features (2m, 2m+1) of a row are packed into
// one word and stored at the row's 128-byte swizzled position.
__device__ __forceinline__ void ef_h_chunk(const float (&v)[32], int c0, int q, int lane, uint8_t *hblk) {
  float hv[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const float send = lane < 16 ? v[16 + j] : v[j];
    const float recv = __shfl_xor_sync(FULL_MASK, send, 16);
    const float g = lane < 16 ? v[j] : recv;
    const float u = lane < 16 ? recv : v[16 + j];
    hv[j] = __fdividef(g, 1.0f + __expf(-g)) * u;
  }
  const int fl = lane & 15, cbase = lane < 16 ? 0 : 16;
  const bool odd = lane & 1;
  const int chunk = 2 * q + (fl >> 3), off = 2 * (fl & 6);
#pragma unroll
  for (int j = 0; j < 16; j += 2) {
    const float xo = __shfl_xor_sync(FULL_MASK, odd ? hv[j] : hv[j + 1], 1);
    const __nv_bfloat162 w2 = odd ? __floats2bfloat162_rn(xo, hv[j + 1]) : __floats2bfloat162_rn(hv[j], xo);
    const int row = c0 + cbase + j + (odd ? 1 : 0);
    *(uint32_t *)(hblk + row * 128 + ((chunk ^ (row & 7)) << 4) + off) = *reinterpret_cast<const uint32_t *>(&w2);
  }
}

__global__ void __launch_bounds__(EF_THREADS, 1)
etp_fused_kernel(const __grid_constant__ EfMaps maps, const EfParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  auto sa = [&](int s) { return base + s * EF_STAGE_BYTES; };
  auto sb = [&](int s) { return base + s * EF_STAGE_BYTES + EF_A_BYTES; };
  uint8_t *hs = base + EF_STAGES * EF_STAGE_BYTES;  // h: K block 0 (features 0-63), then K block 1
  uint64_t *bars = (uint64_t *)(hs + EF_H_BYTES);
  uint64_t *full = bars, *empty = full + EF_STAGES;
  uint64_t *t1full = empty + EF_STAGES, *t1empty = t1full + 1, *hfull = t1empty + 1;
  uint64_t *t2full = hfull + 1, *t2empty = t2full + 2, *mma_done = t2empty + 2;
  uint64_t *rows = mma_done + 1;  // [EF_STAGES]: a phase-1 stage's gathered rows landed
  uint32_t *tmem_slot = (uint32_t *)(rows + EF_STAGES);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < EF_STAGES; ++s) {
      mbar_init(&full[s], 1);  // the producer's expect-tx arrival (weight tile bytes)
      mbar_init(&empty[s], 1);
      mbar_init(&rows[s], 1);  // the gather warp's expect-tx arrival (row bytes), phase-1 uses only
    }
    mbar_init(t1full, 1);
    mbar_init(t1empty, 32 * EF_EPI_WARPS);
    mbar_init(hfull, 32 * EF_EPI_WARPS);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&t2full[b], 1);
      mbar_init(&t2empty[b], 32 * EF_EPI_WARPS);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&maps.gu);
    prefetch_tmap(&maps.dn);
  }
  if (warp == 1) tmem_alloc(tmem_slot, EF_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  griddep_launch();
  griddep_wait();
  const int total = __ldg(p.item_start + p.E + 1);
  const int n_mine = total > (int)blockIdx.x ? (int)ceil_div(total - (int)blockIdx.x, gridDim.x) : 0;
  const int NT = p.H / 128;  // phase-2 output tiles per item = phase-1 K blocks / 2
  auto item_of = [&](int c) { return ef_item((int)blockIdx.x + c * (int)gridDim.x, p); };

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer (weight tiles)
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      int stage = 0;
      uint32_t phase = 0, issued = 0, issued_phase = 0;
      bool ok = true;
      for (int c = 0; c <= n_mine && ok; ++c) {
        const EfItem cur = c < n_mine ? item_of(c) : EfItem{}, prev = c > 0 ? item_of(c - 1) : EfItem{};
        const int nst = (c < n_mine ? 2 : 0) + (c > 0 ? 1 : 0);
        for (int t = 0; t < NT && ok; ++t) {
          for (int j = 0; j < nst; ++j) {
            const bool is_p1 = c < n_mine && j < 2;
            const EfItem im = is_p1 ? cur : prev;
            if (!mbar_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
            mbar_arrive_expect_tx(&full[stage], EF_A_BYTES);
            const bool sh = im.seg == p.E;
            if (is_p1) {  // K block 2t + j of the slice's 256 gate/up rows
              tma_load_5d(sa(stage), sh ? &maps.gu_sh : &maps.gu, &full[stage], (2 * t + j) * 64, 0, 0, 0,
                          sh ? 0 : im.seg, pol_w);
            } else {      // output tile t: its 128 rows of W_dn, both K blocks
              const int row = (sh ? 0 : im.seg * p.H) + t * 128;
              tma_load_2d(sa(stage), sh ? &maps.dn_sh : &maps.dn, &full[stage], 0, row, pol_w);
              tma_load_2d(sa(stage) + 16384, sh ? &maps.dn_sh : &maps.dn, &full[stage], 64, row, pol_w);
            }
            issued |= 1u << stage;
            issued_phase = (issued_phase & ~(1u << stage)) | (phase << stage);
            if (++stage == EF_STAGES) stage = 0, phase ^= 1;
          }
        }
      }
      if (!ok) {
        volatile int never = 0;
        for (int s = 0; s < EF_STAGES; ++s)
          if (issued & (1u << s)) mbar_wait(&full[s], (issued_phase >> s) & 1, &never, nullptr, 100000000ull);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0, cnt2 = 0, rphase = 0;  // rphase bit s: parity of rows[s]'s next phase-1 use
      bool ok = true;
      for (int c = 0; c <= n_mine && ok; ++c) {
        const EfItem cur = c < n_mine ? item_of(c) : EfItem{}, prev = c > 0 ? item_of(c - 1) : EfItem{};
        const uint32_t id1 = idesc_bf16_f32(128, c < n_mine ? cur.n : 16);
        const uint32_t id2 = idesc_bf16_f32(128, c > 0 ? prev.n : 16);
        if (c < n_mine) {  // the phase-1 accumulator is free (drained by the previous item's epilogue)
          if (!mbar_wait(t1empty, (c & 1) ^ 1, abort_flag, p.status)) break;
          tc_fence_after();
        }
        for (int t = 0; t < NT && ok; ++t) {
          if (c < n_mine) {
            for (int j = 0; j < 2 && ok; ++j) {
              const int kb = 2 * t + j;
              if (!mbar_wait(&full[stage], phase, abort_flag, p.status) ||
                  !mbar_wait(&rows[stage], (rphase >> stage) & 1, abort_flag, p.status)) { ok = false; break; }
              rphase ^= 1u << stage;
              tc_fence_after();
              const uint64_t bd = smem_desc_sw128(smem_u32(sb(stage)));
#pragma unroll
              for (int m = 0; m < 2; ++m) {
                const uint64_t ad = smem_desc_sw128(smem_u32(sa(stage) + m * 16384));
#pragma unroll
                for (int kk = 0; kk < 4; ++kk)
                  mma_bf16(tmem + m * 128, ad + 2 * kk, bd + 2 * kk, id1, (kb | kk) != 0);
              }
              mma_commit(&empty[stage]);
              if (++stage == EF_STAGES) stage = 0, phase ^= 1;
            }
          }
          if (ok && c > 0) {
            // The previous item's h is in shared memory (its epilogue ran
            // while the first phase-1 K blocks of this round were issued).
            if (t == 0 && !mbar_wait(hfull, (c - 1) & 1, abort_flag, p.status)) { ok = false; break; }
            const int b = cnt2 & 1;
            if (!mbar_wait(&t2empty[b], ((cnt2 >> 1) & 1) ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
            tc_fence_after();
#pragma unroll
            for (int kb = 0; kb < 2; ++kb) {  // K = the slice's 128 features: h K block kb
              const uint64_t ad = smem_desc_sw128(smem_u32(sa(stage) + kb * 16384));
              const uint64_t bd = smem_desc_sw128(smem_u32(hs + kb * (EF_H_BYTES / 2)));
#pragma unroll
              for (int kk = 0; kk < 4; ++kk)
                mma_bf16(tmem + 256 + b * 128, ad + 2 * kk, bd + 2 * kk, id2, (kb | kk) != 0);
            }
            mma_commit(&empty[stage]);
            mma_commit(&t2full[b]);
            ++cnt2;
            if (++stage == EF_STAGES) stage = 0, phase ^= 1;
          }
        }
        // Committed after the round's last phase-2 MMA: once it fires, the
        // previous item's h is no longer read and the next h may replace it.
        if (ok && c < n_mine) mma_commit(t1full);
      }
      mma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else if (warp < EF_GATHER_FIRST) {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3, part = (warp - EF_EPI_FIRST) >> 2;  // TMEM lane quarter, column part
    const uint32_t lane_off = (uint32_t)(q * 32) << 16;
    uint32_t cnt2 = 0;
    bool ok = true;
    for (int c = 0; c <= n_mine && ok; ++c) {
      if (c > 0) {
        // ---- phase 2 of item c-1: FP32 partial rows
        const EfItem im = item_of(c - 1);
        const bool sh = im.seg == p.E;
        float *yout = sh ? p.ys : p.yr;
        for (int t = 0; t < NT; ++t) {
          const int b = cnt2 & 1;
          if (!warp_wait_ef(&t2full[b], (cnt2 >> 1) & 1, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const int c0 = EF_CPW * part;
          float v0[32], v1[32];
          int d0 = 0, d1 = 0;
          if (c0 < im.n) {
            if (EF_CPW == 64)
              tmem_ld32x2(tmem + 256 + b * 128 + lane_off + c0, tmem + 256 + b * 128 + lane_off + c0 + 32, v0, v1);
            else
              tmem_ld32(tmem + 256 + b * 128 + lane_off + c0, v0);
            if (c0 + lane < im.rows)
              d0 = sh ? (int)(im.row0 + c0 + lane) : __ldg(p.sorted_route + im.row0 + c0 + lane);
            if (EF_CPW == 64 && c0 + 32 + lane < im.rows)
              d1 = sh ? (int)(im.row0 + c0 + 32 + lane) : __ldg(p.sorted_route + im.row0 + c0 + 32 + lane);
          }
          tc_fence_before();
          mbar_arrive(&t2empty[b]);
          ++cnt2;
          if (c0 < im.n) {
            const int ocol = t * 128 + q * 32;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int r0 = __shfl_sync(FULL_MASK, d0, j);
              if (c0 + j < im.rows) yout[(int64_t)r0 * p.H + ocol + lane] = v0[j];
              if (EF_CPW == 64) {
                const int r1 = __shfl_sync(FULL_MASK, d1, j);
                if (c0 + 32 + j < im.rows) yout[(int64_t)r1 * p.H + ocol + lane] = v1[j];
              }
            }
          }
        }
      }
      if (ok && c < n_mine) {
        // ---- phase 1 of item c: h into shared memory
        const EfItem im = item_of(c);
        if (!warp_wait_ef(t1full, c & 1, abort_flag, p.status)) break;
        tc_fence_after();
        // This warp's 64 columns, one 32-column chunk of both M tiles at a
        // time (M tile m holds the slice's features 64 m .. 64 m + 63, i.e.
        // h K block m); the accumulator is released after the last load.
        bool released = false;
        for (int cc = 0; cc < EF_CPW / 32; ++cc) {
          const int c0 = EF_CPW * part + 32 * cc;
          if (c0 < im.n) {
#pragma unroll
            for (int m = 0; m < 2; ++m) {  // M tile m: features 64 m .. 64 m + 63 = h K block m
              float v[32];
              tmem_ld32(tmem + m * 128 + lane_off + c0, v);
              if (m == 1 && (cc == EF_CPW / 32 - 1 || c0 + 32 >= im.n)) {  // this warp's last load is done
                tc_fence_before();
                mbar_arrive(t1empty);
                released = true;
              }
              ef_h_chunk(v, c0, q, lane, hs + m * (EF_H_BYTES / 2));
            }
          }
        }
        if (!released) {  // no columns of this warp in the item
          tc_fence_before();
          mbar_arrive(t1empty);
        }
        fence_proxy_async_smem();  // h: generic writes -> async proxy (the MMA reads it)
        mbar_arrive(hfull);
      }
    }
  } else {
    // ------------------------------------------------------------ row gather (phase 1)
    // Lane qd copies rows 4 qd .. 4 qd + 3 of the item (one gather4 per
    // K block, landing as four consecutive 128-byte swizzled lines at 512 qd;
    // the bytes complete on the stage's rows barrier, armed here with the
    // item's n x 128 bytes).  Rows past the item's end up to n read token 0:
    // their accumulator columns are never stored.
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0, rphase = 0, issued = 0, issued_rphase = 0;
    bool ok = true;
    for (int c = 0; c <= n_mine && ok; ++c) {
      const EfItem cur = c < n_mine ? item_of(c) : EfItem{};
      const bool mine = c < n_mine && 4 * lane < cur.n;
      int t4[4] = {0, 0, 0, 0};
      if (mine) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int r = 4 * lane + j;
          if (r < cur.rows) {
            const int64_t row = cur.row0 + r;
            t4[j] = cur.seg == p.E ? (int)row : __ldg(p.sorted_route + row) / p.k;
          }
        }
      }
      const int nst = (c < n_mine ? 2 : 0) + (c > 0 ? 1 : 0);
      for (int t = 0; t < NT && ok; ++t) {
        for (int j = 0; j < nst; ++j) {
          if (c < n_mine && j < 2) {
            if (!warp_wait_ef(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
            if (lane == 0) mbar_arrive_expect_tx(&rows[stage], (uint32_t)cur.n * 128);
            __syncwarp();
            if (mine)
              tma_gather4(sb(stage) + lane * 512, &maps.x, &rows[stage], (2 * t + j) * 64, t4[0], t4[1], t4[2], t4[3],
                          pol_x);
            issued |= 1u << stage;
            issued_rphase = (issued_rphase & ~(1u << stage)) | (rphase & (1u << stage));
            rphase ^= 1u << stage;
          }
          if (++stage == EF_STAGES) stage = 0, phase ^= 1;
        }
      }
    }
    if (!ok && lane == 0) {
      // The row copies in flight land before the CTA exits.
      volatile int never = 0;
      for (int s2 = 0; s2 < EF_STAGES; ++s2)
        if (issued & (1u << s2)) mbar_wait(&rows[s2], (issued_rphase >> s2) & 1, &never, nullptr, 100000000ull);
    }
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, EF_TMEM_COLS);
}

// ---------------------------------------------------------------- host side
size_t etp_fused_scratch_bytes(int T, int k, int E) {
  const size_t starts = (size_t)round_up((int64_t)(E + 2) * 4, 256);
  const int64_t items = ceil_div((int64_t)T * k, EF_ROWS) + E + ceil_div(T, EF_ROWS);
  return 2 * starts + (size_t)round_up(items * 16, 256);
}

bool etp_fused_supported(int H, int I, int Is) { return I == EF_SLICE && Is == EF_SLICE && H % 128 == 0; }

cudaError_t launch_etp_fused(const FfnArgs &a, void *scratch, int *status, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  if (!etp_fused_supported(a.H, a.I, a.Is)) return cudaErrorInvalidValue;
  const size_t starts = (size_t)round_up((int64_t)(a.E + 2) * 4, 256);
  const int64_t max_items = ceil_div((int64_t)a.T * a.k, EF_ROWS) + a.E + ceil_div(a.T, EF_ROWS);
  uint8_t *w = (uint8_t *)scratch;
  int32_t *start = (int32_t *)w, *start_unused = (int32_t *)(w + starts);
  int4 *items = (int4 *)(w + 2 * starts);
  cudaError_t e = launch_item_tables(a.E, a.T, 1, 1, 0, 0, a.offsets, start, start_unused, items, items,
                                     (int)max_items, 0, stream, 0, a.E, 1, EF_ROWS);
  if (e != cudaSuccess) return e;
  EfMaps m;
  if (!map_gate_up(&m.gu, a.w_gate_up, a.E, EF_SLICE, a.H, 8) || !map_gate_up(&m.gu_sh, a.ws_gate_up, 1, EF_SLICE, a.H, 8) ||
      !map_2d(&m.dn, a.w_down, (int64_t)a.E * a.H, EF_SLICE, 128) || !map_2d(&m.dn_sh, a.ws_down, a.H, EF_SLICE, 128) ||
      !map_2d(&m.x, a.x, a.T, a.H, 1))
    return cudaErrorInvalidValue;
  EfParams p = {};
  p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k;
  p.sorted_route = a.sorted_route;
  p.item_start = start;
  p.items = items;
  p.x = (const __nv_bfloat16 *)a.x;
  p.yr = (float *)a.y_routed;
  p.ys = (float *)a.y_shared;
  p.status = status;
  if ((e = ensure_smem((const void *)etp_fused_kernel, EF_SMEM)) != cudaSuccess) return e;
  return launch_pdl(etp_fused_kernel, dim3(device_sms()), dim3(EF_THREADS), EF_SMEM, stream, m, p);
}

}  // namespace moe
