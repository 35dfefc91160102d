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
//            (Wr = W1 + W2 + W3, every product exact); epilogue adds the bias
//            and writes logits[t, e] in FP32.
//   GATE_UP  D[f, j] = W_gu[e][f] . x[tok(j)] for the 64 gate and 64 up rows
//            of a feature tile and up to 256 rows j of expert e's segment
//            (x rows gathered by TMA gather4); epilogue h = silu(g) * u.
//   DOWN     D[o, j] = W_dn[e][o] . h[j] for 128 output features; epilogue
//            writes row j to y_routed[sorted_route[j]] (or y_shared).
// The weights are the M = 128 operand and the tokens the N <= 256 operand,
// so a short expert segment costs at most 15 padded columns.  Every output
// element is one FP32 accumulation over K in a fixed order (K blocks of 64,
// four K = 16 MMAs each); tiling decides only where a column sits, never the
// order, so a token's values do not depend on T or on its segment.
//
// Roles (192 threads): warp 0 issues TMA loads into a 4-stage ring; warp 1
// allocates 512 TMEM columns (two 256-column accumulators) and one thread
// issues the MMAs; warps 2-5 drain an accumulator (each warp its 32-lane
// quarter of TMEM) while the next item accumulates in the other buffer.
#include <cuda.h>

#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "kernels.h"
#include "umma.cuh"

namespace moe {

using namespace umma;

constexpr int TC_STAGES = 4;
constexpr int TC_NMAX = 256;
constexpr int TC_A_BYTES = 128 * 128;      // 128 rows x 64 bf16
constexpr int TC_B_BYTES = TC_NMAX * 128;  // 256 rows x 64 bf16
constexpr int TC_THREADS = 192;
constexpr int TC_SMEM_BYTES = 1024 + TC_STAGES * (TC_A_BYTES + TC_B_BYTES) + 256;
constexpr uint32_t TC_TMEM_COLS = 512;

enum { TC_ROUTER = 0, TC_GATE_UP = 1, TC_DOWN = 2 };

struct TcParams {
  int T, H, E, k, I, Is;
  int n_items;  // ROUTER: number of items; others read item_start[E+1]
  const int32_t *offsets;
  const int32_t *sorted_route;
  const int32_t *item_start;
  const float *bias;
  float *logits;
  __nv_bfloat16 *h_routed, *h_shared;
  __nv_bfloat16 *gu_routed, *gu_shared;
  __nv_bfloat16 *y_routed, *y_shared;
  int *status;
};

struct Item {
  int seg;       // expert segment (E = shared); ROUTER: unused
  int f;         // M tile: expert tile (ROUTER), feature tile (GATE_UP, DOWN)
  int64_t row0;  // first row of the N tile (token for ROUTER / shared, sorted row otherwise)
  int rows;      // valid rows in the tile
  int n;         // MMA N = rows rounded up to 16
  int nk;        // K blocks of 64
};

// Rows of a segment are cut into ceil(n/256) tiles of equal size rounded up
// to 16; the cut depends only on the segment's own length.
template <int MODE>
__device__ inline Item decode_item(int it, const TcParams &p) {
  Item r;
  if (MODE == TC_ROUTER) {
    const int ntile = (int)ceil_div(p.T, TC_NMAX);
    const int rpt = (int)round_up(ceil_div(p.T, ntile), 16);
    const int nt = it % ntile;
    r.seg = 0;
    r.f = it / ntile;
    r.row0 = (int64_t)nt * rpt;
    r.rows = min(rpt, p.T - nt * rpt);
    r.nk = 3 * p.H / 64;
  } else {
    int lo = 0, hi = p.E;
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (__ldg(p.item_start + mid) <= it) lo = mid;
      else hi = mid - 1;
    }
    const bool sh = lo == p.E;
    const int local = it - __ldg(p.item_start + lo);
    const int64_t base = sh ? 0 : __ldg(p.offsets + lo);
    const int n_s = sh ? p.T : __ldg(p.offsets + lo + 1) - (int)base;
    const int ntile = (int)ceil_div(n_s, TC_NMAX);
    const int rpt = (int)round_up(ceil_div(n_s, ntile), 16);
    const int nt = local % ntile;
    r.seg = lo;
    r.f = local / ntile;
    r.row0 = base + (int64_t)nt * rpt;
    r.rows = min(rpt, n_s - nt * rpt);
    r.nk = (MODE == TC_GATE_UP ? p.H : (sh ? p.Is : p.I)) / 64;
  }
  r.n = (int)round_up(r.rows, 16);
  return r;
}

// Warp-uniform bounded wait: lane 0 polls, the verdict is broadcast.
__device__ inline bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, int *status) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mbar_wait(bar, parity, abort_flag, status) ? 1 : 0;
  return __shfl_sync(FULL_MASK, ok, 0) != 0;
}

template <int MODE>
__global__ void __launch_bounds__(TC_THREADS, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_a_sh,
               const __grid_constant__ CUtensorMap map_b, const __grid_constant__ CUtensorMap map_b_sh,
               const TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
  uint8_t *sa = base;
  uint8_t *sb = base + TC_STAGES * TC_A_BYTES;
  uint64_t *bars = (uint64_t *)(sb + TC_STAGES * TC_B_BYTES);
  uint64_t *full = bars, *empty = bars + TC_STAGES;
  uint64_t *tfull = bars + 2 * TC_STAGES, *tempty = tfull + 2, *mma_done = tempty + 2;
  uint32_t *tmem_slot = (uint32_t *)(mma_done + 1);
  volatile int *abort_flag = (volatile int *)(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < TC_STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 128);
    }
    mbar_init(mma_done, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&map_a);
    prefetch_tmap(&map_b);
    if (MODE != TC_ROUTER) {
      prefetch_tmap(&map_a_sh);
      if (MODE == TC_DOWN) prefetch_tmap(&map_b_sh);
    }
  }
  if (warp == 1) tmem_alloc(tmem_slot, TC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = MODE == TC_ROUTER ? p.n_items : __ldg(p.item_start + p.E + 1);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    int stage = 0;
    uint32_t phase = 0;
    int issued[TC_STAGES];
    uint32_t issued_phase[TC_STAGES];
#pragma unroll
    for (int s = 0; s < TC_STAGES; ++s) issued[s] = 0, issued_phase[s] = 0;
    bool ok = true;
    for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
      const Item im = decode_item<MODE>(it, p);
      const bool sh = MODE != TC_ROUTER && im.seg == p.E;
      int gidx[2][4];
      if (MODE == TC_GATE_UP) {
#pragma unroll
        for (int q = 0; q < 2; ++q)
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            int r = (lane + 32 * q) * 4 + j;
            r = r < im.rows ? r : im.rows - 1;  // pad columns repeat the last row
            const int64_t row = im.row0 + r;
            gidx[q][j] = sh ? (int)row : __ldg(p.sorted_route + row) / p.k;
          }
      }
      const int b_boxes = (int)ceil_div(im.n, 32);
      const uint32_t bytes = TC_A_BYTES + (MODE == TC_GATE_UP ? im.n * 128 : b_boxes * 32 * 128);
      for (int kb = 0; kb < im.nk; ++kb) {
        if (!warp_wait(&empty[stage], phase ^ 1, abort_flag, p.status)) { ok = false; break; }
        uint8_t *a_dst = sa + stage * TC_A_BYTES;
        uint8_t *b_dst = sb + stage * TC_B_BYTES;
        if (lane == 0) {
          mbar_arrive_expect_tx(&full[stage], bytes);
          if (MODE == TC_ROUTER) {
            tma_load_2d(a_dst, &map_a, &full[stage], kb * 64, im.f * 128);
          } else if (MODE == TC_GATE_UP) {
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tma_load_3d(a_dst + b * 4096, sh ? &map_a_sh : &map_a, &full[stage], kb * 64, im.f * 64 + 16 * b,
                          sh ? 0 : 2 * im.seg);
          } else {
            tma_load_2d(a_dst, sh ? &map_a_sh : &map_a, &full[stage], kb * 64,
                        sh ? im.f * 128 : im.seg * p.H + im.f * 128);
          }
        }
        __syncwarp();
        if (MODE == TC_GATE_UP) {
          const int n_ops = im.n / 4;
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            const int g = lane + 32 * q;
            if (g < n_ops)
              tma_gather4(b_dst + g * 512, &map_b, &full[stage], kb * 64, gidx[q][0], gidx[q][1], gidx[q][2],
                          gidx[q][3]);
          }
        } else if (lane < b_boxes) {
          const int kx = MODE == TC_ROUTER ? (kb % (p.H / 64)) * 64 : kb * 64;
          tma_load_2d(b_dst + lane * 4096, (MODE == TC_DOWN && sh) ? &map_b_sh : &map_b, &full[stage], kx,
                      (int)(im.row0 + 32 * lane));
        }
        issued[stage] = 1;
        issued_phase[stage] = phase;
        if (++stage == TC_STAGES) stage = 0, phase ^= 1;
      }
    }
    if (!ok && lane == 0) {
      // Let the copies already in flight land before the CTA exits.
      volatile int never = 0;
      for (int s = 0; s < TC_STAGES; ++s)
        if (issued[s]) mbar_wait(&full[s], issued_phase[s], &never, nullptr, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int it = blockIdx.x; it < total && ok; it += gridDim.x) {
        const Item im = decode_item<MODE>(it, p);
        if (!mbar_wait(&tempty[acc], acc_phase ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t d = tmem + acc * TC_NMAX;
        const uint32_t idesc = idesc_bf16_f32(128, im.n);
        for (int kb = 0; kb < im.nk; ++kb) {
          if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
          tc_fence_after();
          const uint64_t ad = smem_desc_sw128(smem_u32(sa + stage * TC_A_BYTES));
          const uint64_t bd = smem_desc_sw128(smem_u32(sb + stage * TC_B_BYTES));
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 16 per MMA: +32 bytes = +2 in the descriptor address field
            mma_bf16(d, ad + 2 * kk, bd + 2 * kk, idesc, (kb | kk) != 0);
          mma_commit(&empty[stage]);
          if (++stage == TC_STAGES) stage = 0, phase ^= 1;
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
        if (++acc == 2) acc = 0, acc_phase ^= 1;
      }
      // Every MMA this thread issued has finished before TMEM is released.
      mma_commit(mma_done);
      volatile int never = 0;
      mbar_wait(mma_done, 0, &never, p.status);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int it = blockIdx.x; it < total; it += gridDim.x) {
      const Item im = decode_item<MODE>(it, p);
      if (!warp_wait(&tfull[acc], acc_phase, abort_flag, p.status)) break;
      tc_fence_after();
      const uint32_t tb = tmem + acc * TC_NMAX + ((uint32_t)(q * 32) << 16);
      if (MODE == TC_ROUTER) {
        const int e = im.f * 128 + q * 32 + lane;
        const float b = (p.bias && e < p.E) ? __ldg(p.bias + e) : 0.f;
        for (int c0 = 0; c0 < im.n; c0 += 32) {
          float v[32];
          tmem_ld32(tb + c0, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int c = c0 + j;
            if (c < im.rows && e < p.E) {
              float val = v[j];
              if (p.bias) val += b;
              p.logits[(im.row0 + c) * p.E + e] = val;
            }
          }
        }
      } else if (MODE == TC_GATE_UP) {
        const bool sh = im.seg == p.E;
        const int Iseg = sh ? p.Is : p.I;
        const int f = im.f * 64 + 16 * q + (lane & 15);
        __nv_bfloat16 *hout = sh ? p.h_shared : p.h_routed;
        __nv_bfloat16 *guout = sh ? p.gu_shared : p.gu_routed;
        for (int c0 = 0; c0 < im.n; c0 += 32) {
          float v[32];
          tmem_ld32(tb + c0, v);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            // lanes 0-15 hold gate values, lanes 16-31 the up values of the same features
            const float other = __shfl_xor_sync(FULL_MASK, v[j], 16);
            const int c = c0 + j;
            if (c < im.rows) {
              const int64_t row = im.row0 + c;
              if (lane < 16) hout[row * Iseg + f] = __float2bfloat16_rn(silu_f32(v[j]) * other);
              if (guout) guout[row * 2 * Iseg + (lane < 16 ? 0 : Iseg) + f] = __float2bfloat16_rn(v[j]);
            }
          }
        }
      } else {
        const bool sh = im.seg == p.E;
        const int o = im.f * 128 + q * 32 + lane;
        for (int c0 = 0; c0 < im.n; c0 += 32) {
          float v[32];
          tmem_ld32(tb + c0, v);
          int my_dst = 0;
          if (c0 + lane < im.rows) my_dst = sh ? (int)(im.row0 + c0 + lane) : __ldg(p.sorted_route + im.row0 + c0 + lane);
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int dst = __shfl_sync(FULL_MASK, my_dst, j);
            if (c0 + j < im.rows) {
              __nv_bfloat16 *yrow = (sh ? p.y_shared : p.y_routed) + (int64_t)dst * p.H;
              yrow[o] = __float2bfloat16_rn(v[j]);
            }
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&tempty[acc]);
      if (++acc == 2) acc = 0, acc_phase ^= 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, TC_TMEM_COLS);
}

// ---------------------------------------------------------------------------
// Exact three-way bf16 split of the FP32 router weight: Wr3[e] = [W1 | W2 | W3]
// with W1 = rn(w), W2 = rn(w - W1), W3 = rn(w - W1 - W2).  Each residual is
// exact in FP32 and holds at most 16 then 8 significant bits, so W3 captures
// the rest and W1 + W2 + W3 = w exactly.
// ---------------------------------------------------------------------------
__global__ void split_router_weight_kernel(int64_t n, int H, const float *__restrict__ wr,
                                           __nv_bfloat16 *__restrict__ wr3) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int64_t e = i / H, h = i % H;
  const float w = wr[i];
  const __nv_bfloat16 w1 = __float2bfloat16_rn(w);
  const float r1 = w - __bfloat162float(w1);
  const __nv_bfloat16 w2 = __float2bfloat16_rn(r1);
  const float r2 = r1 - __bfloat162float(w2);
  const __nv_bfloat16 w3 = __float2bfloat16_rn(r2);
  __nv_bfloat16 *row = wr3 + e * 3 * H;
  row[h] = w1;
  row[H + h] = w2;
  row[2 * H + h] = w3;
}

// item_start[s] = sum_{s' < s} ceil(n_s' / 256) * nf_s', routed segments
// with nf_routed feature tiles, the shared segment (n = T) with nf_shared.
__global__ void __launch_bounds__(1024)
build_items_kernel(int E, int T, int nf_routed, int nf_shared, const int32_t *__restrict__ offsets,
                   int32_t *__restrict__ item_start) {
  __shared__ int32_t buf[1024];
  __shared__ int32_t carry;
  if (threadIdx.x == 0) carry = 0;
  __syncthreads();
  for (int base = 0; base <= E; base += 1024) {
    const int s = base + threadIdx.x;
    int32_t v = 0;
    if (s < E) v = (int32_t)ceil_div(offsets[s + 1] - offsets[s], TC_NMAX) * nf_routed;
    else if (s == E) v = (int32_t)ceil_div(T, TC_NMAX) * nf_shared;
    buf[threadIdx.x] = v;
    __syncthreads();
    for (int d = 1; d < 1024; d <<= 1) {
      int32_t add = (int)threadIdx.x >= d ? buf[threadIdx.x - d] : 0;
      __syncthreads();
      buf[threadIdx.x] += add;
      __syncthreads();
    }
    if (s <= E) item_start[s] = carry + buf[threadIdx.x] - v;
    if (s == E) item_start[E + 1] = carry + buf[threadIdx.x];
    __syncthreads();
    if (threadIdx.x == 1023) carry += buf[1023];
    __syncthreads();
  }
}

// ---------------------------------------------------------------- host side
using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (EncodeTiledFn)p;
  });
  return fn;
}

// bf16 tensor map, 128-byte swizzle, box inner width 64 elements.
static bool encode_map(CUtensorMap *m, const void *ptr, int rank, const uint64_t *dims, const uint64_t *strides_bytes,
                       const uint32_t *box) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t gd[5], gs[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    gd[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) gs[i] = strides_bytes[i];
  }
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, (cuuint32_t)rank, const_cast<void *>(ptr), gd, gs, bx, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Row-major [rows, cols] matrix, box = box_rows x 64.
static bool map_2d(CUtensorMap *m, const void *ptr, int64_t rows, int64_t cols, uint32_t box_rows) {
  const uint64_t dims[2] = {(uint64_t)cols, (uint64_t)rows};
  const uint64_t strides[1] = {(uint64_t)cols * 2};
  const uint32_t box[2] = {64, box_rows};
  return encode_map(m, ptr, 2, dims, strides, box);
}

// Gate/up weights [n_mat, 2*Iw, H] viewed as (H, Iw, 2*n_mat): box (64, 16, 2)
// = 16 gate rows followed by the 16 up rows of the same features.
static bool map_gate_up(CUtensorMap *m, const void *ptr, int n_mat, int Iw, int H) {
  const uint64_t dims[3] = {(uint64_t)H, (uint64_t)Iw, (uint64_t)2 * n_mat};
  const uint64_t strides[2] = {(uint64_t)H * 2, (uint64_t)Iw * H * 2};
  const uint32_t box[3] = {64, 16, 2};
  return encode_map(m, ptr, 3, dims, strides, box);
}

struct DevInfo {
  int sms = 0;
  bool attr[3] = {false, false, false};
};

static DevInfo &dev_info() {
  static std::mutex mu;
  static DevInfo info[64];
  int dev = 0;
  cudaGetDevice(&dev);
  std::lock_guard<std::mutex> lock(mu);
  DevInfo &d = info[dev & 63];
  if (!d.sms) cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
  return d;
}

template <int MODE>
static cudaError_t launch_tc(const CUtensorMap &a, const CUtensorMap &a_sh, const CUtensorMap &b,
                             const CUtensorMap &b_sh, const TcParams &p, int grid, cudaStream_t stream) {
  DevInfo &di = dev_info();
  if (!di.attr[MODE]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TC_SMEM_BYTES);
    if (e != cudaSuccess) return e;
    di.attr[MODE] = true;
  }
  tc_gemm_kernel<MODE><<<grid, TC_THREADS, TC_SMEM_BYTES, stream>>>(a, a_sh, b, b_sh, p);
  return cudaGetLastError();
}

size_t router_tc_scratch_bytes(int E, int H) { return (size_t)E * 3 * H * 2; }

cudaError_t launch_router_logits_tc(int T, int H, int E, const void *x, const float *wr, const float *bias,
                                    float *logits, void *scratch, int *status, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  __nv_bfloat16 *wr3 = (__nv_bfloat16 *)scratch;
  const int64_t n = (int64_t)E * H;
  split_router_weight_kernel<<<(unsigned)ceil_div(n, 256), 256, 0, stream>>>(n, H, wr, wr3);
  CUtensorMap ma, mb;
  if (!map_2d(&ma, wr3, E, 3 * (int64_t)H, 128) || !map_2d(&mb, x, T, H, 32)) return cudaErrorInvalidValue;
  TcParams p = {};
  p.T = T; p.H = H; p.E = E;
  p.n_items = (int)(ceil_div(E, 128) * ceil_div(T, TC_NMAX));
  p.bias = bias;
  p.logits = logits;
  p.status = status;
  const int grid = std::min(p.n_items, dev_info().sms);
  return launch_tc<TC_ROUTER>(ma, ma, mb, mb, p, grid, stream);
}

size_t ffn_tc_scratch_bytes(int E) { return (size_t)2 * 256 * (((E + 2) * 4 + 255) / 256); }

cudaError_t launch_ffn_tc(const FfnArgs &a, void *scratch, int *status, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  int32_t *items_gu = (int32_t *)scratch;
  int32_t *items_dn = items_gu + round_up(a.E + 2, 64);
  build_items_kernel<<<1, 1024, 0, stream>>>(a.E, a.T, a.I / 64, a.Is / 64, a.offsets, items_gu);
  build_items_kernel<<<1, 1024, 0, stream>>>(a.E, a.T, a.H / 128, a.H / 128, a.offsets, items_dn);
  const int64_t R = (int64_t)a.T * a.k;
  CUtensorMap a_gu, a_gu_sh, b_x, a_dn, a_dn_sh, b_h, b_h_sh;
  if (!map_gate_up(&a_gu, a.w_gate_up, a.E, a.I, a.H) || !map_gate_up(&a_gu_sh, a.ws_gate_up, 1, a.Is, a.H) ||
      !map_2d(&b_x, a.x, a.T, a.H, 1) || !map_2d(&a_dn, a.w_down, (int64_t)a.E * a.H, a.I, 128) ||
      !map_2d(&a_dn_sh, a.ws_down, a.H, a.Is, 128) || !map_2d(&b_h, a.h_routed, R, a.I, 32) ||
      !map_2d(&b_h_sh, a.h_shared, a.T, a.Is, 32))
    return cudaErrorInvalidValue;
  TcParams p = {};
  p.T = a.T; p.H = a.H; p.E = a.E; p.k = a.k; p.I = a.I; p.Is = a.Is;
  p.offsets = a.offsets;
  p.sorted_route = a.sorted_route;
  p.h_routed = (__nv_bfloat16 *)a.h_routed;
  p.h_shared = (__nv_bfloat16 *)a.h_shared;
  p.gu_routed = (__nv_bfloat16 *)a.gu_routed;
  p.gu_shared = (__nv_bfloat16 *)a.gu_shared;
  p.y_routed = (__nv_bfloat16 *)a.y_routed;
  p.y_shared = (__nv_bfloat16 *)a.y_shared;
  p.status = status;
  const int grid = dev_info().sms;
  p.item_start = items_gu;
  cudaError_t e = launch_tc<TC_GATE_UP>(a_gu, a_gu_sh, b_x, b_x, p, grid, stream);
  if (e != cudaSuccess) return e;
  p.item_start = items_dn;
  return launch_tc<TC_DOWN>(a_dn, a_dn_sh, b_h, b_h_sh, p, grid, stream);
}

}  // namespace moe
