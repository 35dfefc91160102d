// Grouped SwiGLU FFN on CUDA cores (the MOE_F32 path: FP32 has no tensor-core
// format that keeps the 1e-4 bar, so FP32 products are summed on CUDA cores).
//
// RL-Kernel PR #557, embedded #503 commit message, bullet "Experts":
// per-route gate_up and down projections through one fixed-configuration
// grouped GEMM; no routed-weight multiply and no sum inside the kernel, so
// every (token, route) row has exactly one writer.  The shared expert runs
// as segment E over all T tokens.
//
// Every output element is accumulated by one thread with fmaf over the
// reduction index in ascending order; tiling only decides which thread does
// it, so a row's value does not depend on its segment, its tile or T.
#include "common.cuh"
#include "kernels.h"

namespace moe {

constexpr int SIMT_BM = 32;  // rows per tile
constexpr int SIMT_BK = 32;  // reduction step staged in shared memory

size_t ffn_simt_scratch_bytes(int E) { return (size_t)(E + 2) * sizeof(int32_t); }

struct TileRows {
  int seg;         // segment (E = shared)
  int64_t r0, r1;  // rows [r0, r1) of the segment's row space
};

// Segment of tile `ti`: the largest s with tile_start[s] <= ti.
__device__ inline TileRows decode_tile(int ti, int E, int T, const int32_t *tile_start, const int32_t *offsets) {
  int lo = 0, hi = E;  // answer in [0, E]
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= ti) lo = mid;
    else hi = mid - 1;
  }
  TileRows tr;
  tr.seg = lo;
  int i = ti - tile_start[lo];
  if (lo < E) {
    tr.r0 = offsets[lo] + (int64_t)i * SIMT_BM;
    tr.r1 = min((int64_t)offsets[lo + 1], tr.r0 + SIMT_BM);
  } else {
    tr.r0 = (int64_t)i * SIMT_BM;
    tr.r1 = min((int64_t)T, tr.r0 + SIMT_BM);
  }
  return tr;
}

// gate_up + SwiGLU: tile of 32 rows x 32 features; thread (ty, tx) owns rows
// 2ty, 2ty+1 and features 2tx, 2tx+1 (gate and up for each).
template <typename TE>
__global__ void __launch_bounds__(256) ffn_gate_up_simt_kernel(FfnArgs a, const int32_t *__restrict__ tile_start) {
  griddep_launch();
  griddep_wait();
  __shared__ float xs[SIMT_BK][SIMT_BM + 1];
  __shared__ float wg[SIMT_BK][33];
  __shared__ float wu[SIMT_BK][33];
  __shared__ int64_t tok[SIMT_BM];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int total = tile_start[a.E + 1];
  const TE *x = (const TE *)a.x;
  for (int ti = blockIdx.x; ti < total; ti += gridDim.x) {
    TileRows tr = decode_tile(ti, a.E, a.T, tile_start, a.offsets);
    const bool shared = tr.seg == a.E;
    const int Iseg = shared ? a.Is : a.I;
    const int f0 = blockIdx.y * 32;
    if (f0 >= Iseg) continue;  // uniform over the block
    const TE *wgu =
        shared ? (const TE *)a.ws_gate_up : (const TE *)a.w_gate_up + (int64_t)(tr.seg - a.e_begin) * 2 * a.I * a.H;
    if (threadIdx.x < SIMT_BM) {
      int64_t j = tr.r0 + threadIdx.x;
      tok[threadIdx.x] = j < tr.r1 ? (shared ? j : (int64_t)(a.sorted_route[j] / a.k)) : -1;
    }
    __syncthreads();
    float g[2][2] = {{0.f, 0.f}, {0.f, 0.f}}, u[2][2] = {{0.f, 0.f}, {0.f, 0.f}};
    for (int h0 = 0; h0 < a.H; h0 += SIMT_BK) {
      for (int i = threadIdx.x; i < SIMT_BM * SIMT_BK; i += 256) {
        int r = i / SIMT_BK, c = i % SIMT_BK, h = h0 + c;
        int64_t t = tok[r];
        xs[c][r] = (t >= 0 && h < a.H) ? Elem<TE>::load(x + t * a.H + h) : 0.f;
        int f = f0 + r;  // 32 features, same index range as rows
        bool ok = f < Iseg && h < a.H;
        wg[c][r] = ok ? Elem<TE>::load(wgu + (int64_t)f * a.H + h) : 0.f;
        wu[c][r] = ok ? Elem<TE>::load(wgu + (int64_t)(Iseg + f) * a.H + h) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < SIMT_BK; ++kk) {
        float xv0 = xs[kk][2 * ty], xv1 = xs[kk][2 * ty + 1];
        float g0 = wg[kk][2 * tx], g1 = wg[kk][2 * tx + 1];
        float u0 = wu[kk][2 * tx], u1 = wu[kk][2 * tx + 1];
        g[0][0] = fmaf(xv0, g0, g[0][0]);
        g[0][1] = fmaf(xv0, g1, g[0][1]);
        g[1][0] = fmaf(xv1, g0, g[1][0]);
        g[1][1] = fmaf(xv1, g1, g[1][1]);
        u[0][0] = fmaf(xv0, u0, u[0][0]);
        u[0][1] = fmaf(xv0, u1, u[0][1]);
        u[1][0] = fmaf(xv1, u0, u[1][0]);
        u[1][1] = fmaf(xv1, u1, u[1][1]);
      }
      __syncthreads();
    }
    TE *hout = shared ? (TE *)a.h_shared : (TE *)a.h_routed;
    TE *guout = shared ? (TE *)a.gu_shared : (TE *)a.gu_routed;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      int64_t row = tr.r0 + 2 * ty + i;
      if (row >= tr.r1) continue;
#pragma unroll
      for (int j = 0; j < 2; ++j) {
        int f = f0 + 2 * tx + j;
        if (f >= Iseg) continue;
        float hv = silu_f32(g[i][j]) * u[i][j];
        hout[row * Iseg + f] = Elem<TE>::from_f32(hv);
        if (guout) {
          guout[row * 2 * Iseg + f] = Elem<TE>::from_f32(g[i][j]);
          guout[row * 2 * Iseg + Iseg + f] = Elem<TE>::from_f32(u[i][j]);
        }
      }
    }
  }
}

// down: tile of 32 rows x 64 outputs; thread (ty, tx) owns rows 2ty, 2ty+1
// and outputs 4tx..4tx+3.  Routed row j is written to y_routed[sorted_route[j]].
template <typename TE>
__global__ void __launch_bounds__(256) ffn_down_simt_kernel(FfnArgs a, const int32_t *__restrict__ tile_start) {
  griddep_launch();
  griddep_wait();
  __shared__ float hs[SIMT_BK][SIMT_BM + 1];
  __shared__ float wd[SIMT_BK][65];
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int total = tile_start[a.E + 1];
  const int o0 = blockIdx.y * 64;
  for (int ti = blockIdx.x; ti < total; ti += gridDim.x) {
    TileRows tr = decode_tile(ti, a.E, a.T, tile_start, a.offsets);
    const bool shared = tr.seg == a.E;
    const int Iseg = shared ? a.Is : a.I;
    const TE *hin = shared ? (const TE *)a.h_shared : (const TE *)a.h_routed;
    const TE *wdn = shared ? (const TE *)a.ws_down : (const TE *)a.w_down + (int64_t)(tr.seg - a.e_begin) * a.H * a.I;
    float acc[2][4];
#pragma unroll
    for (int i = 0; i < 2; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
    for (int i0 = 0; i0 < Iseg; i0 += SIMT_BK) {
      for (int i = threadIdx.x; i < SIMT_BM * SIMT_BK; i += 256) {
        int r = i / SIMT_BK, c = i % SIMT_BK, ii = i0 + c;
        int64_t row = tr.r0 + r;
        hs[c][r] = (row < tr.r1 && ii < Iseg) ? Elem<TE>::load(hin + row * Iseg + ii) : 0.f;
      }
      for (int i = threadIdx.x; i < 64 * SIMT_BK; i += 256) {
        int o = i / SIMT_BK, c = i % SIMT_BK, ii = i0 + c;
        wd[c][o] = (o0 + o < a.H && ii < Iseg) ? Elem<TE>::load(wdn + (int64_t)(o0 + o) * Iseg + ii) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < SIMT_BK; ++kk) {
        float hv0 = hs[kk][2 * ty], hv1 = hs[kk][2 * ty + 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          float wv = wd[kk][4 * tx + j];
          acc[0][j] = fmaf(hv0, wv, acc[0][j]);
          acc[1][j] = fmaf(hv1, wv, acc[1][j]);
        }
      }
      __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 2; ++i) {
      int64_t row = tr.r0 + 2 * ty + i;
      if (row >= tr.r1) continue;
      TE *dst = shared ? (TE *)a.y_shared + row * a.H
                       : (TE *)a.y_routed + (a.y_sorted ? row : (int64_t)a.sorted_route[row]) * a.H;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        int o = o0 + 4 * tx + j;
        if (o < a.H) dst[o] = Elem<TE>::from_f32(acc[i][j]);
      }
    }
  }
}

cudaError_t launch_ffn_simt(const FfnArgs &a, void *scratch, cudaStream_t stream) {
  if (a.T == 0) return cudaSuccess;
  int32_t *tile_start = (int32_t *)scratch;
  cudaError_t err = launch_build_tiles(a.E, a.T, SIMT_BM, a.offsets, tile_start, stream, a.e_begin, a.e_end,
                                       a.with_shared);
  if (err != cudaSuccess) return err;
  const int64_t R = (int64_t)a.T * a.k;
  const int64_t max_tiles = ceil_div(R + a.T, SIMT_BM) + a.E + 1;
  const unsigned gx = (unsigned)(max_tiles < 65535 ? max_tiles : 65535);
  dim3 g1(gx, (unsigned)ceil_div(a.I > a.Is ? a.I : a.Is, 32));
  dim3 g2(gx, (unsigned)ceil_div(a.H, 64));
  const int32_t *ts = tile_start;
  err = launch_pdl(ffn_gate_up_simt_kernel<float>, g1, dim3(256), 0, stream, a, ts);
  if (err != cudaSuccess) return err;
  return launch_pdl(ffn_down_simt_kernel<float>, g2, dim3(256), 0, stream, a, ts);
}

}  // namespace moe
