// Backward of the MoE layer on CUDA cores.
//
// RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503 commit
// message, bullet "Backward": per-expert GEMMs write the per-route input
// gradients into one dense buffer, and dx sums them in ascending expert
// order (PR #557 "What").  "Results (4 x H100)", footnote 1: a torch.sum over
// hidden for the route-weight gradient was not batch invariant; here every
// reduction has a fixed order that does not depend on T or on the position.
//
// With L = sum_t dy_t . y_t and the routes held fixed:
//   b1  dw[t,s] = dy_t . Yr[t,s]          dsig[t] = dy_t . Ys[t]
//       dlogit[t,s] = w_s (dw_s - sum_j w_j dw_j)   dz[t] = dsig sig (1 - sig)
//       dYr[j] = w dy_t (row of route r at sorted row j)   dYs[t] = sig dy_t
//   b2  dh = dYr Wdn[e]                   dWdn[e] = sum_j dYr[j]^T h[j]
//   b3  dg = dh u silu'(g)    du = dh silu(g)      (fused into b2's dgrad)
//   b4  dXr = [dg du] Wgu[e]              dWgu[e] = sum_j [dg du][j]^T x[tok(j)]
//   b5  the shared expert: the same with dYs, over all T tokens
//   b6  dw_sg = sum_t dz[t] x[t]
//   b7  dWr[e] = sum over e's routes (ascending) of dlogit x[tok]
//   b8  dx[t] = sum over t's routes in ascending expert id of dXr
//               + dXs[t] + sum_s dlogit[t,s] Wr[e_s] + dz[t] w_sg
//       accumulated in FP32 in that order, cast once.
// Reductions over hidden use lane-partial sums in ascending h and a fixed
// butterfly; reductions over a segment's rows run in ascending row order.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------- b1
template <typename TE>
__global__ void __launch_bounds__(256)
combine_bwd_kernel(int T, int H, int k, const TE *__restrict__ dy, const TE *__restrict__ yr,
                   const TE *__restrict__ ys, const float *__restrict__ w, const float *__restrict__ sig,
                   const int32_t *__restrict__ route_pos, TE *__restrict__ dyr_sorted, TE *__restrict__ dys,
                   float *__restrict__ dlogit, float *__restrict__ dz, int yr_sorted) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const TE *dyr = dy + t * H;
  float dws[16];
  for (int s = 0; s < k; ++s) {
    const TE *row = yr + (yr_sorted ? (int64_t)route_pos[t * k + s] : t * k + s) * H;
    float part = 0.f;
    for (int h = lane * VN; h < H; h += 32 * VN) {
      float a[VN], b[VN];
      Vec16<TE>::load(dyr + h, a);
      Vec16<TE>::load(row + h, b);
#pragma unroll
      for (int j = 0; j < VN; ++j) part = fmaf(a[j], b[j], part);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(FULL_MASK, part, off);
    dws[s] = part;
  }
  float ps = 0.f;
  for (int h = lane * VN; h < H; h += 32 * VN) {
    float a[VN], b[VN];
    Vec16<TE>::load(dyr + h, a);
    Vec16<TE>::load(ys + t * H + h, b);
#pragma unroll
    for (int j = 0; j < VN; ++j) ps = fmaf(a[j], b[j], ps);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(FULL_MASK, ps, off);
  // router Jacobian of the softmax over the selected set, slot order
  float wdw = 0.f;
  for (int s = 0; s < k; ++s) wdw = fmaf(w[t * k + s], dws[s], wdw);
  if (lane < k) {
    float dwl = 0.f;
    for (int s = 0; s < k; ++s)
      if (s == lane) dwl = dws[s];
    dlogit[t * k + lane] = w[t * k + lane] * (dwl - wdw);
  }
  const float g = sig[t];
  if (lane == 0) dz[t] = ps * g * (1.f - g);
  // scaled rows
  for (int h = lane * VN; h < H; h += 32 * VN) {
    float a[VN], o[VN];
    Vec16<TE>::load(dyr + h, a);
    for (int s = 0; s < k; ++s) {
      const float ws = w[t * k + s];
#pragma unroll
      for (int j = 0; j < VN; ++j) o[j] = ws * a[j];
      Vec16<TE>::store(dyr_sorted + (int64_t)route_pos[t * k + s] * H + h, o);
    }
#pragma unroll
    for (int j = 0; j < VN; ++j) o[j] = g * a[j];
    Vec16<TE>::store(dys + t * H + h, o);
  }
}

// The same step with the row held in registers: for H = NCH * 32 * VN (each
// lane owns NCH 16-byte chunks of a row) and k <= KMAX, dy is loaded once and
// every chunk of a routed row is requested before its dot product starts,
// so the loads of one row (and, as the unrolled slots allow, of the next)
// are in flight together instead of one chunk at a time.  Every sum, product
// and store is the one above in the same order: the results are identical.
template <typename TE, int NCH, int KMAX>
__global__ void __launch_bounds__(128)
combine_bwd_rows_kernel(int T, int H, int k, const TE *__restrict__ dy, const TE *__restrict__ yr,
                        const TE *__restrict__ ys, const float *__restrict__ w, const float *__restrict__ sig,
                        const int32_t *__restrict__ route_pos, TE *__restrict__ dyr_sorted, TE *__restrict__ dys,
                        float *__restrict__ dlogit, float *__restrict__ dz, int yr_sorted) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const TE *dyr = dy + t * H + lane * VN;
  uint4 a[NCH];
#pragma unroll
  for (int i = 0; i < NCH; ++i) a[i] = __ldg((const uint4 *)(dyr + i * 32 * VN));
  float dws[KMAX];
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    dws[s] = 0.f;
    if (s < k) {
      const TE *row = yr + (yr_sorted ? (int64_t)__ldg(route_pos + t * k + s) : t * k + s) * H + lane * VN;
      uint4 b[NCH];
#pragma unroll
      for (int i = 0; i < NCH; ++i) b[i] = __ldg((const uint4 *)(row + i * 32 * VN));
      float part = 0.f;
#pragma unroll
      for (int i = 0; i < NCH; ++i) {
        float av[VN], bv[VN];
        Vec16<TE>::unpack(a[i], av);
        Vec16<TE>::unpack(b[i], bv);
#pragma unroll
        for (int j = 0; j < VN; ++j) part = fmaf(av[j], bv[j], part);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(FULL_MASK, part, off);
      dws[s] = part;
    }
  }
  float ps = 0.f;
  {
    uint4 b[NCH];
#pragma unroll
    for (int i = 0; i < NCH; ++i) b[i] = __ldg((const uint4 *)(ys + t * H + lane * VN + i * 32 * VN));
#pragma unroll
    for (int i = 0; i < NCH; ++i) {
      float av[VN], bv[VN];
      Vec16<TE>::unpack(a[i], av);
      Vec16<TE>::unpack(b[i], bv);
#pragma unroll
      for (int j = 0; j < VN; ++j) ps = fmaf(av[j], bv[j], ps);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) ps += __shfl_xor_sync(FULL_MASK, ps, off);
  // router Jacobian of the softmax over the selected set, slot order
  float wv[KMAX];
  float wdw = 0.f;
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    wv[s] = s < k ? __ldg(w + t * k + s) : 0.f;
    if (s < k) wdw = fmaf(wv[s], dws[s], wdw);
  }
  if (lane < k) {
    float dwl = 0.f, wl = 0.f;
#pragma unroll
    for (int s = 0; s < KMAX; ++s)
      if (s == lane) dwl = dws[s], wl = wv[s];
    dlogit[t * k + lane] = wl * (dwl - wdw);
  }
  const float g = __ldg(sig + t);
  if (lane == 0) dz[t] = ps * g * (1.f - g);
  // scaled rows
  int pos[KMAX];
#pragma unroll
  for (int s = 0; s < KMAX; ++s) pos[s] = s < k ? __ldg(route_pos + t * k + s) : 0;
#pragma unroll
  for (int i = 0; i < NCH; ++i) {
    const int h = lane * VN + i * 32 * VN;
    float av[VN], o[VN];
    Vec16<TE>::unpack(a[i], av);
#pragma unroll
    for (int s = 0; s < KMAX; ++s) {
      if (s < k) {
#pragma unroll
        for (int j = 0; j < VN; ++j) o[j] = wv[s] * av[j];
        Vec16<TE>::store(dyr_sorted + (int64_t)pos[s] * H + h, o);
      }
    }
#pragma unroll
    for (int j = 0; j < VN; ++j) o[j] = g * av[j];
    Vec16<TE>::store(dys + t * H + h, o);
  }
}

template <typename TE, int NCH>
static cudaError_t launch_combine_bwd_rows(const BwArgs &a, cudaStream_t stream) {
  const dim3 g((unsigned)ceil_div(a.T, 4)), b(128);
  const TE *dy = (const TE *)a.dy, *yr = (const TE *)a.y_routed, *ys = (const TE *)a.y_shared;
  TE *dyr = (TE *)a.dyr, *dys = (TE *)a.dys;
  if (a.k <= 8)
    return launch_pdl(combine_bwd_rows_kernel<TE, NCH, 8>, g, b, 0, stream, a.T, a.H, a.k, dy, yr, ys, a.topk_w,
                      a.shared_sig, a.route_pos, dyr, dys, a.dlogit, a.dz, a.yr_sorted);
  if (a.k <= 10)
    return launch_pdl(combine_bwd_rows_kernel<TE, NCH, 10>, g, b, 0, stream, a.T, a.H, a.k, dy, yr, ys, a.topk_w,
                      a.shared_sig, a.route_pos, dyr, dys, a.dlogit, a.dz, a.yr_sorted);
  return launch_pdl(combine_bwd_rows_kernel<TE, NCH, 16>, g, b, 0, stream, a.T, a.H, a.k, dy, yr, ys, a.topk_w,
                    a.shared_sig, a.route_pos, dyr, dys, a.dlogit, a.dz, a.yr_sorted);
}

// b1: the register form when H is 1, 2, 4 or 8 chunks of 16 bytes per lane, else the loop form.
template <typename TE>
static cudaError_t launch_combine_bwd(const BwArgs &a, cudaStream_t stream) {
  constexpr int VN = Vec16<TE>::N;
  if (a.H % (32 * VN) == 0) {
    switch (a.H / (32 * VN)) {
      case 1: return launch_combine_bwd_rows<TE, 1>(a, stream);
      case 2: return launch_combine_bwd_rows<TE, 2>(a, stream);
      case 4: return launch_combine_bwd_rows<TE, 4>(a, stream);
      case 8: return launch_combine_bwd_rows<TE, 8>(a, stream);
      default: break;
    }
  }
  return launch_pdl(combine_bwd_kernel<TE>, dim3((unsigned)ceil_div(a.T, 8)), dim3(256), 0, stream, a.T, a.H, a.k,
                    (const TE *)a.dy, (const TE *)a.y_routed, (const TE *)a.y_shared, a.topk_w, a.shared_sig,
                    a.route_pos, (TE *)a.dyr, (TE *)a.dys, a.dlogit, a.dz, a.yr_sorted);
}

// ---------------------------------------------------------------- tiles
// Segment s < E: sorted rows offsets[s]..offsets[s+1]; segment E: tokens 0..T.
constexpr int BW_BM = 32;  // rows per tile of the row-parallel GEMMs

struct BwTile {
  int seg;
  int64_t r0, r1;
};

__device__ inline BwTile bw_decode(int ti, int E, int T, const int32_t *tile_start, const int32_t *offsets,
                                   int bm = BW_BM) {
  int lo = 0, hi = E;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (tile_start[mid] <= ti) lo = mid;
    else hi = mid - 1;
  }
  BwTile tr;
  tr.seg = lo;
  const int i = ti - tile_start[lo];
  if (lo < E) {
    tr.r0 = offsets[lo] + (int64_t)i * bm;
    tr.r1 = min((int64_t)offsets[lo + 1], tr.r0 + bm);
  } else {
    tr.r0 = (int64_t)i * bm;
    tr.r1 = min((int64_t)T, tr.r0 + bm);
  }
  return tr;
}

// ---------------------------------------------------------------- b2 + b3
// dh[j, i] = sum_h dYr[j, h] Wdn[e][h, i] (h ascending); then
// dGU[j] = [dh u silu'(g) | dh silu(g)] from the saved [g | u] of row j.
template <typename TE>
__global__ void __launch_bounds__(256)
down_dgrad_swiglu_kernel(BwArgs a, const int32_t *__restrict__ tile_start) {
  griddep_launch();
  griddep_wait();
  __shared__ float ds[32][BW_BM + 1];   // [h][row]
  __shared__ float wd[32][65];          // [h][i]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int total = tile_start[a.E + 1];
  const int i0 = blockIdx.y * 64;
  for (int ti = blockIdx.x; ti < total; ti += gridDim.x) {
    const BwTile tr = bw_decode(ti, a.E, a.T, tile_start, a.offsets);
    const bool sh = tr.seg == a.E;
    const int Iseg = sh ? a.Is : a.I;
    if (i0 >= Iseg) continue;
    const TE *dyrow = sh ? (const TE *)a.dys : (const TE *)a.dyr;
    const TE *wdn = sh ? (const TE *)a.ws_down : (const TE *)a.w_down + (int64_t)(tr.seg - a.e_begin) * a.H * a.I;
    float acc[2][4] = {};
    for (int h0 = 0; h0 < a.H; h0 += 32) {
      for (int idx = threadIdx.x; idx < BW_BM * 32; idx += 256) {
        const int r = idx / 32, c = idx % 32;
        const int64_t row = tr.r0 + r;
        ds[c][r] = row < tr.r1 && h0 + c < a.H ? Elem<TE>::load(dyrow + row * a.H + h0 + c) : 0.f;
      }
      for (int idx = threadIdx.x; idx < 64 * 32; idx += 256) {
        const int c = idx / 64, i = idx % 64;
        wd[c][i] = i0 + i < Iseg && h0 + c < a.H ? Elem<TE>::load(wdn + (int64_t)(h0 + c) * Iseg + i0 + i) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const float d0 = ds[kk][2 * ty], d1 = ds[kk][2 * ty + 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float wv = wd[kk][4 * tx + j];
          acc[0][j] = fmaf(d0, wv, acc[0][j]);
          acc[1][j] = fmaf(d1, wv, acc[1][j]);
        }
      }
      __syncthreads();
    }
    const TE *gu = sh ? (const TE *)a.gu_shared : (const TE *)a.gu_routed;
    TE *dgu = sh ? (TE *)a.dgu_shared : (TE *)a.dgu_routed;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int64_t row = tr.r0 + 2 * ty + r;
      if (row >= tr.r1) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int i = i0 + 4 * tx + j;
        if (i >= Iseg) continue;
        const float g = Elem<TE>::load(gu + row * 2 * Iseg + i);
        const float u = Elem<TE>::load(gu + row * 2 * Iseg + Iseg + i);
        const float s = sigmoid_f32(g);
        const float dh = acc[r][j];
        dgu[row * 2 * Iseg + i] = Elem<TE>::from_f32(dh * u * (s * (1.f + g * (1.f - s))));
        dgu[row * 2 * Iseg + Iseg + i] = Elem<TE>::from_f32(dh * (g * s));
      }
    }
  }
}

// ---------------------------------------------------------------- b4 dgrad
// dXr[j, h] = sum_f dGU[j, f] Wgu[e][f, h] (f ascending), FP32 rows.
template <typename TE>
__global__ void __launch_bounds__(256)
gate_up_dgrad_kernel(BwArgs a, const int32_t *__restrict__ tile_start) {
  griddep_launch();
  griddep_wait();
  __shared__ float gs[32][BW_BM + 1];  // [f][row]
  __shared__ float wg[32][65];         // [f][h]
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  const int total = tile_start[a.E + 1];
  const int h0 = blockIdx.y * 64;
  for (int ti = blockIdx.x; ti < total; ti += gridDim.x) {
    const BwTile tr = bw_decode(ti, a.E, a.T, tile_start, a.offsets);
    const bool sh = tr.seg == a.E;
    const int Iseg = sh ? a.Is : a.I;
    const TE *dgu = sh ? (const TE *)a.dgu_shared : (const TE *)a.dgu_routed;
    const TE *wgu =
        sh ? (const TE *)a.ws_gate_up : (const TE *)a.w_gate_up + (int64_t)(tr.seg - a.e_begin) * 2 * a.I * a.H;
    float acc[2][4] = {};
    for (int f0 = 0; f0 < 2 * Iseg; f0 += 32) {
      for (int idx = threadIdx.x; idx < BW_BM * 32; idx += 256) {
        const int r = idx / 32, c = idx % 32;
        const int64_t row = tr.r0 + r;
        gs[c][r] = row < tr.r1 && f0 + c < 2 * Iseg ? Elem<TE>::load(dgu + row * 2 * Iseg + f0 + c) : 0.f;
      }
      for (int idx = threadIdx.x; idx < 64 * 32; idx += 256) {
        const int c = idx / 64, hh = idx % 64;
        wg[c][hh] = h0 + hh < a.H && f0 + c < 2 * Iseg ? Elem<TE>::load(wgu + (int64_t)(f0 + c) * a.H + h0 + hh) : 0.f;
      }
      __syncthreads();
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const float d0 = gs[kk][2 * ty], d1 = gs[kk][2 * ty + 1];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float wv = wg[kk][4 * tx + j];
          acc[0][j] = fmaf(d0, wv, acc[0][j]);
          acc[1][j] = fmaf(d1, wv, acc[1][j]);
        }
      }
      __syncthreads();
    }
    float *out = sh ? a.dxs : a.dxr;
#pragma unroll
    for (int r = 0; r < 2; ++r) {
      const int64_t row = tr.r0 + 2 * ty + r;
      if (row >= tr.r1) continue;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int hh = h0 + 4 * tx + j;
        if (hh < a.H) out[row * a.H + hh] = acc[r][j];
      }
    }
  }
}

// ---------------------------------------------------------------- weight grads
// out[e][m, n] = sum over the segment's rows j (ascending) of A_j[m] B_j[n],
// one 64 x 64 output tile per block, each output summed by one thread.
//   DOWN:    A = dYr rows (m = h), B = h rows (n = i)           -> dWdn [H, I]
//   GATE_UP: A = dGU rows (m = f), B = x rows of the tokens     -> dWgu [2I, H]
//   ROUTER:  A = dlogit of the routes (m = 0 only), B = x rows  -> dWr [E, H]
enum { WG_DOWN = 0, WG_GATE_UP = 1 };

template <typename TE, int KIND>
__global__ void __launch_bounds__(256) wgrad_kernel(BwArgs a) {
  griddep_launch();
  griddep_wait();
  __shared__ float as[16][65];  // [row][m]
  __shared__ float bs[16][65];  // [row][n]
  // blockIdx.z: the partition's experts in order, then the shared expert
  const int n_local = (a.e_end < 0 ? a.E : a.e_end) - a.e_begin;
  const int seg = (int)blockIdx.z < n_local ? a.e_begin + (int)blockIdx.z : a.E;
  const bool sh = seg == a.E;
  const int Iseg = sh ? a.Is : a.I;
  const int M = KIND == WG_DOWN ? a.H : 2 * Iseg;
  const int N = KIND == WG_DOWN ? Iseg : a.H;
  const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
  if (m0 >= M || n0 >= N) return;
  const int64_t r0 = sh ? 0 : a.offsets[seg];
  const int64_t r1 = sh ? a.T : a.offsets[seg + 1];
  const TE *A = KIND == WG_DOWN ? (const TE *)(sh ? a.dys : a.dyr) : (const TE *)(sh ? a.dgu_shared : a.dgu_routed);
  const int lda = KIND == WG_DOWN ? a.H : 2 * Iseg;
  const TE *Bh = (const TE *)(sh ? a.h_shared : a.h_routed);
  const TE *x = (const TE *)a.x;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4] = {};
  for (int64_t j0 = r0; j0 < r1; j0 += 16) {
    for (int idx = threadIdx.x; idx < 16 * 64; idx += 256) {
      const int r = idx / 64, c = idx % 64;
      const int64_t row = j0 + r;
      const bool ok = row < r1;
      as[r][c] = ok && m0 + c < M ? Elem<TE>::load(A + row * lda + m0 + c) : 0.f;
      float bv = 0.f;
      if (ok && n0 + c < N) {
        if (KIND == WG_DOWN) {
          bv = Elem<TE>::load(Bh + row * Iseg + n0 + c);
        } else {
          const int64_t tok = sh ? row : (int64_t)(a.sorted_route[row] / a.k);
          bv = Elem<TE>::load(x + tok * a.H + n0 + c);
        }
      }
      bs[r][c] = bv;
    }
    __syncthreads();
#pragma unroll
    for (int r = 0; r < 16; ++r) {
      float av[4], bv[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) av[i] = as[r][4 * ty + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) bv[j] = bs[r][4 * tx + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(av[i], bv[j], acc[i][j]);
    }
    __syncthreads();
  }
  const int64_t le = seg - a.e_begin;  // index in the partition's weight arrays
  float *out = KIND == WG_DOWN ? (sh ? a.dws_down : a.dw_down + le * a.H * a.I)
                               : (sh ? a.dws_gate_up : a.dw_gate_up + le * 2 * a.I * a.H);
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int m = m0 + 4 * ty + i, n = n0 + 4 * tx + j;
      if (m < M && n < N) out[(int64_t)m * N + n] = acc[i][j];
    }
}

// b7: dWr[e, h] = sum over e's sorted rows j of dlogit[route] x[tok, h];
// b6: dw_sg[h] = sum_t dz[t] x[t, h] (segment E).  Two passes with a fixed
// order: a segment's rows are cut into chunks of RG_CHUNK consecutive rows,
// pass 1 sums each chunk in ascending row order into a partial row, pass 2
// sums a segment's partial rows in ascending chunk order.
constexpr int RG_CHUNK = 64;

template <typename TE>
__global__ void __launch_bounds__(256)
router_gate_partial_kernel(BwArgs a, const int32_t *__restrict__ chunk_start, float *__restrict__ partial) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;  // columns per thread (16 bytes of x)
  __shared__ int64_t srow[RG_CHUNK];  // element offset of each row's x
  __shared__ float scoef[RG_CHUNK];
  const int total = chunk_start[a.E + 1];
  const int h = (blockIdx.y * 256 + threadIdx.x) * VN;
  const TE *x = (const TE *)a.x;
  for (int c = blockIdx.x; c < total; c += gridDim.x) {
    const BwTile tr = bw_decode(c, a.E, a.T, chunk_start, a.offsets, RG_CHUNK);
    const int n = (int)(tr.r1 - tr.r0);
    __syncthreads();
    if (threadIdx.x < n) {
      const int64_t j = tr.r0 + threadIdx.x;
      if (tr.seg < a.E) {
        const int r = a.sorted_route[j];
        srow[threadIdx.x] = (int64_t)(r / a.k) * a.H;
        scoef[threadIdx.x] = a.dlogit[r];
      } else {
        srow[threadIdx.x] = j * a.H;
        scoef[threadIdx.x] = a.dz[j];
      }
    }
    __syncthreads();
    if (h >= a.H) continue;
    float acc[VN];
#pragma unroll
    for (int v = 0; v < VN; ++v) acc[v] = 0.f;
#pragma unroll 4
    for (int i = 0; i < n; ++i) {
      float xv[VN];
      Vec16<TE>::load(x + srow[i] + h, xv);
      const float cf = scoef[i];
#pragma unroll
      for (int v = 0; v < VN; ++v) acc[v] = fmaf(cf, xv[v], acc[v]);
    }
    float *dst = partial + (int64_t)c * a.H + h;
#pragma unroll
    for (int v = 0; v < VN; v += 4) *(float4 *)(dst + v) = make_float4(acc[v], acc[v + 1], acc[v + 2], acc[v + 3]);
  }
}

__global__ void __launch_bounds__(256)
router_gate_reduce_kernel(BwArgs a, const int32_t *__restrict__ chunk_start, const float *__restrict__ partial) {
  griddep_launch();
  griddep_wait();
  const int seg = blockIdx.y;
  const int h = blockIdx.x * 256 + threadIdx.x;
  if (h >= a.H) return;
  float acc = 0.f;
  for (int c = chunk_start[seg]; c < chunk_start[seg + 1]; ++c) acc += partial[(int64_t)c * a.H + h];
  if (seg < a.E) a.dw_router[(int64_t)seg * a.H + h] = acc;
  else a.dw_shared_gate[h] = acc;
}

// ---------------------------------------------------------------- b8
// One warp per (token, 32 x 16-byte chunk of the row): the slots are ranked
// by expert id (ids of a token are distinct), then each lane assembles one
// 16-byte chunk.  Five blocks per SM (48 registers): the kernel is bound by
// the latency of its row loads, and more resident warps keep more of them in
// flight (T = 4096 backward: 102 us with three blocks per SM, 91-97 with
// five, 104 with six, 117 with eight).
template <typename TE>
__global__ void __launch_bounds__(256, 5) dx_kernel(BwArgs a) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;
  const int lane = threadIdx.x & 31;
  const int per_row = a.H / (32 * VN);  // warps per token (H is a multiple of 32 VN here)
  const int64_t gw = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (gw >= (int64_t)a.T * per_row) return;
  const int64_t t = gw / per_row;
  const int h = (int)(gw % per_row) * 32 * VN + lane * VN;
  const int k = a.k;
  const int id = lane < k ? a.topk_ids[t * k + lane] : 0x7fffffff;
  int rank = 0;
  for (int s = 0; s < k; ++s) rank += __shfl_sync(FULL_MASK, id, s) < id;
  const int pos = lane < k ? a.route_pos[t * k + lane] : 0;
  const float dl = lane < k ? a.dlogit[t * k + lane] : 0.f;
  float acc[VN];
#pragma unroll
  for (int v = 0; v < VN; ++v) acc[v] = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const unsigned m = __ballot_sync(FULL_MASK, lane < k && rank == i);
    const int64_t row = __shfl_sync(FULL_MASK, pos, m ? __ffs(m) - 1 : 0);
    if (i < k) {
      const float4 *src = reinterpret_cast<const float4 *>(a.dxr + row * a.H + h);
#pragma unroll
      for (int v = 0; v < VN / 4; ++v) {
        const float4 q = src[v];
        acc[4 * v] += q.x;
        acc[4 * v + 1] += q.y;
        acc[4 * v + 2] += q.z;
        acc[4 * v + 3] += q.w;
      }
    }
  }
  {
    const float4 *src = reinterpret_cast<const float4 *>(a.dxs + t * a.H + h);
#pragma unroll
    for (int v = 0; v < VN / 4; ++v) {
      const float4 q = src[v];
      acc[4 * v] += q.x;
      acc[4 * v + 1] += q.y;
      acc[4 * v + 2] += q.z;
      acc[4 * v + 3] += q.w;
    }
  }
  float rt[VN];
#pragma unroll
  for (int v = 0; v < VN; ++v) rt[v] = 0.f;
#pragma unroll
  for (int s = 0; s < 16; ++s) {
    const int e = __shfl_sync(FULL_MASK, id, s);
    const float d = __shfl_sync(FULL_MASK, dl, s);
    if (s < k) {
      const float4 *wr = reinterpret_cast<const float4 *>(a.w_router + (int64_t)e * a.H + h);
#pragma unroll
      for (int v = 0; v < VN / 4; ++v) {
        const float4 q = wr[v];
        rt[4 * v] = fmaf(d, q.x, rt[4 * v]);
        rt[4 * v + 1] = fmaf(d, q.y, rt[4 * v + 1]);
        rt[4 * v + 2] = fmaf(d, q.z, rt[4 * v + 2]);
        rt[4 * v + 3] = fmaf(d, q.w, rt[4 * v + 3]);
      }
    }
  }
  float gv[VN];
  Vec16<TE>::load((const TE *)a.w_shared_gate + h, gv);
  const float dzt = a.dz[t];
  float o[VN];
#pragma unroll
  for (int v = 0; v < VN; ++v) o[v] = fmaf(dzt, gv[v], acc[v] + rt[v]);
  Vec16<TE>::store((TE *)a.dx + t * a.H + h, o);
}

// Simple variant for rows whose length is not a multiple of 32 x 16 bytes:
// one thread per (token, 16-byte chunk), same order of the sums.
template <typename TE>
__global__ void __launch_bounds__(256) dx_thread_kernel(BwArgs a) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;
  const int per_row = a.H / VN;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)a.T * per_row) return;
  const int64_t t = gid / per_row;
  const int h = (int)(gid % per_row) * VN;
  const int k = a.k;
  float acc[VN];
#pragma unroll
  for (int v = 0; v < VN; ++v) acc[v] = 0.f;
  int order[16];  // slots in ascending expert id (insertion sort; ids are distinct)
  for (int s = 0; s < k; ++s) {
    const int e = a.topk_ids[t * k + s];
    int j = s - 1;
    while (j >= 0 && a.topk_ids[t * k + order[j]] > e) {
      order[j + 1] = order[j];
      --j;
    }
    order[j + 1] = s;
  }
  for (int i = 0; i < k; ++i) {
    const float4 *src = reinterpret_cast<const float4 *>(a.dxr + (int64_t)a.route_pos[t * k + order[i]] * a.H + h);
#pragma unroll
    for (int v = 0; v < VN / 4; ++v) {
      const float4 q = src[v];
      acc[4 * v] += q.x;
      acc[4 * v + 1] += q.y;
      acc[4 * v + 2] += q.z;
      acc[4 * v + 3] += q.w;
    }
  }
  const float4 *src = reinterpret_cast<const float4 *>(a.dxs + t * a.H + h);
#pragma unroll
  for (int v = 0; v < VN / 4; ++v) {
    const float4 q = src[v];
    acc[4 * v] += q.x;
    acc[4 * v + 1] += q.y;
    acc[4 * v + 2] += q.z;
    acc[4 * v + 3] += q.w;
  }
  float rt[VN];
#pragma unroll
  for (int v = 0; v < VN; ++v) rt[v] = 0.f;
  for (int s = 0; s < k; ++s) {
    const float d = a.dlogit[t * k + s];
    const float *wr = a.w_router + (int64_t)a.topk_ids[t * k + s] * a.H + h;
#pragma unroll
    for (int v = 0; v < VN; ++v) rt[v] = fmaf(d, wr[v], rt[v]);
  }
  float gv[VN];
  Vec16<TE>::load((const TE *)a.w_shared_gate + h, gv);
  const float dzt = a.dz[t];
  float o[VN];
#pragma unroll
  for (int v = 0; v < VN; ++v) o[v] = fmaf(dzt, gv[v], acc[v] + rt[v]);
  Vec16<TE>::store((TE *)a.dx + t * a.H + h, o);
}

// ---------------------------------------------------------------- launcher
// Scratch: [GEMM tiles or item tables][chunk starts (E+2)][partial rows].
static size_t gemm_scratch_bytes(int dtype, int T, int k, int E, int H, int I, int Is) {
  const size_t tiles = (size_t)(E + 2) * sizeof(int32_t);
  if (dtype != 0 && backward_tc_supported(H, I, Is)) return std::max(tiles, dgrad_tc_scratch_bytes(T, k, E, H, I, Is));
  return tiles;
}
static int64_t max_chunks(int T, int k, int E) { return ceil_div((int64_t)T * k + T, RG_CHUNK) + E + 1; }

size_t backward_scratch_bytes(int dtype, int T, int k, int E, int H, int I, int Is) {
  return (size_t)round_up((int64_t)gemm_scratch_bytes(dtype, T, k, E, H, I, Is), 256) +
         (size_t)round_up((int64_t)(E + 2) * 4, 256) + (size_t)max_chunks(T, k, E) * H * sizeof(float);
}

template <typename TE>
static cudaError_t run_backward(const BwArgs &a, void *scratch, int *status, cudaStream_t stream, int phase) {
  const int64_t R = (int64_t)a.T * a.k;
  const int eb = a.e_begin, ee = a.e_end < 0 ? a.E : a.e_end;
  cudaError_t err;
#define MOE_TRY(x) \
  if ((err = (x)) != cudaSuccess) return err
  if (phase & BWD_PHASE_EXPERTS) {
    MOE_TRY(launch_combine_bwd<TE>(a, stream));
    const int Imax = a.I > a.Is ? a.I : a.Is;
    if (sizeof(TE) == 2 && backward_tc_supported(a.H, a.I, a.Is)) {
      MOE_TRY(launch_dgrad_tc(a, scratch, status, stream));
      MOE_TRY(launch_wgrad_tc(a, status, stream));
    } else {
      int32_t *tile_start = (int32_t *)scratch;
      const int32_t *ts = tile_start;
      MOE_TRY(launch_build_tiles(a.E, a.T, BW_BM, a.offsets, tile_start, stream, eb, ee, 1));
      const int64_t max_tiles = ceil_div(R + a.T, BW_BM) + a.E + 1;
      const unsigned gx = (unsigned)(max_tiles < 65535 ? max_tiles : 65535);
      const unsigned nseg = (unsigned)(ee - eb + 1);
      MOE_TRY(launch_pdl(down_dgrad_swiglu_kernel<TE>, dim3(gx, (unsigned)ceil_div(Imax, 64)), dim3(256), 0, stream,
                         a, ts));
      MOE_TRY(launch_pdl(gate_up_dgrad_kernel<TE>, dim3(gx, (unsigned)ceil_div(a.H, 64)), dim3(256), 0, stream, a,
                         ts));
      MOE_TRY(launch_pdl(wgrad_kernel<TE, WG_DOWN>, dim3((unsigned)ceil_div(Imax, 64), (unsigned)ceil_div(a.H, 64), nseg),
                         dim3(256), 0, stream, a));
      MOE_TRY(launch_pdl(wgrad_kernel<TE, WG_GATE_UP>,
                         dim3((unsigned)ceil_div(a.H, 64), (unsigned)ceil_div(2 * Imax, 64), nseg), dim3(256), 0,
                         stream, a));
    }
    const int dtype = sizeof(TE) == 4 ? 0 : 1;
    uint8_t *rest =
        (uint8_t *)scratch + round_up((int64_t)gemm_scratch_bytes(dtype, a.T, a.k, a.E, a.H, a.I, a.Is), 256);
    int32_t *chunk_start = (int32_t *)rest;
    const int32_t *cs = chunk_start;
    float *partial = (float *)(rest + round_up((int64_t)(a.E + 2) * 4, 256));
    const float *pc = partial;
    MOE_TRY(launch_build_tiles(a.E, a.T, RG_CHUNK, a.offsets, chunk_start, stream));
    const int64_t mc = max_chunks(a.T, a.k, a.E);
    MOE_TRY(launch_pdl(router_gate_partial_kernel<TE>,
                       dim3((unsigned)std::min<int64_t>(mc, 65535), (unsigned)ceil_div(a.H, 256 * Vec16<TE>::N)),
                       dim3(256), 0, stream, a, cs, partial));
    MOE_TRY(launch_pdl(router_gate_reduce_kernel, dim3((unsigned)ceil_div(a.H, 256), a.E + 1), dim3(256), 0, stream,
                       a, cs, pc));
  }
  if (!(phase & BWD_PHASE_DX)) return cudaSuccess;
  if (a.H % (32 * Vec16<TE>::N) == 0)
    return launch_pdl(dx_kernel<TE>, dim3((unsigned)ceil_div((int64_t)a.T * (a.H / (32 * Vec16<TE>::N)), 8)),
                      dim3(256), 0, stream, a);
  return launch_pdl(dx_thread_kernel<TE>, dim3((unsigned)ceil_div((int64_t)a.T * (a.H / Vec16<TE>::N), 256)),
                    dim3(256), 0, stream, a);
#undef MOE_TRY
}

cudaError_t launch_backward(int dtype, const BwArgs &a, void *scratch, int *status, cudaStream_t stream, int phase) {
  if (a.T == 0) return cudaSuccess;
  if (dtype == 0) return run_backward<float>(a, scratch, status, stream, phase);
  return run_backward<__nv_bfloat16>(a, scratch, status, stream, phase);
}

}  // namespace moe
