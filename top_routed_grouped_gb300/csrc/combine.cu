// combine_routes.
//
// RL-Kernel PR #557, embedded #503 commit message, bullet "Combine": the k
// weighted routed rows are summed with ordered FP32 multiply-adds and cast
// once to the output type, no atomics; PR #557 "What": every rank applies
// combine_routes in FP32 route order.  The gated shared-expert row is added
// after the k routed terms in the same FP32 accumulator:
//   acc = 0; for s = 0..k-1: acc = fma(w[t,s], Yr[t*k+s], acc);
//   acc = fma(sig[t], Ys[t], acc);  y = cast(acc)
// One thread owns 16 bytes of one output row, so the order is the same for
// every batch.  y_routed is in route order (row t*k + s), so a token's k rows
// are contiguous, or, on the expert-partitioned path, in sorted order.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// SORTED: the routed rows are in sorted order and route r's row is
// yr[route_pos[r]] (the expert-partitioned path); otherwise yr[r].
// KMAX >= k: the routed chunks one thread keeps in flight (a template
// parameter so that they live in registers).  stream_rows: the routed rows
// are loaded evict-first (ld.global.cs; each is read once), so that of the
// rows the down GEMM left in L2 the consumed ones go first and the ones not
// yet read stay.  The host sets it where the routed rows span more than
// twice the L2 (T = 8192: 335 MB, forward -5 µs; at T = 4096, 168 MB, the
// same loads measured +4 µs and are not used).
template <typename TE, bool SORTED, int KMAX>
__global__ void __launch_bounds__(256)
combine_kernel(int T, int H, int k, const TE *__restrict__ yr, const TE *__restrict__ ys,
               const float *__restrict__ w, const float *__restrict__ sig, TE *__restrict__ y,
               const int32_t *__restrict__ route_pos, int stream_rows) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;
  const int vec_per_row = H / VN;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)T * vec_per_row) return;
  const int64_t t = gid / vec_per_row;
  const int h = (int)(gid % vec_per_row) * VN;
  // All k routed chunks and the shared chunk are requested before the first
  // multiply-add (k <= KMAX loads in flight per thread instead of one), then
  // accumulated in slot order.
  uint4 raw[KMAX];
  float wv[KMAX];
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    if (s < k) {
      const int64_t row = SORTED ? (int64_t)__ldg(route_pos + t * k + s) : t * k + s;
      const uint4 *src = (const uint4 *)(yr + row * H + h);
      raw[s] = stream_rows ? __ldcs(src) : __ldg(src);
      wv[s] = __ldg(w + t * k + s);
    }
  }
  const uint4 rs = __ldg((const uint4 *)(ys + t * H + h));
  const float g = __ldg(sig + t);
  float acc[VN];
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = 0.f;
#pragma unroll
  for (int s = 0; s < KMAX; ++s) {
    if (s < k) {
      float v[VN];
      Vec16<TE>::unpack(raw[s], v);
#pragma unroll
      for (int j = 0; j < VN; ++j) acc[j] = fmaf(wv[s], v[j], acc[j]);
    }
  }
  float v[VN];
  Vec16<TE>::unpack(rs, v);
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = fmaf(g, v[j], acc[j]);
  Vec16<TE>::store(y + t * H + h, acc);
}

template <typename TE, int KMAX>
static cudaError_t launch_combine_k(dim3 g, int T, int H, int k, const TE *yr, const TE *ys, const float *w,
                                   const float *sig, TE *y, cudaStream_t stream, const int32_t *route_pos) {
  int dev = 0, l2 = 0;
  cudaGetDevice(&dev);
  if (cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, dev) != cudaSuccess) {
    cudaGetLastError();
    l2 = 0;
  }
  const int stream_rows = l2 > 0 && (int64_t)T * k * H * (int64_t)sizeof(TE) > 2 * (int64_t)l2;
  if (route_pos)
    return launch_pdl(combine_kernel<TE, true, KMAX>, g, dim3(256), 0, stream, T, H, k, yr, ys, w, sig, y, route_pos,
                      stream_rows);
  return launch_pdl(combine_kernel<TE, false, KMAX>, g, dim3(256), 0, stream, T, H, k, yr, ys, w, sig, y, route_pos,
                    stream_rows);
}

template <typename TE>
static cudaError_t launch_combine_t(int T, int H, int k, const void *y_routed, const void *y_shared, const float *w,
                                   const float *sig, void *y, cudaStream_t stream, const int32_t *route_pos) {
  const int64_t n = (int64_t)T * (H / Vec16<TE>::N);
  const dim3 g((unsigned)ceil_div(n, 256));
  const TE *yr = (const TE *)y_routed, *ys = (const TE *)y_shared;
  TE *yo = (TE *)y;
  if (k <= 2) return launch_combine_k<TE, 2>(g, T, H, k, yr, ys, w, sig, yo, stream, route_pos);
  if (k <= 4) return launch_combine_k<TE, 4>(g, T, H, k, yr, ys, w, sig, yo, stream, route_pos);
  if (k <= 8) return launch_combine_k<TE, 8>(g, T, H, k, yr, ys, w, sig, yo, stream, route_pos);
  if (k <= 10) return launch_combine_k<TE, 10>(g, T, H, k, yr, ys, w, sig, yo, stream, route_pos);
  return launch_combine_k<TE, 16>(g, T, H, k, yr, ys, w, sig, yo, stream, route_pos);
}

cudaError_t launch_combine(int dtype, int T, int H, int k, const void *y_routed, const void *y_shared,
                           const float *w, const float *sig, void *y, cudaStream_t stream, const int32_t *route_pos) {
  if (T == 0) return cudaSuccess;
  if (dtype == 0) return launch_combine_t<float>(T, H, k, y_routed, y_shared, w, sig, y, stream, route_pos);
  return launch_combine_t<__nv_bfloat16>(T, H, k, y_routed, y_shared, w, sig, y, stream, route_pos);
}

}  // namespace moe
