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
template <typename TE, bool SORTED>
__global__ void __launch_bounds__(256)
combine_kernel(int T, int H, int k, const TE *__restrict__ yr, const TE *__restrict__ ys,
               const float *__restrict__ w, const float *__restrict__ sig, TE *__restrict__ y,
               const int32_t *__restrict__ route_pos) {
  griddep_launch();
  griddep_wait();
  constexpr int VN = Vec16<TE>::N;
  const int vec_per_row = H / VN;
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)T * vec_per_row) return;
  const int64_t t = gid / vec_per_row;
  const int h = (int)(gid % vec_per_row) * VN;
  float acc[VN];
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = 0.f;
  for (int s = 0; s < k; ++s) {
    const float ws = w[t * k + s];
    float v[VN];
    const int64_t row = SORTED ? (int64_t)__ldg(route_pos + t * k + s) : t * k + s;
    Vec16<TE>::load(yr + row * H + h, v);
#pragma unroll
    for (int j = 0; j < VN; ++j) acc[j] = fmaf(ws, v[j], acc[j]);
  }
  const float g = sig[t];
  float v[VN];
  Vec16<TE>::load(ys + t * H + h, v);
#pragma unroll
  for (int j = 0; j < VN; ++j) acc[j] = fmaf(g, v[j], acc[j]);
  Vec16<TE>::store(y + t * H + h, acc);
}

cudaError_t launch_combine(int dtype, int T, int H, int k, const void *y_routed, const void *y_shared,
                           const float *w, const float *sig, void *y, cudaStream_t stream, const int32_t *route_pos) {
  if (T == 0) return cudaSuccess;
  const int VN = dtype == 0 ? 4 : 8;
  const int64_t n = (int64_t)T * (H / VN);
  const dim3 g((unsigned)ceil_div(n, 256)), b(256);
  if (dtype == 0) {
    const float *yr = (const float *)y_routed, *ys = (const float *)y_shared;
    if (route_pos) return launch_pdl(combine_kernel<float, true>, g, b, 0, stream, T, H, k, yr, ys, w, sig, (float *)y,
                                     route_pos);
    return launch_pdl(combine_kernel<float, false>, g, b, 0, stream, T, H, k, yr, ys, w, sig, (float *)y, route_pos);
  }
  const __nv_bfloat16 *yr = (const __nv_bfloat16 *)y_routed, *ys = (const __nv_bfloat16 *)y_shared;
  if (route_pos) return launch_pdl(combine_kernel<__nv_bfloat16, true>, g, b, 0, stream, T, H, k, yr, ys, w, sig,
                                   (__nv_bfloat16 *)y, route_pos);
  return launch_pdl(combine_kernel<__nv_bfloat16, false>, g, b, 0, stream, T, H, k, yr, ys, w, sig,
                    (__nv_bfloat16 *)y, route_pos);
}

}  // namespace moe
