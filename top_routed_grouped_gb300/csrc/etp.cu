// Expert-tensor-parallel (ETP) reduction of the routed and shared rows.
//
// RL-Kernel PR #557 "What", bullet "Fail closed" (EP 1 = the experts
// expert-tensor-parallel over 4 ranks), the embedded #503 commit message,
// bullet "TP4 block" (every expert on every rank, results reduced across
// ranks), and PR #557 "What" again for the exchange (a byte copy and
// fixed-order local sums, no reduction collective): with the intermediate
// dimension I split across ranks, each
// rank's down projection is a partial sum over its slice of I.  Every rank
// gathers all partials (a byte copy) and sums them here in rank order, in
// FP32, with one rounding to the row type: the result depends on the number
// of ranks (the rounding order does), never on T, on which rank computes, or
// on the exchange's algorithm.
#include "common.cuh"
#include "kernels.h"

namespace moe {

struct EtpParts {
  const float *p[ETP_MAX_PARTS];
};

__device__ inline void store4(float *p, const float (&o)[4]) {
  *reinterpret_cast<float4 *>(p) = make_float4(o[0], o[1], o[2], o[3]);
}
__device__ inline void store4(__nv_bfloat16 *p, const float (&o)[4]) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(o[0], o[1]), b = __floats2bfloat162_rn(o[2], o[3]);
  *reinterpret_cast<uint2 *>(p) = make_uint2(*reinterpret_cast<const uint32_t *>(&a), *reinterpret_cast<const uint32_t *>(&b));
}

template <typename TO>
__global__ void __launch_bounds__(256) etp_reduce_kernel(const __grid_constant__ EtpParts parts, int n, int64_t count4, TO *__restrict__ out) {
  griddep_launch();
  griddep_wait();
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < count4; i += stride) {
    float4 acc = __ldg(reinterpret_cast<const float4 *>(parts.p[0]) + i);
    for (int q = 1; q < n; ++q) {
      const float4 v = __ldg(reinterpret_cast<const float4 *>(parts.p[q]) + i);
      acc.x += v.x;
      acc.y += v.y;
      acc.z += v.z;
      acc.w += v.w;
    }
    const float o[4] = {acc.x, acc.y, acc.z, acc.w};
    store4(out + 4 * i, o);
  }
}

cudaError_t launch_etp_reduce(int dtype, int n, const float *const *parts, int64_t count, void *out,
                              cudaStream_t stream) {
  if (n < 1 || n > ETP_MAX_PARTS || count % 4 != 0) return cudaErrorInvalidValue;
  if (count == 0) return cudaSuccess;
  EtpParts ps = {};
  for (int q = 0; q < n; ++q) ps.p[q] = parts[q];
  const int64_t count4 = count / 4;
  int sms = 0, dev = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const int64_t want = ceil_div(count4, 256);
  const unsigned grid = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
  if (dtype == 0) return launch_pdl(etp_reduce_kernel<float>, dim3(grid), dim3(256), 0, stream, ps, n, count4, (float *)out);
  return launch_pdl(etp_reduce_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, stream, ps, n, count4,
                    (__nv_bfloat16 *)out);
}

}  // namespace moe
