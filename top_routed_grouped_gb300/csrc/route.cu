// Routing kernels.
//
// RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503 commit
// message, bullet "Routing": FP32 router through a batch-invariant GEMM, a
// fixed-order softmax, stable descending top-k (ties to the lower expert id)
// and FP32 renormalisation of the selected weights.  Shared-expert gate:
// #503 "TP4 block" (replicated shared-expert gate), a sigmoid of x . w_sg.
//
// Batch invariance: every value a token receives is computed by one thread
// or one warp from that token's row alone, in an order fixed by H and E only.
#include "common.cuh"
#include "kernels.h"

namespace moe {

// ---------------------------------------------------------------------------
// FP32 router GEMM on CUDA cores: logits[t,e] = sum_h x[t,h] wr[e,h] (+bias).
// 64x64 output tile per block, each output accumulated by one thread with
// fmaf over h = 0, 1, ..., H-1 in that order (zero padding past H adds exact
// zeros), so the value does not depend on the tile a token falls in.
// ---------------------------------------------------------------------------
template <typename TX>
__global__ void __launch_bounds__(256)
router_logits_simt_kernel(int T, int H, int E, const TX *__restrict__ x, const float *__restrict__ wr,
                          const float *__restrict__ bias, float *__restrict__ logits) {
  griddep_launch();
  griddep_wait();
  __shared__ float xs[32][68];
  __shared__ float wsm[32][68];
  const int t0 = blockIdx.x * 64, e0 = blockIdx.y * 64;
  const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
  float acc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;

  for (int h0 = 0; h0 < H; h0 += 32) {
    for (int i = threadIdx.x; i < 64 * 32; i += 256) {
      int r = i >> 5, c = i & 31;
      int t = t0 + r, e = e0 + r, h = h0 + c;
      xs[c][r] = (t < T && h < H) ? Elem<TX>::load(x + (int64_t)t * H + h) : 0.f;
      wsm[c][r] = (e < E && h < H) ? wr[(int64_t)e * H + h] : 0.f;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < 32; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = xs[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = wsm[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      int t = t0 + ty * 4 + i, e = e0 + tx * 4 + j;
      if (t < T && e < E) {
        float v = acc[i][j];
        if (bias) v += bias[e];
        logits[(int64_t)t * E + e] = v;
      }
    }
}

cudaError_t launch_router_logits_simt(int T, int H, int E, const float *x, const float *wr, const float *bias,
                                      float *logits, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  dim3 grid((unsigned)ceil_div(T, 64), (unsigned)ceil_div(E, 64));
  return launch_pdl(router_logits_simt_kernel<float>, grid, dim3(256), 0, stream, T, H, E, x, wr, bias, logits);
}

// ---------------------------------------------------------------------------
// Top-k + weights + shared gate, one warp per token.
//
// Each candidate expert e is ranked by (order value of its logit, -e):
// numbers above NaNs above already-taken slots, larger logit first, equal
// logits to the lower expert id.  Every lane keeps the best of its own
// candidates; a round takes the warp maximum (a strict total order, so the
// result does not depend on the reduction shape) and only the winning lane
// rescans.  Slot s receives the s-th winner, which is the stable descending
// order of the logits.
//
// Weights: w_s = exp(l_s - l_0) / sum_j exp(l_j - l_0) over the k selected
// logits (l_0 is the largest), the softmax over all experts followed by
// renormalisation of the selected ones; the sum runs over s = 0..k-1.
// Shared gate: z = x . w_sg, lane-partial sums in ascending h per lane, then
// a fixed butterfly; sig = 1 / (1 + exp(-z)).
// ---------------------------------------------------------------------------
// Unsigned order of a logit: 0 = taken / absent, 1 = NaN, numbers above, a
// larger logit giving a larger value (-0 and +0 map to the same value).
__device__ inline uint32_t topk_ord(float l) {
  if (l != l) return 1u;
  const uint32_t u = __float_as_uint(l + 0.0f);  // -0 -> +0: equal logits must tie
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ inline float ord_logit(uint32_t o) {
  if (o == 1u) return __uint_as_float(0x7FC00000u);  // NaN
  return __uint_as_float((o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o);
}

// (o, e) ranks above (bo, be): larger order value, or equal and lower id.
__device__ inline bool topk_better(uint32_t o, int e, uint32_t bo, int be) {
  return o > bo || (o == bo && e < be);
}

// Order values are formed once per token; the gate operands are loaded in
// small batches so that the kernel stays within 64 registers (four 256-thread
// blocks per SM).
constexpr int GATE_BATCH = 4;  // 16-byte chunks of x / w_sg loaded together per lane

// Shared-expert gate logit x_t . w_sg of one token, by one warp: lane chunks
// h = (lane + 32 m) VN, m ascending, summed in that order per lane, then a
// fixed butterfly (every lane returns the same value).
template <typename TX>
__device__ inline float gate_dot(const TX *__restrict__ xr, const TX *__restrict__ wsg, int H, int lane) {
  constexpr int VN = Vec16<TX>::N;
  float part = 0.f;
  for (int h0 = lane * VN; h0 < H; h0 += 32 * VN * GATE_BATCH) {
    uint4 xa[GATE_BATCH], ga[GATE_BATCH];
#pragma unroll
    for (int i = 0; i < GATE_BATCH; ++i) {
      const int h = h0 + 32 * VN * i;
      if (h < H) {
        xa[i] = __ldg(reinterpret_cast<const uint4 *>(xr + h));
        ga[i] = __ldg(reinterpret_cast<const uint4 *>(wsg + h));
      }
    }
#pragma unroll
    for (int i = 0; i < GATE_BATCH; ++i) {
      if (h0 + 32 * VN * i < H) {
        float xv[VN], gv[VN];
        Vec16<TX>::unpack(xa[i], xv);
        Vec16<TX>::unpack(ga[i], gv);
#pragma unroll
        for (int j = 0; j < VN; ++j) part = fmaf(xv[j], gv[j], part);
      }
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(FULL_MASK, part, off);
  return part;
}

template <typename TX, int EPL>
__global__ void __launch_bounds__(256, 4)
topk_gate_kernel(int T, int H, int E, int k, const float *__restrict__ logits, const TX *__restrict__ x,
                 const TX *__restrict__ wsg, int32_t *__restrict__ ids, float *__restrict__ w,
                 float *__restrict__ sig) {
  griddep_launch();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;

  // The token's logits are requested first, so that they arrive while the
  // gate operands stream in.
  float lv[EPL];
  const float *lrow = logits + t * E;
#pragma unroll
  for (int i = 0; i < EPL; ++i) lv[i] = lane + 32 * i < E ? __ldg(lrow + lane + 32 * i) : 0.f;

  const float part = gate_dot<TX>(x + t * (int64_t)H, wsg, H, lane);

  // Top-k: order values formed once; the winner's owner zeroes its value and rescans.
  uint32_t ov[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) ov[i] = lane + 32 * i < E ? topk_ord(lv[i]) : 0u;
  // Each lane keeps its best and second-best candidates (ties: lower slot =
  // lower id first).  When the lane's best wins, the second is promoted; only
  // when no valid second is left does the lane rescan its candidates.
  uint32_t bo = 0u, bo2 = 0u;
  int bi = 0, bi2 = 0;
#pragma unroll
  for (int i = 0; i < EPL; ++i) {
    if (ov[i] > bo) bo2 = bo, bi2 = bi, bo = ov[i], bi = i;
    else if (ov[i] > bo2) bo2 = ov[i], bi2 = i;
  }
  bool has2 = true;

  float sel_v = 0.f;  // lane s keeps the logit of slot s
  int sel_e = 0;
  for (int s = 0; s < k; ++s) {
    // Warp maximum of the lanes' best order values, then the lowest expert
    // id among the lanes that hold it (the strict total order of above).
    const uint32_t mo = __reduce_max_sync(FULL_MASK, bo);
    const int me = (int)__reduce_min_sync(FULL_MASK, bo == mo ? (uint32_t)(lane + 32 * bi) : 0xFFFFFFFFu);
    if (lane == s) {
      sel_v = ord_logit(mo);
      sel_e = me;
    }
    if (lane == (me & 31)) {  // the owner drops the winner
#pragma unroll
      for (int i = 0; i < EPL; ++i)
        if (i == bi) ov[i] = 0u;
      if (has2) {
        bo = bo2, bi = bi2, has2 = false;
      } else {
        bo = bo2 = 0u;
        bi = bi2 = 0;
#pragma unroll
        for (int i = 0; i < EPL; ++i) {
          if (ov[i] > bo) bo2 = bo, bi2 = bi, bo = ov[i], bi = i;
          else if (ov[i] > bo2) bo2 = ov[i], bi2 = i;
        }
        has2 = true;
      }
    }
  }

  // Route weights: lane s forms exp(l_s - l_0) once; every lane sums them in slot order.
  const float m0 = __shfl_sync(FULL_MASK, sel_v, 0);
  const float ex = lane < k ? expf(sel_v - m0) : 0.f;
  float z = 0.f;
  for (int s = 0; s < k; ++s) z += __shfl_sync(FULL_MASK, ex, s);
  if (lane < k) {
    ids[t * k + lane] = sel_e;
    w[t * k + lane] = ex / z;
  }
  if (lane == 0) sig[t] = sigmoid_f32(part);
}

// ---------------------------------------------------------------------------
// Router replay: the k experts of each token are given (the routes of an
// earlier pass); only the route weights and the shared gate are computed,
// with the same formulas as above: w_s = exp(l_s - m) / sum_j exp(l_j - m)
// over the given slots in their order, m = the largest of the k logits.  Ids
// out of range or repeated within a token fail closed: the token's weights
// are written as zeros and the device status records code 1 (out of range)
// or 4 (repeated).
// ---------------------------------------------------------------------------
template <typename TX>
__global__ void __launch_bounds__(256)
replay_gate_kernel(int T, int H, int E, int k, const float *__restrict__ logits, const TX *__restrict__ x,
                   const TX *__restrict__ wsg, const int32_t *__restrict__ ids, float *__restrict__ w,
                   float *__restrict__ sig, int *status) {
  griddep_launch();
  griddep_wait();
  const int lane = threadIdx.x & 31;
  const int64_t t = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  if (t >= T) return;
  const int e = lane < k ? __ldg(ids + t * k + lane) : -1;
  const bool in_range = e >= 0 && e < E;
  const unsigned dup = __match_any_sync(FULL_MASK, e);
  const bool bad_range = __any_sync(FULL_MASK, lane < k && !in_range);
  const bool bad_dup = __any_sync(FULL_MASK, lane < k && __popc(dup) > 1);
  const float l = lane < k && in_range ? __ldg(logits + t * E + e) : -INFINITY;
  const float part = gate_dot<TX>(x + t * (int64_t)H, wsg, H, lane);
  float m = l;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(FULL_MASK, m, off));
  const float ex = lane < k ? expf(l - m) : 0.f;
  float z = 0.f;
  for (int s = 0; s < k; ++s) z += __shfl_sync(FULL_MASK, ex, s);
  if (lane < k) w[t * k + lane] = (bad_range || bad_dup) ? 0.f : ex / z;
  if (lane == 0) {
    sig[t] = sigmoid_f32(part);
    if (bad_range) record_status(status, STATUS_BAD_EXPERT_ID);
    else if (bad_dup) record_status(status, STATUS_REPEATED_EXPERT_ID);
  }
}

cudaError_t launch_replay_gate(int dtype, int T, int H, int E, int k, const float *logits, const void *x,
                               const void *w_shared_gate, const int32_t *ids, float *w, float *sig, int *status,
                               cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  const dim3 grid((unsigned)ceil_div(T, 8));
  if (dtype == 0)
    return launch_pdl(replay_gate_kernel<float>, grid, dim3(256), 0, stream, T, H, E, k, logits, (const float *)x,
                      (const float *)w_shared_gate, ids, w, sig, status);
  return launch_pdl(replay_gate_kernel<__nv_bfloat16>, grid, dim3(256), 0, stream, T, H, E, k, logits,
                    (const __nv_bfloat16 *)x, (const __nv_bfloat16 *)w_shared_gate, ids, w, sig, status);
}

template <typename TX>
static cudaError_t topk_dispatch(int T, int H, int E, int k, const float *logits, const void *x, const void *wsg,
                                 int32_t *ids, float *w, float *sig, cudaStream_t stream) {
  dim3 grid((unsigned)ceil_div(T, 8));
  const TX *xx = (const TX *)x;
  const TX *gg = (const TX *)wsg;
#define MOE_TOPK(EPL) \
  launch_pdl(topk_gate_kernel<TX, EPL>, grid, dim3(256), 0, stream, T, H, E, k, logits, xx, gg, ids, w, sig)
  if (E <= 32) return MOE_TOPK(1);
  if (E <= 64) return MOE_TOPK(2);
  if (E <= 128) return MOE_TOPK(4);
  if (E <= 256) return MOE_TOPK(8);
  if (E <= 512) return MOE_TOPK(16);
  return MOE_TOPK(32);
#undef MOE_TOPK
}

cudaError_t launch_topk_gate(int dtype, int T, int H, int E, int k, const float *logits, const void *x,
                             const void *w_shared_gate, int32_t *ids, float *w, float *sig, cudaStream_t stream) {
  if (T == 0) return cudaSuccess;
  if (dtype == 0) return topk_dispatch<float>(T, H, E, k, logits, x, w_shared_gate, ids, w, sig, stream);
  return topk_dispatch<__nv_bfloat16>(T, H, E, k, logits, x, w_shared_gate, ids, w, sig, stream);
}

}  // namespace moe
