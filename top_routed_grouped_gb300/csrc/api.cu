// C ABI of the MoE layer (declarations and contracts in include/moe.h):
// argument validation, workspace carving and the launch sequence of each
// entry point.  No device memory is allocated here.
#include <mutex>

#include "../../include/moe.h"
#include "common.cuh"
#include "kernels.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {

// Device status word: first failed device-side check since the last reset.
__device__ int g_moe_status;

int *device_status_ptr() {
  static std::mutex mu;
  static int *cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_moe_status) != cudaSuccess) return nullptr;
    cache[dev] = (int *)p;
  }
  return cache[dev];
}

// Sequential sub-allocation of the caller's workspace at 256-byte alignment.
// With base == nullptr it only measures.
struct Carver {
  char *base;
  size_t off = 0;
  explicit Carver(void *b) : base((char *)b) {}
  void *take(size_t bytes) {
    size_t o = (size_t)round_up((int64_t)off, 256);
    off = o + bytes;
    return base ? (void *)(base + o) : nullptr;
  }
};

static size_t esize(const moe_dims_t *d) { return d->dtype == MOE_F32 ? 4 : 2; }

static int check_dims(const moe_dims_t *d) {
  if (!d) return MOE_ERR_INVALID_ARG;
  if (d->T < 0 || d->H <= 0 || d->E <= 0 || d->k <= 0 || d->I <= 0 || d->Is <= 0) return MOE_ERR_INVALID_ARG;
  if (d->k > d->E || d->k > 16) return MOE_ERR_INVALID_ARG;
  if (d->dtype != MOE_F32 && d->dtype != MOE_BF16) return MOE_ERR_INVALID_ARG;
  if (d->E > 1024) return MOE_ERR_UNSUPPORTED;
  if ((int64_t)d->T * d->k >= ((int64_t)1 << 31)) return MOE_ERR_UNSUPPORTED;
  if (d->dtype == MOE_F32) {
    if (d->H % 4 || d->I % 4 || d->Is % 4) return MOE_ERR_UNSUPPORTED;
  } else {
    if (d->H % 256 || d->I % 128 || d->Is % 128) return MOE_ERR_UNSUPPORTED;
  }
  return MOE_OK;
}

// A buffer of `n` elements: may be NULL only when empty; else 16-byte aligned.
static bool buf_ok(const void *p, int64_t n) {
  if (n == 0) return true;
  return p != nullptr && ((uintptr_t)p & 15) == 0;
}

static bool opt_ok(const void *p) { return p == nullptr || ((uintptr_t)p & 15) == 0; }

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---------------------------------------------------------------- sizes
static void route_ws(const moe_dims_t *d, Carver &c) {
  c.take((size_t)d->T * d->E * sizeof(float));  // logits when the caller passes none
  if (d->dtype == MOE_BF16) c.take(router_tc_scratch_bytes(d->T, d->E, d->H));  // split router weight
}

static void permute_ws(const moe_dims_t *d, Carver &c) {
  c.take(permute_scratch_bytes((int64_t)d->T * d->k, d->E));
}

struct FfnScratch {
  void *tiles, *h_routed, *h_shared;
};

static FfnScratch ffn_ws(const moe_dims_t *d, Carver &c) {
  FfnScratch s;
  const int64_t R = (int64_t)d->T * d->k;
  s.tiles = c.take(d->dtype == MOE_F32 ? ffn_simt_scratch_bytes(d->E) : ffn_tc_scratch_bytes(d->T, d->k, d->E, d->H, d->I, d->Is));
  s.h_routed = c.take((size_t)R * d->I * esize(d));
  s.h_shared = c.take((size_t)d->T * d->Is * esize(d));
  return s;
}

struct FwdScratch {
  int32_t *ids;
  float *w, *sig;
  int32_t *offsets, *sorted_route, *route_pos;
  void *y_routed, *y_shared;
  void *inner;  // scratch shared by the four steps (they run one after another)
  size_t inner_bytes;
  void *side_tiles, *side_h_shared;  // bf16: the shared expert's item tables and h (its own stream)
};

static FwdScratch fwd_ws(const moe_dims_t *d, Carver &c) {
  FwdScratch s;
  const int64_t R = (int64_t)d->T * d->k;
  s.ids = (int32_t *)c.take((size_t)R * 4);
  s.w = (float *)c.take((size_t)R * 4);
  s.sig = (float *)c.take((size_t)d->T * 4);
  s.offsets = (int32_t *)c.take((size_t)(d->E + 1) * 4);
  s.sorted_route = (int32_t *)c.take((size_t)R * 4);
  s.route_pos = (int32_t *)c.take((size_t)R * 4);
  s.y_routed = c.take((size_t)R * d->H * esize(d));
  s.y_shared = c.take((size_t)d->T * d->H * esize(d));
  Carver a(nullptr), b(nullptr), f(nullptr);
  route_ws(d, a);
  permute_ws(d, b);
  ffn_ws(d, f);
  size_t inner = a.off;
  if (b.off > inner) inner = b.off;
  if (f.off > inner) inner = f.off;
  s.inner_bytes = (size_t)round_up((int64_t)inner, 256);
  s.inner = c.take(s.inner_bytes);
  s.side_tiles = s.side_h_shared = nullptr;
  if (d->dtype == MOE_BF16) {
    s.side_tiles = c.take(ffn_tc_scratch_bytes(d->T, d->k, d->E, d->H, d->I, d->Is));
    s.side_h_shared = c.take((size_t)d->T * d->Is * esize(d));
  }
  return s;
}

// The second stream of the shared expert (one per device, created once).
static cudaStream_t side_stream() {
  static std::mutex mu;
  static cudaStream_t streams[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  cudaStream_t &s = streams[dev & 63];
  if (!s && cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) s = nullptr;
  return s;
}


struct BwdScratch {
  void *dyr, *dys, *dgu_routed, *dgu_shared;
  float *dxr, *dxs, *dlogit, *dz;
  void *x_sorted;
  void *inner;
};

static BwdScratch bwd_ws(const moe_dims_t *d, Carver &c) {
  BwdScratch s;
  const int64_t T = d->T, R = T * d->k;
  s.dyr = c.take((size_t)R * d->H * esize(d));
  s.dys = c.take((size_t)T * d->H * esize(d));
  s.dgu_routed = c.take((size_t)R * 2 * d->I * esize(d));
  s.dgu_shared = c.take((size_t)T * 2 * d->Is * esize(d));
  s.dxr = (float *)c.take((size_t)R * d->H * sizeof(float));
  s.dxs = (float *)c.take((size_t)T * d->H * sizeof(float));
  s.dlogit = (float *)c.take((size_t)R * sizeof(float));
  s.dz = (float *)c.take((size_t)T * sizeof(float));
  s.x_sorted = (d->dtype == MOE_BF16 && backward_tc_supported(d->H, d->I, d->Is))
                   ? c.take((size_t)R * d->H * esize(d)) : nullptr;
  s.inner = c.take(backward_scratch_bytes(d->dtype, d->T, d->k, d->E, d->H, d->I, d->Is));
  return s;
}

static size_t ws_size(const moe_dims_t *d, int op) {
  Carver c(nullptr);
  switch (op) {
    case MOE_OP_BACKWARD: bwd_ws(d, c); break;
    case MOE_OP_ROUTE: route_ws(d, c); break;
    case MOE_OP_PERMUTE: permute_ws(d, c); break;
    case MOE_OP_GROUPED_FFN: ffn_ws(d, c); break;
    case MOE_OP_COMBINE: break;
    case MOE_OP_FORWARD: fwd_ws(d, c); break;
    default: return 0;
  }
  return (size_t)round_up((int64_t)c.off, 256);
}

}  // namespace moe

using namespace moe;

MOE_API size_t moe_workspace_size(const moe_dims_t *d, int op) {
  if (check_dims(d) != MOE_OK) return 0;
  return ws_size(d, op);
}

MOE_API const char *moe_status_string(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument (null or misaligned pointer, bad size, k > E or k > 16)";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or dtype";
    case MOE_ERR_WORKSPACE: return "workspace too small";
    case MOE_ERR_CUDA: return "CUDA runtime error";
    case MOE_ERR_DEVICE: return "a kernel recorded a failed device-side check";
    default: return "unknown status";
  }
}

// moe_route (replay == nullptr: top-k of the logits into topk_ids) and
// moe_route_replay (the given ids, replay == topk_ids).  `after_router` runs
// on the host between the router launch and the top-k (or replay gate)
// launch; moe_forward forks its second stream there.
template <class F>
static int route_impl(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
                      const void *w_shared_gate, const int32_t *replay, int32_t *topk_ids, float *topk_w,
                      float *shared_sig, float *logits, void *ws, size_t ws_bytes, void *stream, F &&after_router) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  const int64_t T = d->T, R = T * d->k;
  const int32_t *ids_in = replay ? replay : topk_ids;
  if (!buf_ok(x, T * d->H) || !buf_ok(w_router, 1) || !opt_ok(router_bias) || !buf_ok(w_shared_gate, 1) ||
      !buf_ok(ids_in, R) || !buf_ok(topk_w, R) || !buf_ok(shared_sig, T) || !opt_ok(logits) || !opt_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_ROUTE)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  Carver c(ws);
  float *lg = (float *)c.take((size_t)T * d->E * sizeof(float));
  if (logits) lg = logits;
  cudaError_t e;
  if (d->dtype == MOE_F32)
    e = launch_router_logits_simt(d->T, d->H, d->E, (const float *)x, w_router, router_bias, lg, s);
  else
    e = launch_router_logits_tc(d->T, d->H, d->E, x, w_router, router_bias, lg,
                                c.take(router_tc_scratch_bytes(d->T, d->E, d->H)), device_status_ptr(), s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  st = after_router();
  if (st != MOE_OK) return st;
  if (replay)
    e = launch_replay_gate(d->dtype, d->T, d->H, d->E, d->k, lg, x, w_shared_gate, replay, topk_w, shared_sig,
                           device_status_ptr(), s);
  else
    e = launch_topk_gate(d->dtype, d->T, d->H, d->E, d->k, lg, x, w_shared_gate, topk_ids, topk_w, shared_sig, s);
  return cuda_status(e);
}

MOE_API int moe_route(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
                      const void *w_shared_gate, int32_t *topk_ids, float *topk_w, float *shared_sig, float *logits,
                      void *ws, size_t ws_bytes, void *stream) {
  return route_impl(d, x, w_router, router_bias, w_shared_gate, nullptr, topk_ids, topk_w, shared_sig, logits, ws,
                    ws_bytes, stream, [] { return (int)MOE_OK; });
}

MOE_API int moe_router_logits(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
                              int32_t exact, float *logits, void *ws, size_t ws_bytes, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  if (exact != 0 && exact != 1) return MOE_ERR_INVALID_ARG;
  const int64_t T = d->T;
  if (!buf_ok(x, T * d->H) || !buf_ok(w_router, 1) || !opt_ok(router_bias) || !buf_ok(logits, T * d->E) ||
      !opt_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (d->dtype == MOE_F32 && !exact) return MOE_ERR_UNSUPPORTED;
  if (ws_bytes < ws_size(d, MOE_OP_ROUTE)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  cudaStream_t s = (cudaStream_t)stream;
  Carver c(ws);
  c.take((size_t)T * d->E * sizeof(float));  // the logits slot of the ROUTE layout (unused here)
  if (d->dtype == MOE_F32)
    return cuda_status(launch_router_logits_simt(d->T, d->H, d->E, (const float *)x, w_router, router_bias, logits, s));
  return cuda_status(launch_router_logits_tc(d->T, d->H, d->E, x, w_router, router_bias, logits,
                                             c.take(router_tc_scratch_bytes(d->T, d->E, d->H)), device_status_ptr(), s,
                                             exact ? 3 : 1));
}

MOE_API int moe_route_replay(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
                             const void *w_shared_gate, const int32_t *topk_ids, float *topk_w, float *shared_sig,
                             float *logits, void *ws, size_t ws_bytes, void *stream) {
  return route_impl(d, x, w_router, router_bias, w_shared_gate, topk_ids, nullptr, topk_w, shared_sig, logits, ws,
                    ws_bytes, stream, [] { return (int)MOE_OK; });
}

// The checks of the permutation's dims and buffers (shared by moe_permute and
// moe_permute_noalloc; the workspace is checked by moe_permute alone).
int moe::permute_args_check(const moe_dims_t *d, const int32_t *topk_ids, const int32_t *expert_offsets,
                            const int32_t *sorted_route, const int32_t *route_pos) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  const int64_t R = (int64_t)d->T * d->k;
  if (!buf_ok(topk_ids, R) || !buf_ok(expert_offsets, 1) || !buf_ok(sorted_route, R) || !buf_ok(route_pos, R))
    return MOE_ERR_INVALID_ARG;
  return MOE_OK;
}

static int permute_check(const moe_dims_t *d, const int32_t *topk_ids, int32_t *expert_offsets,
                         int32_t *sorted_route, int32_t *route_pos, void *ws, size_t ws_bytes) {
  int st = permute_args_check(d, topk_ids, expert_offsets, sorted_route, route_pos);
  if (st != MOE_OK) return st;
  if (!opt_ok(ws)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_PERMUTE)) return MOE_ERR_WORKSPACE;
  return MOE_OK;
}

// The sort runs as one launch where the cluster it needs fits (it uses no
// workspace then), else as four kernels over the workspace; same result.
MOE_API int moe_permute(const moe_dims_t *d, const int32_t *topk_ids, int32_t *expert_offsets,
                        int32_t *sorted_route, int32_t *route_pos, void *ws, size_t ws_bytes, void *stream) {
  int st = permute_check(d, topk_ids, expert_offsets, sorted_route, route_pos, ws, ws_bytes);
  if (st != MOE_OK) return st;
  const int64_t R = (int64_t)d->T * d->k;
  if (permute_cluster_ok(R, d->E))
    return cuda_status(launch_permute_cluster(R, d->E, topk_ids, expert_offsets, sorted_route, route_pos,
                                              device_status_ptr(), (cudaStream_t)stream));
  return cuda_status(launch_permute(R, d->E, topk_ids, expert_offsets, sorted_route, route_pos, ws, device_status_ptr(),
                                    (cudaStream_t)stream));
}

// Checks the arguments of moe_grouped_ffn and fills `a` and `sc` (MOE_OK), or
// returns the error.
static int grouped_ffn_prepare(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                               const int32_t *sorted_route, const void *w_gate_up, const void *w_down,
                               const void *ws_gate_up, const void *ws_down, void *y_routed, void *y_shared,
                               const moe_saved_t *saved, void *ws, size_t ws_bytes, FfnArgs *a, FfnScratch *sc) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  const int64_t T = d->T, R = T * d->k;
  if (!buf_ok(x, T * d->H) || !buf_ok(expert_offsets, 1) || !buf_ok(sorted_route, R) || !buf_ok(w_gate_up, 1) ||
      !buf_ok(w_down, 1) || !buf_ok(ws_gate_up, 1) || !buf_ok(ws_down, 1) || !buf_ok(y_routed, R * d->H) ||
      !buf_ok(y_shared, T * d->H) || !opt_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (saved && (!opt_ok(saved->gu) || !opt_ok(saved->h) || !opt_ok(saved->gu_shared) || !opt_ok(saved->h_shared)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_GROUPED_FFN)) return MOE_ERR_WORKSPACE;
  Carver c(ws);
  *sc = ffn_ws(d, c);
  a->T = d->T; a->H = d->H; a->E = d->E; a->k = d->k; a->I = d->I; a->Is = d->Is;
  a->x = x; a->offsets = expert_offsets; a->sorted_route = sorted_route;
  a->w_gate_up = w_gate_up; a->w_down = w_down; a->ws_gate_up = ws_gate_up; a->ws_down = ws_down;
  a->y_routed = y_routed; a->y_shared = y_shared;
  a->h_routed = (saved && saved->h) ? saved->h : sc->h_routed;
  a->h_shared = (saved && saved->h_shared) ? saved->h_shared : sc->h_shared;
  a->gu_routed = saved ? saved->gu : nullptr;
  a->gu_shared = saved ? saved->gu_shared : nullptr;
  return MOE_OK;
}

static int grouped_ffn_run(const moe_dims_t *d, const FfnArgs &a, const FfnScratch &sc, void *stream) {
  if (d->T == 0) return MOE_OK;
  if (d->dtype == MOE_F32) return cuda_status(launch_ffn_simt(a, sc.tiles, (cudaStream_t)stream));
  return cuda_status(launch_ffn_tc(a, sc.tiles, device_status_ptr(), (cudaStream_t)stream));
}

MOE_API int moe_grouped_ffn(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                            const int32_t *sorted_route, const void *w_gate_up, const void *w_down,
                            const void *ws_gate_up, const void *ws_down, void *y_routed, void *y_shared,
                            const moe_saved_t *saved, void *ws, size_t ws_bytes, void *stream) {
  FfnArgs a;
  FfnScratch sc;
  int st = grouped_ffn_prepare(d, x, expert_offsets, sorted_route, w_gate_up, w_down, ws_gate_up, ws_down, y_routed,
                               y_shared, saved, ws, ws_bytes, &a, &sc);
  if (st != MOE_OK) return st;
  return grouped_ffn_run(d, a, sc, stream);
}

MOE_API int moe_grouped_ffn_etp(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                                const int32_t *sorted_route, const void *w_gate_up, const void *w_down,
                                const void *ws_gate_up, const void *ws_down, float *yr_partial, float *ys_partial,
                                const moe_saved_t *saved, void *ws, size_t ws_bytes, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  const int64_t T = d->T, R = T * d->k;
  if (!buf_ok(x, T * d->H) || !buf_ok(expert_offsets, 1) || !buf_ok(sorted_route, R) || !buf_ok(w_gate_up, 1) ||
      !buf_ok(w_down, 1) || !buf_ok(ws_gate_up, 1) || !buf_ok(ws_down, 1) || !buf_ok(yr_partial, R * d->H) ||
      !buf_ok(ys_partial, T * d->H) || !opt_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (saved && (!opt_ok(saved->gu) || !opt_ok(saved->h) || !opt_ok(saved->gu_shared) || !opt_ok(saved->h_shared)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_GROUPED_FFN)) return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  Carver c(ws);
  FfnScratch sc = ffn_ws(d, c);
  FfnArgs a;
  a.T = d->T; a.H = d->H; a.E = d->E; a.k = d->k; a.I = d->I; a.Is = d->Is;
  a.x = x; a.offsets = expert_offsets; a.sorted_route = sorted_route;
  a.w_gate_up = w_gate_up; a.w_down = w_down; a.ws_gate_up = ws_gate_up; a.ws_down = ws_down;
  a.y_routed = yr_partial; a.y_shared = ys_partial;
  a.y_f32 = 1;
  a.h_routed = (saved && saved->h) ? saved->h : sc.h_routed;
  a.h_shared = (saved && saved->h_shared) ? saved->h_shared : sc.h_shared;
  a.gu_routed = saved ? saved->gu : nullptr;
  a.gu_shared = saved ? saved->gu_shared : nullptr;
  // The FP32 path's rows are float already: the partial sums are its outputs.
  if (d->dtype == MOE_F32) return cuda_status(launch_ffn_simt(a, sc.tiles, (cudaStream_t)stream));
  return cuda_status(launch_ffn_tc(a, sc.tiles, device_status_ptr(), (cudaStream_t)stream));
}

MOE_API int moe_grouped_ffn_etp_fused(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                                      const int32_t *sorted_route, const void *w_gate_up, const void *w_down,
                                      const void *ws_gate_up, const void *ws_down, float *yr_partial, float *ys_partial,
                                      void *ws, size_t ws_bytes, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  if (d->dtype != MOE_BF16 || !etp_fused_supported(d->H, d->I, d->Is)) return MOE_ERR_UNSUPPORTED;
  const int64_t T = d->T, R = T * d->k;
  if (!buf_ok(x, T * d->H) || !buf_ok(expert_offsets, 1) || !buf_ok(sorted_route, R) || !buf_ok(w_gate_up, 1) ||
      !buf_ok(w_down, 1) || !buf_ok(ws_gate_up, 1) || !buf_ok(ws_down, 1) || !buf_ok(yr_partial, R * d->H) ||
      !buf_ok(ys_partial, T * d->H) || !opt_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_GROUPED_FFN) || ws_bytes < etp_fused_scratch_bytes(d->T, d->k, d->E))
    return MOE_ERR_WORKSPACE;
  if (T == 0) return MOE_OK;
  FfnArgs a;
  a.T = d->T; a.H = d->H; a.E = d->E; a.k = d->k; a.I = d->I; a.Is = d->Is;
  a.x = x; a.offsets = expert_offsets; a.sorted_route = sorted_route;
  a.w_gate_up = w_gate_up; a.w_down = w_down; a.ws_gate_up = ws_gate_up; a.ws_down = ws_down;
  a.y_routed = yr_partial; a.y_shared = ys_partial;
  a.y_f32 = 1;
  return cuda_status(launch_etp_fused(a, ws, device_status_ptr(), (cudaStream_t)stream));
}

MOE_API int moe_etp_reduce(const moe_dims_t *d, int32_t n_parts, const float *const *yr_parts,
                           const float *const *ys_parts, void *y_routed, void *y_shared, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  if (n_parts < 1 || n_parts > ETP_MAX_PARTS || !yr_parts || !ys_parts) return MOE_ERR_INVALID_ARG;
  const int64_t T = d->T, R = T * d->k;
  for (int q = 0; q < n_parts; ++q)
    if (!buf_ok(yr_parts[q], R * d->H) || !buf_ok(ys_parts[q], T * d->H)) return MOE_ERR_INVALID_ARG;
  if (!buf_ok(y_routed, R * d->H) || !buf_ok(y_shared, T * d->H)) return MOE_ERR_INVALID_ARG;
  if (T == 0) return MOE_OK;
  const int dtype = d->dtype == MOE_F32 ? 0 : 1;
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e = launch_etp_reduce(dtype, n_parts, yr_parts, R * d->H, y_routed, s);
  if (e != cudaSuccess) return cuda_status(e);
  return cuda_status(launch_etp_reduce(dtype, n_parts, ys_parts, T * d->H, y_shared, s));
}

MOE_API int moe_grouped_ffn_ep(const moe_dims_t *d, int32_t e_begin, int32_t e_end, int32_t with_shared,
                               const void *x, const int32_t *expert_offsets, const int32_t *sorted_route,
                               const void *w_gate_up, const void *w_down, const void *ws_gate_up, const void *ws_down,
                               void *y_sorted, void *y_shared, const moe_saved_t *saved, void *ws, size_t ws_bytes,
                               void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  if (e_begin < 0 || e_end < e_begin || e_end > d->E || (with_shared != 0 && with_shared != 1))
    return MOE_ERR_INVALID_ARG;
  const int64_t T = d->T, R = T * d->k, n_local = e_end - e_begin;
  if (!buf_ok(x, T * d->H) || !buf_ok(expert_offsets, 1) || !buf_ok(sorted_route, R) || !buf_ok(w_gate_up, n_local) ||
      !buf_ok(w_down, n_local) || !buf_ok(ws_gate_up, with_shared) || !buf_ok(ws_down, with_shared) ||
      !buf_ok(y_sorted, n_local ? R * d->H : 0) || !buf_ok(y_shared, with_shared ? T * d->H : 0) || !opt_ok(ws))
    return MOE_ERR_INVALID_ARG;
  if (saved && (!opt_ok(saved->gu) || !opt_ok(saved->h) || !opt_ok(saved->gu_shared) || !opt_ok(saved->h_shared)))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_GROUPED_FFN)) return MOE_ERR_WORKSPACE;
  if (T == 0 || (n_local == 0 && !with_shared)) return MOE_OK;
  Carver c(ws);
  FfnScratch sc = ffn_ws(d, c);
  FfnArgs a;
  a.T = d->T; a.H = d->H; a.E = d->E; a.k = d->k; a.I = d->I; a.Is = d->Is;
  a.x = x; a.offsets = expert_offsets; a.sorted_route = sorted_route;
  // The maps of an unused half still need a valid address; nothing is read through them.
  a.w_gate_up = n_local ? w_gate_up : ws_gate_up;
  a.w_down = n_local ? w_down : ws_down;
  a.ws_gate_up = with_shared ? ws_gate_up : a.w_gate_up;
  a.ws_down = with_shared ? ws_down : a.w_down;
  a.y_routed = y_sorted; a.y_shared = y_shared;
  a.h_routed = (saved && saved->h) ? saved->h : sc.h_routed;
  a.h_shared = (saved && saved->h_shared) ? saved->h_shared : sc.h_shared;
  a.gu_routed = saved ? saved->gu : nullptr;
  a.gu_shared = saved ? saved->gu_shared : nullptr;
  a.e_begin = e_begin; a.e_end = e_end; a.with_shared = with_shared; a.y_sorted = 1;
  if (d->dtype == MOE_F32) return cuda_status(launch_ffn_simt(a, sc.tiles, (cudaStream_t)stream));
  return cuda_status(launch_ffn_tc(a, sc.tiles, device_status_ptr(), (cudaStream_t)stream));
}

MOE_API int moe_combine_sorted(const moe_dims_t *d, const void *y_sorted, const int32_t *route_pos,
                               const void *y_shared, const float *topk_w, const float *shared_sig, void *y,
                               void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  const int64_t T = d->T, R = T * d->k;
  if (!buf_ok(y_sorted, R * d->H) || !buf_ok(route_pos, R) || !buf_ok(y_shared, T * d->H) || !buf_ok(topk_w, R) ||
      !buf_ok(shared_sig, T) || !buf_ok(y, T * d->H))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(d->dtype, d->T, d->H, d->k, y_sorted, y_shared, topk_w, shared_sig, y,
                                    (cudaStream_t)stream, route_pos));
}

MOE_API int moe_combine(const moe_dims_t *d, const void *y_routed, const void *y_shared, const float *topk_w,
                        const float *shared_sig, void *y, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  const int64_t T = d->T, R = T * d->k;
  if (!buf_ok(y_routed, R * d->H) || !buf_ok(y_shared, T * d->H) || !buf_ok(topk_w, R) || !buf_ok(shared_sig, T) ||
      !buf_ok(y, T * d->H))
    return MOE_ERR_INVALID_ARG;
  return cuda_status(launch_combine(d->dtype, d->T, d->H, d->k, y_routed, y_shared, topk_w, shared_sig, y,
                                    (cudaStream_t)stream));
}

MOE_API int moe_forward(const moe_dims_t *d, const moe_fwd_args_t *a, void *ws, size_t ws_bytes, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!a || !opt_ok(ws)) return MOE_ERR_INVALID_ARG;
  const int64_t T = d->T, R = T * d->k;
  if (!buf_ok(a->x, T * d->H) || !buf_ok(a->y, T * d->H)) return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_FORWARD)) return MOE_ERR_WORKSPACE;
  Carver c(ws);
  FwdScratch s = fwd_ws(d, c);
  int32_t *ids = a->topk_ids ? a->topk_ids : s.ids;
  float *w = a->topk_w ? a->topk_w : s.w;
  float *sig = a->shared_sig ? a->shared_sig : s.sig;
  int32_t *off = a->expert_offsets ? a->expert_offsets : s.offsets;
  int32_t *srt = a->sorted_route ? a->sorted_route : s.sorted_route;
  int32_t *pos = a->route_pos ? a->route_pos : s.route_pos;
  void *yr = a->y_routed ? a->y_routed : s.y_routed;
  void *ys = a->y_shared ? a->y_shared : s.y_shared;
  if (a->replay_ids && !buf_ok(a->replay_ids, T * d->k)) return MOE_ERR_INVALID_ARG;
  const int32_t *route_ids = a->replay_ids ? a->replay_ids : ids;
  st = permute_check(d, route_ids, off, srt, pos, s.inner, s.inner_bytes);
  if (st != MOE_OK) return st;
  FfnArgs fa;
  FfnScratch fs;
  st = grouped_ffn_prepare(d, a->x, off, srt, a->w_gate_up, a->w_down, a->ws_gate_up, a->ws_down, yr, ys, &a->saved,
                           s.inner, s.inner_bytes, &fa, &fs);
  if (st != MOE_OK) return st;
  cudaStream_t ms = (cudaStream_t)stream;
  // On the bf16 path with the one-launch sort, the shared expert needs no
  // routes: above 2048 tokens its GEMMs run on a second stream, joined before
  // the combine, with their own rows and tables in scratch.  The routed GEMMs
  // then take only the routed segments (the sort writes their tables); every
  // output is the same MMA chain as in one launch.  Where the routed GEMMs
  // stream their weights (fewer than 256 routes per expert on average), the
  // second stream forks after the router launch: the shared gate_up takes the
  // SMs that top-k leaves and runs beside the permute and the start of the
  // routed gate_up, the shared down beside the routed down.  With more routes
  // per expert the routed GEMMs are bound by the tensor pipe themselves, and
  // the fork comes first, so that both shared GEMMs run ahead of the router.
  // Measured on one GB300, back-to-back calls, against the shared expert as
  // items of the routed launches: T = 4096 -6 µs, 8192 -9 µs, 16384 skewed
  // -37 µs; with the other fork point +7, +3 and +10 µs more; at T = 2048 the
  // second stream would cost 8 µs.
  const bool one_launch = d->dtype == MOE_BF16 && T > 0 && permute_cluster_ok(R, d->E);
  cudaStream_t ss = (one_launch && T > 2048) ? side_stream() : nullptr;
  const bool fork_first = ss && T * d->k >= (int64_t)256 * d->E;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  if (ss && (cudaEventCreateWithFlags(&ev_fork, cudaEventDisableTiming) != cudaSuccess ||
             cudaEventCreateWithFlags(&ev_join, cudaEventDisableTiming) != cudaSuccess)) {
    if (ev_fork) cudaEventDestroy(ev_fork);
    return MOE_ERR_CUDA;
  }
  bool recorded = false;  // ev_join marks the end of the second stream's work
  // The second stream waits for the work queued so far on the caller's
  // stream (x is ready) and takes the shared expert.
  auto fork = [&]() -> int {
    if (!ss) return MOE_OK;
    FfnArgs sa = fa;
    sa.e_begin = 0;
    sa.e_end = 0;  // no routed segment
    sa.with_shared = 1;
    sa.items_ready = 0;
    if (!a->saved.h_shared) sa.h_shared = s.side_h_shared;
    fa.with_shared = 0;
    cudaError_t e = cudaEventRecord(ev_fork, ms);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(ss, ev_fork, 0);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    e = launch_ffn_tc(sa, s.side_tiles, device_status_ptr(), ss);
    recorded = cudaEventRecord(ev_join, ss) == cudaSuccess;  // also after a failed launch
    return (e == cudaSuccess && recorded) ? MOE_OK : MOE_ERR_CUDA;
  };
  // Whatever happens after the fork, the caller's stream joins the second
  // stream before returning.
  auto join = [&](int status) {
    if (!ss) return status;
    const cudaError_t e = recorded ? cudaStreamWaitEvent(ms, ev_join, 0) : cudaSuccess;
    cudaEventDestroy(ev_fork);
    cudaEventDestroy(ev_join);
    return (status == MOE_OK && e != cudaSuccess) ? MOE_ERR_CUDA : status;
  };
  auto fork_after_router = [&]() { return fork_first ? (int)MOE_OK : fork(); };
  if (fork_first && (st = fork()) != MOE_OK) return join(st);
  if (a->replay_ids) {
    st = route_impl(d, a->x, a->w_router, a->router_bias, a->w_shared_gate, a->replay_ids, nullptr, w, sig,
                    a->logits, s.inner, s.inner_bytes, stream, fork_after_router);
    if (st != MOE_OK) return join(st);
    if (a->topk_ids && a->topk_ids != a->replay_ids && T > 0 &&
        cudaMemcpyAsync(a->topk_ids, a->replay_ids, (size_t)T * d->k * sizeof(int32_t), cudaMemcpyDeviceToDevice,
                        ms) != cudaSuccess)
      return join(MOE_ERR_CUDA);
  } else {
    st = route_impl(d, a->x, a->w_router, a->router_bias, a->w_shared_gate, nullptr, ids, w, sig, a->logits, s.inner,
                    s.inner_bytes, stream, fork_after_router);
    if (st != MOE_OK) return join(st);
  }
  // Permute and grouped FFN.  On the bf16 path with the one-launch sort, that
  // launch also writes the FFN's item tables into its scratch (the sort
  // itself uses none), so the FFN starts with its GEMMs.
  PermuteItems items;
  if (one_launch && ffn_tc_item_tables(fa, fs.tiles, &items)) {
    st = cuda_status(launch_permute_cluster(R, d->E, route_ids, off, srt, pos, device_status_ptr(), ms, &items));
    fa.items_ready = 1;
  } else {
    st = moe_permute(d, route_ids, off, srt, pos, s.inner, s.inner_bytes, stream);
  }
  if (st != MOE_OK) return join(st);
  st = grouped_ffn_run(d, fa, fs, stream);
  if (st != MOE_OK) return join(st);
  st = join(MOE_OK);
  if (st != MOE_OK) return st;
  return moe_combine(d, yr, ys, w, sig, a->y, stream);
}

// moe_backward and moe_backward_ep: experts [eb, ee) run their GEMMs, weight
// arrays hold those experts only; dxr (if not NULL) receives the routed input
// gradients in sorted order instead of the workspace.
static int backward_impl(const moe_dims_t *d, const moe_bwd_args_t *a, int eb, int ee, int phase, int yr_sorted,
                         float *dxr, void *ws, size_t ws_bytes, void *stream) {
  int st = check_dims(d);
  if (st != MOE_OK) return st;
  if (!a || !opt_ok(ws) || !opt_ok(dxr)) return MOE_ERR_INVALID_ARG;
  const int64_t T = d->T, R = T * d->k, H = d->H, E = d->E, I = d->I, Is = d->Is, nl = ee - eb;
  if (!buf_ok(a->x, T * H) || !buf_ok(a->w_router, E * H) || !buf_ok(a->w_shared_gate, H) ||
      !buf_ok(a->w_gate_up, nl) || !buf_ok(a->w_down, nl) || !buf_ok(a->ws_gate_up, 1) || !buf_ok(a->ws_down, 1) ||
      !buf_ok(a->topk_ids, R) || !buf_ok(a->topk_w, R) || !buf_ok(a->shared_sig, T) ||
      !buf_ok(a->expert_offsets, 1) || !buf_ok(a->sorted_route, R) || !buf_ok(a->route_pos, R) ||
      !buf_ok(a->y_routed, R * H) || !buf_ok(a->y_shared, T * H) || !buf_ok(a->saved.gu, R * 2 * I) ||
      !buf_ok(a->saved.h, R * I) || !buf_ok(a->saved.gu_shared, T * 2 * Is) || !buf_ok(a->saved.h_shared, T * Is) ||
      !buf_ok(a->dy, T * H) || !buf_ok(a->dx, T * H) || !buf_ok(a->dw_gate_up, nl) || !buf_ok(a->dw_down, nl) ||
      !buf_ok(a->dw_router, 1) || !buf_ok(a->dw_shared_gate, 1) || !buf_ok(a->dws_gate_up, 1) ||
      !buf_ok(a->dws_down, 1) || !opt_ok(a->dlogit) || !opt_ok(a->dz))
    return MOE_ERR_INVALID_ARG;
  if (ws_bytes < ws_size(d, MOE_OP_BACKWARD)) return MOE_ERR_WORKSPACE;
  cudaStream_t s = (cudaStream_t)stream;
  if (T == 0) {  // every weight gradient is an empty sum
    if (!(phase & BWD_PHASE_EXPERTS)) return MOE_OK;
    const size_t f = sizeof(float);
    const void *bufs[6] = {a->dw_gate_up, a->dw_down, a->dw_router, a->dw_shared_gate, a->dws_gate_up, a->dws_down};
    const size_t bytes[6] = {(size_t)(nl * 2 * I * H) * f, (size_t)(nl * H * I) * f, (size_t)(E * H) * f,
                             (size_t)H * f, (size_t)(2 * Is * H) * f, (size_t)(H * Is) * f};
    for (int i = 0; i < 6; ++i) {
      if (bytes[i] == 0) continue;
      cudaError_t e = cudaMemsetAsync((void *)bufs[i], 0, bytes[i], s);
      if (e != cudaSuccess) return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  Carver c(ws);
  BwdScratch sc = bwd_ws(d, c);
  BwArgs b;
  b.T = d->T; b.H = d->H; b.E = d->E; b.k = d->k; b.I = d->I; b.Is = d->Is;
  b.x = a->x; b.w_router = a->w_router; b.w_shared_gate = a->w_shared_gate;
  // The maps of an empty partition still need a valid address; nothing is read or written through them.
  b.w_gate_up = nl ? a->w_gate_up : a->ws_gate_up;
  b.w_down = nl ? a->w_down : a->ws_down;
  b.ws_gate_up = a->ws_gate_up; b.ws_down = a->ws_down;
  b.topk_ids = a->topk_ids; b.topk_w = a->topk_w; b.shared_sig = a->shared_sig;
  b.offsets = a->expert_offsets; b.sorted_route = a->sorted_route; b.route_pos = a->route_pos;
  b.y_routed = a->y_routed; b.y_shared = a->y_shared;
  b.gu_routed = a->saved.gu; b.gu_shared = a->saved.gu_shared; b.h_routed = a->saved.h; b.h_shared = a->saved.h_shared;
  b.dy = a->dy; b.dx = a->dx;
  b.dw_gate_up = nl ? a->dw_gate_up : a->dws_gate_up;
  b.dw_down = nl ? a->dw_down : a->dws_down;
  b.dw_router = a->dw_router;
  b.dw_shared_gate = a->dw_shared_gate; b.dws_gate_up = a->dws_gate_up; b.dws_down = a->dws_down;
  b.dyr = sc.dyr; b.dys = sc.dys; b.dgu_routed = sc.dgu_routed; b.dgu_shared = sc.dgu_shared;
  b.dxr = dxr ? dxr : sc.dxr;
  b.dxs = sc.dxs; b.x_sorted = sc.x_sorted;
  b.dlogit = a->dlogit ? a->dlogit : sc.dlogit;
  b.dz = a->dz ? a->dz : sc.dz;
  b.e_begin = eb;
  b.e_end = ee;
  b.yr_sorted = yr_sorted;
  return cuda_status(launch_backward(d->dtype, b, sc.inner, device_status_ptr(), s, phase));
}

MOE_API int moe_backward(const moe_dims_t *d, const moe_bwd_args_t *a, void *ws, size_t ws_bytes, void *stream) {
  if (!d) return MOE_ERR_INVALID_ARG;
  return backward_impl(d, a, 0, d->E, BWD_PHASE_ALL, 0, nullptr, ws, ws_bytes, stream);
}

MOE_API int moe_backward_ep(const moe_dims_t *d, int32_t e_begin, int32_t e_end, int32_t phase,
                            const moe_bwd_args_t *a, float *dxr_sorted, void *ws, size_t ws_bytes, void *stream) {
  if (!d || e_begin < 0 || e_end < e_begin || e_end > d->E || phase < 1 || phase > 3) return MOE_ERR_INVALID_ARG;
  if (!buf_ok(dxr_sorted, (int64_t)d->T * d->k * d->H)) return MOE_ERR_INVALID_ARG;
  return backward_impl(d, a, e_begin, e_end, phase, 1, dxr_sorted, ws, ws_bytes, stream);
}

MOE_API int moe_device_status(int reset, int32_t *detail) {
  int v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_moe_status, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  if (reset) {
    int zero = 0;
    if (cudaMemcpyToSymbol(g_moe_status, &zero, sizeof(int)) != cudaSuccess) return MOE_ERR_CUDA;
  }
  if (detail) *detail = v;
  return v == 0 ? MOE_OK : MOE_ERR_DEVICE;
}
