// Host-side launchers of the MoE kernels (internal; the public surface is
// include/moe.h).  Every launcher only enqueues work on `stream` and returns
// the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/moe.h"

namespace moe {

// ---- route.cu ----
// logits[t,e] = sum_h x[t,h] * wr[e,h] (+ bias[e]) with FP32 products summed
// sequentially over h (the MOE_F32 router; x is float).
cudaError_t launch_router_logits_simt(int T, int H, int E, const float *x, const float *wr, const float *bias,
                                      float *logits, cudaStream_t stream);
// Top-k, route weights and shared gate, one warp per token.
cudaError_t launch_topk_gate(int dtype, int T, int H, int E, int k, const float *logits, const void *x,
                             const void *w_shared_gate, int32_t *ids, float *w, float *sig,
                             cudaStream_t stream);

// Route weights and shared gate for given expert ids (router replay).
cudaError_t launch_replay_gate(int dtype, int T, int H, int E, int k, const float *logits, const void *x,
                               const void *w_shared_gate, const int32_t *ids, float *w, float *sig, int *status,
                               cudaStream_t stream);

// ---- api.cu ----
// Device address of the status word on the current device (nullptr on error).
int *device_status_ptr();
// Checks of moe_permute's dims and buffers, without the workspace (MOE_OK or
// the error status).
int permute_args_check(const moe_dims_t *d, const int32_t *topk_ids, const int32_t *expert_offsets,
                       const int32_t *sorted_route, const int32_t *route_pos);

// ---- permute.cu ----
// Routes per warp of the count and scatter kernels: 128 by default (more
// warps in flight), 512 where the scratch (ceil(R / chunk) * E + E ints) must
// stay small.  The result does not depend on the chunk.
constexpr int PERMUTE_CHUNK_SMALL = 128, PERMUTE_CHUNK_LARGE = 512;
size_t permute_scratch_bytes(int64_t R, int E, int chunk = PERMUTE_CHUNK_SMALL);
cudaError_t launch_permute(int64_t R, int E, const int32_t *ids, int32_t *offsets, int32_t *sorted_route,
                           int32_t *route_pos, void *scratch, int *status, cudaStream_t stream,
                           int chunk = PERMUTE_CHUNK_SMALL);
// Item tables of the two forward grouped GEMMs, written by the one-launch
// sort below when it is given them (the layout launch_ffn_tc reads).
struct PermuteItems {
  int T, nf_a_r, nf_a_s, nf_b_r, nf_b_s, max_a, max_b;
  int32_t *start_a, *start_b;
  int4 *items_a, *items_b;
};
// ---- permute_cluster.cu ----
// The same stable counting sort in one launch (a cluster of sixteen CTAs, no
// scratch) for R <= 2^20 routes and E <= 1024 on devices where that cluster
// fits; with `items`, also the grouped GEMMs' item tables of all E experts
// and the shared expert.
bool permute_cluster_ok(int64_t R, int E);
cudaError_t launch_permute_cluster(int64_t R, int E, const int32_t *ids, int32_t *offsets, int32_t *sorted_route,
                                   int32_t *route_pos, int *status, cudaStream_t stream,
                                   const PermuteItems *items = nullptr);
// tile_start[s] for s in [0, E+1]: prefix of ceil(n_s / bn) over the E routed
// segments (n_s from offsets) and the shared segment (n_E = T); only routed
// segments in [e_begin, e_end) (e_end < 0: E) and, if with_shared, the shared
// segment get tiles.
cudaError_t launch_build_tiles(int E, int T, int bn, const int32_t *offsets, int32_t *tile_start,
                               cudaStream_t stream, int e_begin = 0, int e_end = -1, int with_shared = 1);

// ---- ffn_simt.cu ----
struct FfnArgs {
  int T, H, E, k, I, Is;
  const void *x;
  const int32_t *offsets;
  const int32_t *sorted_route;
  const void *w_gate_up, *w_down, *ws_gate_up, *ws_down;
  void *y_routed, *y_shared;
  void *h_routed, *h_shared;    // intermediate h (required)
  void *gu_routed, *gu_shared;  // saved pre-activations (nullable)
  // Expert partition: only the routed segments in [e_begin, e_end) (weights
  // w_gate_up / w_down hold those experts only, expert e at index e - e_begin)
  // and, if with_shared, the shared expert; y_sorted: routed rows written in
  // sorted order (row j) instead of route order (row sorted_route[j]).
  int e_begin = 0, e_end = -1, with_shared = 1, y_sorted = 0;
  // bf16 path: y_routed / y_shared are float buffers receiving the FP32
  // accumulators unrounded (a partial sum over a slice of I, for the
  // expert-tensor-parallel reduction).
  int y_f32 = 0;
  // bf16 path: the item tables are already in the scratch (written by the
  // one-launch sort from ffn_tc_item_tables' description).
  int items_ready = 0;
};
size_t ffn_simt_scratch_bytes(int E);
// The MOE_F32 grouped FFN on CUDA cores (all buffers float).
cudaError_t launch_ffn_simt(const FfnArgs &a, void *scratch, cudaStream_t stream);

// ---- etp.cu ----
constexpr int ETP_MAX_PARTS = 16;
// out[i] = cast(((parts[0][i] + parts[1][i]) + ...) + parts[n-1][i]) for
// i < count (FP32 sums in part order, one rounding to `dtype`).
cudaError_t launch_etp_reduce(int dtype, int n, const float *const *parts, int64_t count, void *out,
                              cudaStream_t stream);

// ---- etp_fused.cu ----
// One ETP rank's 128-feature slice (I = Is = 128, bf16) with gate_up and down
// in one kernel, h kept in shared memory; FP32 partial rows like the y_f32
// path of launch_ffn_tc (scratch: etp_fused_scratch_bytes).
bool etp_fused_supported(int H, int I, int Is);
size_t etp_fused_scratch_bytes(int T, int k, int E);
cudaError_t launch_etp_fused(const FfnArgs &a, void *scratch, int *status, cudaStream_t stream);

// ---- gemm_tc.cu (bf16 tensor-core path) ----
size_t router_tc_scratch_bytes(int T, int E, int H);
bool router_split_k(int T, int E);
// Router logits via the exact three-way bf16 split of w_router (splits = 3), or
// with the weight rounded once to bf16 (splits = 1, the BF16-router ablation)
// (scratch: router_tc_scratch_bytes).
cudaError_t launch_router_logits_tc(int T, int H, int E, const void *x, const float *wr, const float *bias,
                                    float *logits, void *scratch, int *status, cudaStream_t stream, int splits = 3);
size_t ffn_tc_scratch_bytes(int T, int k, int E, int H, int I, int Is);
// gate_up + SwiGLU and down as two persistent tcgen05 grouped GEMMs (scratch: ffn_tc_scratch_bytes).
cudaError_t launch_ffn_tc(const FfnArgs &a, void *scratch, int *status, cudaStream_t stream);
// The item tables of launch_ffn_tc for `a` in `scratch`, for the one-launch
// sort to write (false where that sort cannot build them).
bool ffn_tc_item_tables(const FfnArgs &a, void *scratch, PermuteItems *it);
// Item tables of two grouped GEMMs over the same segments: per segment,
// ceil(n_s / tile) token tiles (tile = 256 rows unless given) times nf_*_r
// (routed) or nf_*_s (shared) M-tile pairs; items = int4 (segment, pair,
// first row, rows).
int64_t tc_max_items(int T, int k, int E, int nf_routed, int nf_shared);
cudaError_t launch_item_tables(int E, int T, int nf_a_r, int nf_a_s, int nf_b_r, int nf_b_s, const int32_t *offsets,
                               int32_t *start_a, int32_t *start_b, int4 *items_a, int4 *items_b, int max_a,
                               int max_b, cudaStream_t stream, int e_begin = 0, int e_end = -1, int with_shared = 1,
                               int tile = 256);

// ---- combine.cu ----
// route_pos != nullptr: y_routed rows are in sorted order (route r at row route_pos[r]).
cudaError_t launch_combine(int dtype, int T, int H, int k, const void *y_routed, const void *y_shared,
                           const float *w, const float *sig, void *y, cudaStream_t stream,
                           const int32_t *route_pos = nullptr);

// ---- backward.cu ----
struct BwArgs {
  int T, H, E, k, I, Is;
  // forward inputs and results
  const void *x;
  const float *w_router;
  const void *w_shared_gate, *w_gate_up, *w_down, *ws_gate_up, *ws_down;
  const int32_t *topk_ids;
  const float *topk_w, *shared_sig;
  const int32_t *offsets, *sorted_route, *route_pos;
  const void *y_routed, *y_shared;
  const void *gu_routed, *gu_shared, *h_routed, *h_shared;
  const void *dy;
  // outputs
  void *dx;
  float *dw_gate_up, *dw_down, *dw_router, *dw_shared_gate, *dws_gate_up, *dws_down;
  // intermediates (workspace)
  void *dyr;                    // [T*k, H] dtype, sorted order: w * dy of the route
  void *dys;                    // [T, H] dtype: sig * dy
  void *dgu_routed;             // [T*k, 2I] dtype, sorted order: [dg | du]
  void *dgu_shared;             // [T, 2Is] dtype
  float *dxr;                   // [T*k, H] sorted order: input grad of each route
  float *dxs;                   // [T, H]: input grad through the shared expert
  void *x_sorted;               // [T*k, H] dtype, sorted order: x of the route's token (tensor-core path)
  float *dlogit;                // [T, k]
  float *dz;                    // [T]
  // Expert partition: only experts [e_begin, e_end) run their dgrad and
  // wgrad; w_gate_up, w_down, dw_gate_up, dw_down hold those experts only
  // (expert e at index e - e_begin).  e_end < 0 means E.
  int e_begin = 0, e_end = -1;
  int yr_sorted = 0;            // y_routed rows in sorted order (route r at row route_pos[r])
};
size_t backward_scratch_bytes(int dtype, int T, int k, int E, int H, int I, int Is);
// The backward (dtype 0 = float, 1 = bf16): the four expert GEMMs on the
// tensor cores for bf16 when backward_tc_supported, else on CUDA cores.
// phase bit 1: everything up to the routed input gradients dxr (own experts'
// rows only) and the weight gradients; bit 2: dx from all dxr rows.
enum { BWD_PHASE_EXPERTS = 1, BWD_PHASE_DX = 2, BWD_PHASE_ALL = 3 };
cudaError_t launch_backward(int dtype, const BwArgs &a, void *scratch, int *status, cudaStream_t stream,
                            int phase = BWD_PHASE_ALL);

// ---- grad_tc.cu (bf16 tensor-core backward GEMMs) ----
bool backward_tc_supported(int H, int I, int Is);
size_t dgrad_tc_scratch_bytes(int T, int k, int E, int H, int I, int Is);
// dGU = SwiGLU-backward(dYr Wdn) and dXr = dGU Wgu (and the shared expert's) (scratch: dgrad_tc_scratch_bytes).
cudaError_t launch_dgrad_tc(const BwArgs &a, void *scratch, int *status, cudaStream_t stream);
// dWdn, dWgu and the shared expert's weight gradients.
cudaError_t launch_wgrad_tc(const BwArgs &a, int *status, cudaStream_t stream);

}  // namespace moe
