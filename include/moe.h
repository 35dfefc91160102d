/*
 * moe.h -- C ABI of the batch-invariant MoE layer for NVIDIA GB300 (sm_103a).
 *
 * One Mixture-of-Experts layer: E routed SwiGLU experts with top-k routing
 * plus one sigmoid-gated shared SwiGLU expert (SkyRL PR #2513, section
 * "What": 512 routed experts, top-10, and a shared expert).  The forward and
 * backward are deterministic and batch-invariant: a token's output row and
 * input-gradient row do not depend on the other tokens in the batch, on the
 * batch size or on the token's position (RL-Kernel PR #557 "EP4 distributed
 * logprob parity", section "Prior art & reuse decision": batch-invariant
 * forward and backward; embedded #503 commit message "MoE route/combine
 * contract with a batch-invariant grouped expert GEMM").
 *
 * The layer splits into separate contracts, as the #503 commit message does
 * (bullets "Routing", "Experts", "Combine", "Backward"):
 *
 *   moe_route        router GEMM (FP32 result), softmax, top-k, renormalise,
 *                    shared-expert gate
 *   moe_permute      stable counting sort of the routes by expert
 *   moe_grouped_ffn  per-expert SwiGLU over the expert segments, unweighted
 *                    rows; the shared expert as one more segment
 *   moe_combine      ordered FP32 sum of the k weighted rows, plus the gated
 *                    shared row, one rounding to the output type
 *   moe_backward     all gradients, reduced in fixed orders
 *   moe_backward_ep  one rank's part of moe_backward under an expert partition
 *   moe_grouped_ffn_etp, moe_etp_reduce  the grouped FFN with I split across ranks
 *   moe_grouped_ffn_etp_fused  one rank's slice with gate_up and down fused (h on chip)
 *   moe_forward      the four forward calls in sequence, intermediates in the
 *                    caller's workspace
 *
 * Conventions that hold for every entry point:
 *  - Pointers named as device buffers are CUDA device (or managed) memory of
 *    the current device; they must be 16-byte aligned.  Matrices are dense
 *    row-major with the last dimension contiguous.  The caller owns every
 *    buffer, including the workspace; the library allocates no device memory
 *    and keeps no state between calls apart from per-device kernel
 *    attributes set on first use and one device-side status word.
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *    call is stream-ordered and asynchronous: it never synchronises and never
 *    reads device data on the host.
 *  - Return value: MOE_OK (0) or a negative moe_status.  On a host-detected
 *    error (bad argument, unsupported shape, small workspace) nothing is
 *    launched and no output is written.  There is no fallback path.
 *  - T = 0 is valid: the call succeeds and writes only the fixed-size
 *    outputs (offsets, weight gradients), which become zero.
 *  - Element type: `dtype` selects float (MOE_F32) or bfloat16 (MOE_BF16,
 *    stored as uint16 bit patterns) for x, the expert weights, the shared
 *    gate weight, the expert rows and the outputs y and dx.  The router
 *    weight, router bias, routing weights and gate values are always float.
 *    Every weight gradient is float and is overwritten, not accumulated.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 };

enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1, /* NULL pointer, negative or zero size, k > E, k > 16, misaligned pointer */
  MOE_ERR_UNSUPPORTED = -2, /* a shape or dtype the kernels do not cover (see moe_dims_t) */
  MOE_ERR_WORKSPACE = -3,   /* ws_bytes smaller than moe_workspace_size() */
  MOE_ERR_CUDA = -4,        /* a CUDA runtime call or kernel launch failed */
  MOE_ERR_DEVICE = -5       /* (moe_device_status only) a kernel recorded a failed check */
};

/* Operation selector of moe_workspace_size. */
enum moe_op {
  MOE_OP_ROUTE = 0,
  MOE_OP_PERMUTE = 1,
  MOE_OP_GROUPED_FFN = 2,
  MOE_OP_COMBINE = 3,
  MOE_OP_BACKWARD = 4,
  MOE_OP_FORWARD = 5
};

/*
 * Layer shape.  Limits: T >= 0, T*k < 2^31; 1 <= k <= 16; k <= E <= 1024.
 * MOE_F32: H, I, Is multiples of 4.
 * MOE_BF16: H a multiple of 256, I and Is multiples of 128.
 * Other shapes return MOE_ERR_UNSUPPORTED.
 */
typedef struct moe_dims {
  int32_t T;     /* tokens in this batch */
  int32_t H;     /* hidden size */
  int32_t E;     /* routed experts */
  int32_t k;     /* experts per token */
  int32_t I;     /* routed-expert intermediate size */
  int32_t Is;    /* shared-expert intermediate size */
  int32_t dtype; /* enum moe_dtype */
} moe_dims_t;

/*
 * Activations kept by the forward for the backward.  Each pointer may be
 * NULL (inference); moe_backward needs all four.  Sorted order means the
 * expert-segment order produced by moe_permute (row j holds route
 * sorted_route[j]).
 */
typedef struct moe_saved {
  void *gu;        /* [T*k, 2I] dtype, sorted order: gate pre-activation (I) then up (I) */
  void *h;         /* [T*k, I]  dtype, sorted order: silu(gate) * up, input of the down projection */
  void *gu_shared; /* [T, 2Is]  dtype, token order */
  void *h_shared;  /* [T, Is]   dtype, token order */
} moe_saved_t;

/* Bytes of workspace the operation needs for these dims (0 for an invalid
 * dims pointer).  The workspace must be 256-byte aligned device memory. */
size_t moe_workspace_size(const moe_dims_t *d, int op);

/* Static description of a status code. */
const char *moe_status_string(int status);

/*
 * moe_route -- router and shared-expert gate.
 * RL-Kernel PR #557, #503 commit message "Routing": FP32 router GEMM
 * through a batch-invariant GEMM, fixed-order softmax, stable descending
 * top-k with ties to the lower expert id, FP32 renormalisation of the k
 * selected weights.  Shared gate: #503 "TP4 block", a replicated
 * shared-expert gate, here sigmoid(x . w_shared_gate).
 *
 *   x              [T, H]  dtype   input rows
 *   w_router       [E, H]  float   router weight (nn.Linear layout)
 *   router_bias    [E]     float   added to the logits, or NULL
 *   w_shared_gate  [H]     dtype   shared-expert gate weight
 *   topk_ids       [T, k]  int32   out: expert ids, slot order = descending logit
 *   topk_w         [T, k]  float   out: softmax over the k selected logits
 *   shared_sig     [T]     float   out: sigmoid gate of the shared expert
 *   logits         [T, E]  float   out: router logits (with bias), or NULL
 *
 * The logits are FP32 results of an exact bf16 three-way split of the FP32
 * router weight (MOE_BF16) or FP32 products (MOE_F32), summed in a fixed
 * order that does not depend on T.  Workspace: moe_workspace_size(ROUTE).
 */
int moe_route(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
              const void *w_shared_gate, int32_t *topk_ids, float *topk_w, float *shared_sig,
              float *logits, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_router_logits -- the router GEMM alone, for measuring it.
 * RL-Kernel PR #557, #503 commit message "Routing": the router runs in FP32;
 * "Results (4 x H100)": BF16 routing is the variant that drifts.
 *   exact = 1: the logits moe_route uses (bit for bit).
 *   exact = 0: the BF16-router ablation: the weight rounded once to bf16, the
 *              same FP32 accumulation order otherwise (MOE_BF16 only;
 *              MOE_F32 returns MOE_ERR_UNSUPPORTED).
 *   logits [T, E] float out (with router_bias if not NULL).  Workspace: ROUTE.
 */
int moe_router_logits(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
                      int32_t exact, float *logits, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_route_replay -- route weights and shared gate for GIVEN expert ids.
 * SkyRL PR #2513, section "chunked_mlp fixes (#2532, merged)": per-chunk
 * router replay; SkyRL docs page "Qwen3.8-Flash-Next", section "Example
 * scripts": rollout routing replay.  A training pass reuses the expert
 * choices of an earlier (rollout) pass instead of selecting its own; the
 * router logits are recomputed so that the weights carry their gradient.
 *
 *   topk_ids       [T, k]  int32   in: the replayed expert ids, slot order as given
 *   topk_w         [T, k]  float   out: w_s = exp(l_s - m) / sum_j exp(l_j - m) over
 *                                  the given slots, m = the largest of the k logits
 *   (x, w_router, router_bias, w_shared_gate, shared_sig, logits as moe_route)
 *
 * With the ids moe_route chose, topk_w and shared_sig equal moe_route's bit
 * for bit.  Ids outside [0, E) or repeated within a token fail closed: that
 * token's weights are written as zeros and the device status word records
 * code 1 (out of range) or 4 (repeated); check moe_device_status.
 * moe_backward accepts replayed routes unchanged.  Workspace: ROUTE.
 */
int moe_route_replay(const moe_dims_t *d, const void *x, const float *w_router, const float *router_bias,
                     const void *w_shared_gate, const int32_t *topk_ids, float *topk_w, float *shared_sig,
                     float *logits, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_permute -- dispatch as a stable counting sort of the routes.
 * RL-Kernel PR #557 "What": dispatch is a local selection of the routes;
 * #503 "Experts": one writer per (token, route) row.  Route r = t*k + s.
 *
 *   topk_ids        [T, k]  int32  expert ids from moe_route
 *   expert_offsets  [E+1]   int32  out: first sorted row of each expert; [E] = T*k
 *   sorted_route    [T*k]   int32  out: route of sorted row j, in (expert, t, s) order
 *   route_pos       [T*k]   int32  out: sorted row of route r (inverse of sorted_route)
 *
 * Integer only, no atomics on positions; the result equals a sequential
 * counting sort bit for bit.  An id outside [0, E) is skipped and recorded in
 * the device status word (moe_device_status).  Workspace: PERMUTE.  Up to
 * 2^20 routes, on devices that run clusters of sixteen CTAs, the sort is one
 * launch that leaves the workspace untouched; otherwise it runs as four
 * kernels over the workspace.  Both forms give the same result.
 */
int moe_permute(const moe_dims_t *d, const int32_t *topk_ids, int32_t *expert_offsets,
                int32_t *sorted_route, int32_t *route_pos, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_permute_noalloc -- moe_permute without a workspace argument.
 * The paper has no counterpart: this is a convenience of this library.
 *
 * For callers that cannot allocate device memory: a custom operator or
 * plugin hosted by another runtime that owns the device memory pool and
 * hands out only input and output buffers, or a latency-critical loop that
 * must not call cudaMalloc because it can synchronise the device.  The
 * arguments, their checks and the results are those of moe_permute
 * (bit-identical outputs).  Up to 2^20 routes, where the device runs the
 * one-launch cluster sort, no scratch is used at all; above that the
 * four-kernel sort keeps its scratch in a fixed array of
 * MOE_PERMUTE_NOALLOC_SCRATCH_BYTES in the library's own device memory,
 * held by every GPU that loads the library until the process exits.  No
 * cudaMalloc, cudaFree or other allocating routine is called.
 *
 * Limit (four-kernel sort): the scratch needs (ceil(T*k / 128) * E + E) * 4
 * bytes, or (ceil(T*k / 512) * E + E) * 4 bytes with the larger chunks it
 * takes when the first does not fit; larger sizes return
 * MOE_ERR_UNSUPPORTED before any GPU work (E = 64: up to 8,388,096 routes;
 * E = 512: every size above 2^20 routes is refused).
 * The first call on a device that needs the array looks up its device
 * address (cudaGetSymbolAddress) with that device current; make that first
 * call before any stream capture.  Every call uses the same array: calls that
 * can overlap on the GPU (different streams, no ordering between them) race
 * and must be serialised by the caller.  Each call writes every scratch word
 * it reads, so nothing is carried over from the previous call.
 */
#define MOE_PERMUTE_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)
int moe_permute_noalloc(const moe_dims_t *d, const int32_t *topk_ids, int32_t *expert_offsets,
                        int32_t *sorted_route, int32_t *route_pos, void *stream);

/*
 * moe_grouped_ffn -- per-expert SwiGLU FFN over the expert segments.
 * #503 commit message "Experts": per-route gate_up and down projections
 * through one fixed-configuration grouped GEMM, no routed-weight multiply
 * and no sum inside the kernel, one writer per row.  The shared expert
 * (PR #557 "What") runs as one more segment covering all T tokens.
 *
 *   x               [T, H]      dtype  input rows
 *   expert_offsets  [E+1]       int32  from moe_permute
 *   sorted_route    [T*k]       int32  from moe_permute
 *   w_gate_up       [E, 2I, H]  dtype  per expert: I gate rows, then I up rows
 *   w_down          [E, H, I]   dtype
 *   ws_gate_up      [2Is, H]    dtype  shared expert, same layout
 *   ws_down         [H, Is]     dtype
 *   y_routed        [T*k, H]    dtype  out: row t*k+s = expert topk_ids[t,s] applied to x_t, unweighted
 *   y_shared        [T, H]      dtype  out: shared expert applied to x_t
 *   saved           may be NULL; non-NULL members are written (moe_saved_t)
 *
 * Accumulation in FP32 with a fixed K order; gate/up and h are rounded once
 * to dtype (h is the down projection's input), rows once to dtype.
 * Workspace: GROUPED_FFN.
 */
int moe_grouped_ffn(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                    const int32_t *sorted_route, const void *w_gate_up, const void *w_down,
                    const void *ws_gate_up, const void *ws_down, void *y_routed, void *y_shared,
                    const moe_saved_t *saved, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_combine -- combine_routes.
 * #503 commit message "Combine": k ordered FP32 multiply-adds and one cast
 * to the output type, no atomics.  The shared term is added after the k
 * routed terms in the same FP32 accumulator:
 *   y[t] = cast( fma(sig[t], Ys[t], fma(w[t,k-1], Yr[t*k+k-1], ... fma(w[t,0], Yr[t*k], 0))) )
 *
 *   y_routed [T*k, H] dtype, y_shared [T, H] dtype, topk_w [T, k] float,
 *   shared_sig [T] float, y [T, H] dtype out.  No workspace.
 */
int moe_combine(const moe_dims_t *d, const void *y_routed, const void *y_shared, const float *topk_w,
                const float *shared_sig, void *y, void *stream);

/*
 * moe_grouped_ffn_ep -- moe_grouped_ffn for one rank of an expert partition.
 * RL-Kernel PR #557 "What": experts are split into contiguous ranges across
 * ranks, every rank computes the same routes and runs only the segments of
 * its own experts, one all_gather of the routed rows (a byte copy) follows,
 * and the combine is local (moe_combine_sorted).  This call is one rank's
 * expert part; the exchange belongs to the caller (on one GPU, several calls
 * with disjoint ranges write disjoint row blocks of one buffer).
 *
 *   e_begin, e_end  the rank's experts [e_begin, e_end), 0 <= e_begin <= e_end <= E
 *   with_shared     1: also compute the shared expert into y_shared; 0: leave it
 *   w_gate_up [e_end-e_begin, 2I, H], w_down [e_end-e_begin, H, I]: the rank's
 *                   experts only (expert e at index e - e_begin); NULL if the
 *                   range is empty.  ws_gate_up / ws_down: NULL if !with_shared.
 *   y_sorted [T*k, H] dtype  out: routed rows in SORTED order (row j = route
 *                   sorted_route[j]); only rows expert_offsets[e_begin] ..
 *                   expert_offsets[e_end] - 1 are written, so each rank's
 *                   result is one contiguous block.
 * Every value equals the single-call moe_grouped_ffn's for the same row bit for
 * bit.  Errors as moe_grouped_ffn; a bad range is MOE_ERR_INVALID_ARG.
 * Workspace: GROUPED_FFN.
 */
int moe_grouped_ffn_ep(const moe_dims_t *d, int32_t e_begin, int32_t e_end, int32_t with_shared, const void *x,
                       const int32_t *expert_offsets, const int32_t *sorted_route, const void *w_gate_up,
                       const void *w_down, const void *ws_gate_up, const void *ws_down, void *y_sorted,
                       void *y_shared, const moe_saved_t *saved, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_combine_sorted -- moe_combine reading the routed rows in sorted order
 * (route r at row route_pos[r]), the layout moe_grouped_ffn_ep writes.  Same
 * arithmetic and order as moe_combine, so the same output bits.  No workspace.
 */
int moe_combine_sorted(const moe_dims_t *d, const void *y_sorted, const int32_t *route_pos, const void *y_shared,
                       const float *topk_w, const float *shared_sig, void *y, void *stream);

/*
 * moe_grouped_ffn_etp -- moe_grouped_ffn for one rank of an expert-tensor-
 * parallel (ETP) split of the intermediate dimension.  RL-Kernel PR #557
 * "What", bullet "Fail closed" (EP 1 runs the experts expert-tensor-parallel
 * over 4 ranks) and the embedded #503 commit message, bullet "TP4 block"
 * (every expert on every rank, partial results reduced across ranks); the
 * reduction here is a byte-copy gather plus a fixed-order local sum, as PR
 * #557 "What" does for the EP exchange: rank r holds, for every expert, the gate and up rows of its
 * feature slice [i0, i1) of I and the matching columns of W_down (and a
 * slice of the shared expert's Is).  Since Yr = sum over features i of
 * h_i W_down[:, i], its down projection is a partial sum of every routed and
 * shared row.
 *
 *   d               the layer's dims with I and Is replaced by the rank's
 *                   slice widths (bf16: multiples of 128)
 *   w_gate_up [E, 2 I_r, H]: rows 0..I_r-1 = gate rows i0..i1-1, then the up
 *                   rows i0..i1-1; w_down [E, H, I_r] = W_down[:, :, i0:i1];
 *                   ws_gate_up / ws_down the same for the shared expert
 *   yr_partial [T*k, H] float, route order; ys_partial [T, H] float: this
 *                   rank's partial sums, the FP32 accumulators unrounded
 *   saved           as moe_grouped_ffn, with the slice's widths
 * Errors as moe_grouped_ffn.  Workspace: GROUPED_FFN for `d`.
 */
int moe_grouped_ffn_etp(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                        const int32_t *sorted_route, const void *w_gate_up, const void *w_down, const void *ws_gate_up,
                        const void *ws_down, float *yr_partial, float *ys_partial, const moe_saved_t *saved, void *ws,
                        size_t ws_bytes, void *stream);

/*
 * moe_grouped_ffn_etp_fused -- moe_grouped_ffn_etp for a 128-feature slice
 * with the two projections fused: the intermediate h of a tile of rows stays
 * in shared memory between the gate_up and the down GEMM instead of going
 * through device memory.  Same passages as moe_grouped_ffn_etp (#503 commit
 * message, bullet "TP4 block": every expert on every rank; "Experts":
 * per-route gate_up and down projections).
 * The partial rows equal moe_grouped_ffn_etp's bit for bit (the same
 * roundings, every output one MMA chain over K in the same order).
 *
 *   d               as moe_grouped_ffn_etp; bf16 only, with I = Is = 128 (one
 *                   rank's slice, e.g. I = 512 over four ranks) and H a
 *                   multiple of 128; other shapes return MOE_ERR_UNSUPPORTED
 *   x, expert_offsets, sorted_route, the weight slices, yr_partial,
 *   ys_partial      as moe_grouped_ffn_etp (no saved activations: h is never
 *                   written out, so a training step saves it with
 *                   moe_grouped_ffn_etp instead)
 *   ws              at least moe_workspace_size(d, MOE_OP_GROUPED_FFN) bytes
 * Errors: MOE_ERR_INVALID_ARG for a NULL or misaligned buffer,
 * MOE_ERR_WORKSPACE for a short workspace; nothing is launched then.
 */
int moe_grouped_ffn_etp_fused(const moe_dims_t *d, const void *x, const int32_t *expert_offsets,
                              const int32_t *sorted_route, const void *w_gate_up, const void *w_down,
                              const void *ws_gate_up, const void *ws_down, float *yr_partial, float *ys_partial,
                              void *ws, size_t ws_bytes, void *stream);

/*
 * moe_etp_reduce -- the routed and shared rows from the ranks' partial sums:
 * y_routed = dtype(((p_0 + p_1) + ...) + p_{n-1}), summed in FP32 in rank
 * order with one rounding (same for y_shared), after every rank gathered all
 * partials (a byte copy).  The result depends on the number of ranks (the
 * rounding order does) but not on T, on the exchange, or on which rank
 * reduces; with one rank it equals moe_grouped_ffn's rows bit for bit.
 *
 *   d               the layer's dims (full I, Is)
 *   n_parts         1..16
 *   yr_parts, ys_parts  HOST arrays of n_parts device pointers to the float
 *                   partials ([T*k, H] and [T, H]), in rank order
 *   y_routed [T*k, H], y_shared [T, H] dtype out (feed moe_combine)
 * No workspace.
 */
int moe_etp_reduce(const moe_dims_t *d, int32_t n_parts, const float *const *yr_parts, const float *const *ys_parts,
                   void *y_routed, void *y_shared, void *stream);

/* Everything moe_forward reads and writes. */
typedef struct moe_fwd_args {
  const void *x;             /* [T, H] dtype */
  const float *w_router;     /* [E, H] float */
  const float *router_bias;  /* [E] float or NULL */
  const void *w_shared_gate; /* [H] dtype */
  const void *w_gate_up;     /* [E, 2I, H] dtype */
  const void *w_down;        /* [E, H, I] dtype */
  const void *ws_gate_up;    /* [2Is, H] dtype */
  const void *ws_down;       /* [H, Is] dtype */
  void *y;                   /* out [T, H] dtype */
  /* Optional outputs (NULL: kept in the workspace).  The backward needs
   * all of them, plus every member of `saved`. */
  int32_t *topk_ids;       /* [T, k] */
  float *topk_w;           /* [T, k] */
  float *shared_sig;       /* [T] */
  float *logits;           /* [T, E] (never kept in the workspace) */
  int32_t *expert_offsets; /* [E+1] */
  int32_t *sorted_route;   /* [T*k] */
  int32_t *route_pos;      /* [T*k] */
  void *y_routed;          /* [T*k, H] dtype */
  void *y_shared;          /* [T, H] dtype */
  moe_saved_t saved;
  /* Router replay: if not NULL, these [T, k] ids are the routes (see
   * moe_route_replay) instead of the top-k selection; topk_ids, if given,
   * receives a copy. */
  const int32_t *replay_ids;
} moe_fwd_args_t;

/* moe_forward -- moe_route, moe_permute, moe_grouped_ffn, moe_combine on one
 * stream.  Workspace: FORWARD (covers every optional output left NULL).
 * Same results as the four calls, bit for bit; where the permute runs as one
 * launch (see moe_permute) and dtype is MOE_BF16, that launch also writes
 * the grouped FFN's work lists.  There, above 2048 tokens, the shared
 * expert's GEMMs (they need no routes) run on a second stream of the library
 * (one per device, non-blocking) that starts from an event recorded on
 * `stream` (after the router launch while the routed GEMMs average fewer
 * than 256 routes per expert, at the call otherwise) and is joined back into
 * `stream` before the combine: work on `stream` after the call sees every
 * output, as with one stream.
 * Under CUDA graph capture of `stream` the second stream joins the capture
 * through those events; two threads capturing or running moe_forward on one
 * device at once share that stream (correct, but serialised there). */
int moe_forward(const moe_dims_t *d, const moe_fwd_args_t *a, void *ws, size_t ws_bytes, void *stream);

/* Everything moe_backward reads and writes. */
typedef struct moe_bwd_args {
  /* forward inputs */
  const void *x;
  const float *w_router;
  const void *w_shared_gate;
  const void *w_gate_up;
  const void *w_down;
  const void *ws_gate_up;
  const void *ws_down;
  /* forward results (see moe_fwd_args_t) */
  const int32_t *topk_ids;
  const float *topk_w;
  const float *shared_sig;
  const int32_t *expert_offsets;
  const int32_t *sorted_route;
  const int32_t *route_pos;
  const void *y_routed;
  const void *y_shared;
  moe_saved_t saved;
  /* upstream gradient */
  const void *dy; /* [T, H] dtype */
  /* outputs, all overwritten */
  void *dx;              /* [T, H] dtype */
  float *dw_gate_up;     /* [E, 2I, H] */
  float *dw_down;        /* [E, H, I] */
  float *dw_router;      /* [E, H] */
  float *dw_shared_gate; /* [H] */
  float *dws_gate_up;    /* [2Is, H] */
  float *dws_down;       /* [H, Is] */
  /* optional outputs (NULL: kept in the workspace) */
  float *dlogit; /* [T, k] gradient of the k selected router logits, slot order */
  float *dz;     /* [T] gradient of the shared-gate pre-activation x . w_shared_gate */
} moe_bwd_args_t;

/*
 * moe_backward -- gradients of L = sum(dy * y) with the routes held fixed.
 * #503 commit message "Backward": per-expert GEMMs write the per-route
 * input gradients into one dense buffer; dx sums them in ascending expert
 * order (PR #557 "What").  The route-weight gradient dw[t,s] = dy_t . Yr
 * is reduced per (t, s) over H in a fixed tree, so the backward stays batch
 * invariant (PR #557, "Results (4 x H100)", footnote 1: a torch.sum over
 * hidden there was not batch invariant).
 *   dx = sum over routes in ascending expert id of the routed input grads
 *        + shared-expert input grad + dlogit . W_router + dz * w_shared_gate,
 *   accumulated in FP32 in that order and cast once.  Weight gradients sum
 *   over their rows in ascending (expert-segment) order in FP32, with no
 *   split-K atomics.  Workspace: BACKWARD.
 * Inputs are the forward's own results for the same x and weights (the
 * routes are not recomputed); `saved` must hold all four activations.
 * Weight gradients are float whatever the dtype; with T = 0 they are
 * zero-filled.  Errors: MOE_ERR_INVALID_ARG for a NULL or misaligned buffer,
 * MOE_ERR_WORKSPACE for a short workspace; nothing is launched then.
 */
int moe_backward(const moe_dims_t *d, const moe_bwd_args_t *a, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_backward_ep -- moe_backward for one rank of an expert partition, in two
 * phases around the exchange of the routed input gradients.  RL-Kernel PR
 * #557 "What" (experts split into contiguous ranges, one all_gather of the
 * rows, the reductions local and in ascending expert order) and #503 commit
 * message "Backward" (per-expert GEMMs write per-route input gradients into
 * one dense buffer, which dx sums).
 *
 *   phase 1  the combine backward (route-weight and gate gradients), the
 *            shared expert's gradients, the router and gate weight gradients
 *            (all replicated: every rank computes them in full), and for the
 *            rank's experts [e_begin, e_end) their weight gradients and the
 *            routed input gradients of their rows;
 *   phase 2  dx, from all rows of dxr_sorted;
 *   phase 3  both (with a single rank, [0, E), this is moe_backward).
 * Between phase 1 and phase 2 the caller exchanges the row blocks of
 * dxr_sorted (a byte copy); phase 2 must get the same d, a, workspace and
 * range as phase 1 (the workspace carries the shared expert's input gradient
 * and, when a->dlogit / a->dz are NULL, those gradients, from one to the
 * other).
 *
 *   a->y_routed     [T*k, H] dtype in SORTED order (route r at row route_pos[r]),
 *                   the layout of moe_grouped_ffn_ep after the row exchange
 *   a->saved.gu, a->saved.h  sorted order as moe_grouped_ffn writes them; only
 *                   the rows of the rank's experts are read
 *   a->w_gate_up, a->w_down, a->dw_gate_up, a->dw_down  the rank's experts
 *                   only (expert e at index e - e_begin); NULL if the range is
 *                   empty
 *   dxr_sorted      [T*k, H] float, sorted order: phase 1 writes rows
 *                   expert_offsets[e_begin] .. expert_offsets[e_end] - 1 (one
 *                   contiguous block per rank); phase 2 reads every row
 * Every value equals the single-call moe_backward's bit for bit: the same
 * kernels with the same reduction orders run on the same rows.  Errors as
 * moe_backward; a bad range or phase is MOE_ERR_INVALID_ARG.  Workspace:
 * BACKWARD.
 */
int moe_backward_ep(const moe_dims_t *d, int32_t e_begin, int32_t e_end, int32_t phase, const moe_bwd_args_t *a,
                    float *dxr_sorted, void *ws, size_t ws_bytes, void *stream);

/*
 * moe_device_status -- read (and, if `reset`, clear) the device status word
 * of the current device.  Synchronises the device.  Returns MOE_OK when no
 * kernel recorded a failed check since the last reset, MOE_ERR_DEVICE when
 * one did (`*detail`, if not NULL, receives the first recorded code), or
 * MOE_ERR_CUDA.  Codes: 1 = expert id out of range in moe_permute or
 * moe_route_replay, 4 = expert id repeated within a token in moe_route_replay,
 * 2 = a pipeline wait in a tensor-core kernel timed out,
 * 3 = tensor-memory allocation failed.
 */
int moe_device_status(int reset, int32_t *detail);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
