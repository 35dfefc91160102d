/*
 * moe_oracle.c -- FP64 reference of the batch-invariant MoE layer.
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke
 * check of the package entry module and the CPU-baseline leg of the
 * benchmark may load this library.  It shares no code, header, table or
 * helper with the CUDA path and must never be called by it.
 *
 * What it computes is the plain definition of the layer, in double
 * precision, with plain loops and no blocking or fusion:
 *
 *   logits  l[t,e] = sum_h x[t,h] * Wr[e,h]  (+ bias[e])
 *   ids     the k experts with the largest logits, ties to the lower id,
 *           slot order = descending logit
 *   weights w[t,s] = softmax over the k selected logits (equal to the full
 *           softmax over all experts followed by renormalisation)
 *   expert  Y_e(x) = Wdn[e] (silu(Wg[e] x) * (Wu[e] x))     (SwiGLU FFN)
 *   gate    sig[t] = 1 / (1 + exp(-(x_t . w_sg)))
 *   output  y[t] = sum_s w[t,s] Y_{ids[t,s]}(x_t) + sig[t] Y_shared(x_t)
 *
 * Sources (page title, section):
 *  - RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503
 *    commit message "MoE route/combine contract with a batch-invariant
 *    grouped expert GEMM", bullets Routing, Experts, Combine, Backward.
 *  - RL-Kernel PR #557, section "What" (dispatch is a local selection,
 *    combine_routes in FP32 route order, dx summed in ascending expert order).
 *  - SkyRL PR #2513, section "What" (512 routed experts, top-10, shared expert).
 *
 * Every floating-point input is passed as double: bf16 and fp32 values
 * widen to double exactly, so the oracle reads the same stored numbers the
 * GPU reads.  Build with -ffp-contract=off so results are identical on
 * x86-64 and AArch64.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define IDX2(a, b, nb) ((int64_t)(a) * (int64_t)(nb) + (int64_t)(b))

static double silu(double g) { return g / (1.0 + exp(-g)); }
static double sigmoid(double z) { return 1.0 / (1.0 + exp(-z)); }

/* d/dg silu(g) = s (1 + g (1 - s)), s = sigmoid(g) */
static double silu_grad(double g) {
  double s = sigmoid(g);
  return s * (1.0 + g * (1.0 - s));
}

/* ------------------------------------------------------------------ */
/* Router GEMM.  #503 commit message, "Routing": FP32 router logits.   */
/* Here in FP64: l[t,e] = sum_h x[t,h] Wr[e,h] (+ bias[e]).            */
/* ------------------------------------------------------------------ */
void oracle_router_logits(int64_t T, int64_t H, int64_t E, const double *x,
                          const double *wr, const double *bias,
                          double *logits) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t t = 0; t < T; ++t) {
    const double *xt = x + IDX2(t, 0, H);
    for (int64_t e = 0; e < E; ++e) {
      const double *we = wr + IDX2(e, 0, H);
      double acc = 0.0;
      for (int64_t h = 0; h < H; ++h) acc += xt[h] * we[h];
      if (bias) acc += bias[e];
      logits[IDX2(t, e, E)] = acc;
    }
  }
}

/* ------------------------------------------------------------------ */
/* Top-k selection.  #503 commit message, "Routing": stable descending  */
/* argsort, ties go to the lower expert id.  Repeated arg-max with a    */
/* strict ">" over ascending ids gives exactly that order.  Returns the */
/* number of tokens whose row held a NaN (they select the lowest ids).  */
/* ------------------------------------------------------------------ */
int64_t oracle_topk_select(int64_t T, int64_t E, int64_t k,
                           const double *logits, int32_t *ids) {
  int64_t n_nan = 0;
#pragma omp parallel for schedule(static) reduction(+ : n_nan)
  for (int64_t t = 0; t < T; ++t) {
    const double *l = logits + IDX2(t, 0, E);
    char *taken = (char *)calloc((size_t)E, 1);
    int has_nan = 0;
    for (int64_t s = 0; s < k; ++s) {
      int64_t best = -1;
      for (int64_t e = 0; e < E; ++e) {
        if (taken[e]) continue;
        if (l[e] != l[e]) { has_nan = 1; continue; }
        if (best < 0 || l[e] > l[best]) best = e;
      }
      if (best < 0) { /* only NaNs left: lowest untaken id */
        for (int64_t e = 0; e < E; ++e)
          if (!taken[e]) { best = e; break; }
      }
      taken[best] = 1;
      ids[IDX2(t, s, k)] = (int32_t)best;
    }
    n_nan += has_nan;
    free(taken);
  }
  return n_nan;
}

/* ------------------------------------------------------------------ */
/* Route weights.  #503 commit message, "Routing": softmax over all     */
/* experts then renormalisation of the selected ones.  The full         */
/* denominator cancels, so w_s = exp(l_s - m) / sum_j exp(l_j - m) over */
/* the selected set, m = the largest selected logit.                    */
/* ------------------------------------------------------------------ */
void oracle_topk_weights(int64_t T, int64_t E, int64_t k,
                         const double *logits, const int32_t *ids,
                         double *w) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double *l = logits + IDX2(t, 0, E);
    const int32_t *id = ids + IDX2(t, 0, k);
    double m = l[id[0]];
    for (int64_t s = 1; s < k; ++s)
      if (l[id[s]] > m) m = l[id[s]];
    double z = 0.0;
    for (int64_t s = 0; s < k; ++s) z += exp(l[id[s]] - m);
    for (int64_t s = 0; s < k; ++s) w[IDX2(t, s, k)] = exp(l[id[s]] - m) / z;
  }
}

/* ------------------------------------------------------------------ */
/* Shared-expert gate: sig[t] = sigmoid(x_t . w_sg).                   */
/* RL-Kernel PR #557, #503 commit message "TP4 block": replicated       */
/* shared-expert gate; the gate is a Linear(hidden -> 1) with a sigmoid.*/
/* ------------------------------------------------------------------ */
void oracle_shared_gate(int64_t T, int64_t H, const double *x,
                        const double *wsg, double *sig) {
#pragma omp parallel for schedule(static)
  for (int64_t t = 0; t < T; ++t) {
    const double *xt = x + IDX2(t, 0, H);
    double z = 0.0;
    for (int64_t h = 0; h < H; ++h) z += xt[h] * wsg[h];
    sig[t] = sigmoid(z);
  }
}

/* ------------------------------------------------------------------ */
/* Dispatch as a stable counting sort of the routes (t, s) by expert.   */
/* RL-Kernel PR #557 "What": dispatch is a local selection of routes;   */
/* #503 "Experts": every (token, route) row has one writer.             */
/*   offsets[e]      = number of routes with expert < e  (E+1 entries)  */
/*   sorted_route[j] = t*k + s of the j-th route in (expert, t, s) order */
/*   route_pos[r]    = j such that sorted_route[j] = r                  */
/* Returns 0, or -1 if an id lies outside [0, E) (nothing is written).  */
/* ------------------------------------------------------------------ */
int oracle_permute(int64_t T, int64_t E, int64_t k, const int32_t *ids,
                   int32_t *offsets, int32_t *sorted_route,
                   int32_t *route_pos) {
  int64_t R = T * k;
  for (int64_t r = 0; r < R; ++r)
    if (ids[r] < 0 || ids[r] >= E) return -1;
  int64_t *count = (int64_t *)calloc((size_t)E, sizeof(int64_t));
  for (int64_t r = 0; r < R; ++r) count[ids[r]] += 1;
  int64_t run = 0;
  for (int64_t e = 0; e < E; ++e) {
    offsets[e] = (int32_t)run;
    run += count[e];
  }
  offsets[E] = (int32_t)run;
  int64_t *fill = (int64_t *)calloc((size_t)E, sizeof(int64_t));
  for (int64_t r = 0; r < R; ++r) { /* ascending r = ascending (t, s) */
    int64_t e = ids[r];
    int64_t j = offsets[e] + fill[e];
    fill[e] += 1;
    sorted_route[j] = (int32_t)r;
    route_pos[r] = (int32_t)j;
  }
  free(count);
  free(fill);
  return 0;
}

/* ------------------------------------------------------------------ */
/* One SwiGLU expert on one row.  #503 commit message "Experts":        */
/* per-route gate_up and down projections.  wgu is [2I][H] with the I   */
/* gate rows first and the I up rows after; wdn is [H][I].              */
/* Scratch g,u,h must hold I doubles each (NULL: allocated here).       */
/* ------------------------------------------------------------------ */
static void swiglu_ffn(int64_t H, int64_t I, const double *x,
                       const double *wgu, const double *wdn, double *g,
                       double *u, double *hbuf, double *y) {
  for (int64_t i = 0; i < I; ++i) {
    const double *wg = wgu + IDX2(i, 0, H);
    const double *wu = wgu + IDX2(I + i, 0, H);
    double ag = 0.0, au = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      ag += wg[h] * x[h];
      au += wu[h] * x[h];
    }
    g[i] = ag;
    u[i] = au;
    hbuf[i] = silu(ag) * au;
  }
  for (int64_t o = 0; o < H; ++o) {
    const double *wd = wdn + IDX2(o, 0, I);
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i) acc += wd[i] * hbuf[i];
    y[o] = acc;
  }
}

/* Exported single-row expert for tests: y[H] = FFN(x[H]). */
void oracle_expert_ffn(int64_t H, int64_t I, const double *x,
                       const double *wgu, const double *wdn, double *y) {
  double *s = (double *)malloc(sizeof(double) * (size_t)(3 * I));
  swiglu_ffn(H, I, x, wgu, wdn, s, s + I, s + 2 * I, y);
  free(s);
}

/* ------------------------------------------------------------------ */
/* Expert outputs and combine.  #503 commit message "Experts": rows are */
/* unweighted, one writer each; "Combine": the k weighted rows are      */
/* summed in route (slot) order, then the gated shared expert is added. */
/*   yr [T*k][H] (nullable): unweighted routed rows, row t*k+s          */
/*   ys [T][H]   (nullable): shared-expert rows                         */
/*   y  [T][H]             : layer output                               */
/* Tokens are independent, so any subset of rows may be passed.        */
/* ------------------------------------------------------------------ */
void oracle_moe_forward(int64_t T, int64_t H, int64_t E, int64_t k,
                        int64_t I, int64_t Is, const double *x,
                        const int32_t *ids, const double *w,
                        const double *sig, const double *wgu,
                        const double *wdn, const double *wsgu,
                        const double *wsdn, double *yr, double *ys,
                        double *y) {
  (void)E;
  int64_t Imax = I > Is ? I : Is;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double *scratch = (double *)malloc(sizeof(double) * (size_t)(3 * Imax + 2 * H));
    double *g = scratch, *u = g + Imax, *hb = u + Imax;
    double *row = hb + Imax, *acc = row + H;
    const double *xt = x + IDX2(t, 0, H);
    for (int64_t o = 0; o < H; ++o) acc[o] = 0.0;
    for (int64_t s = 0; s < k; ++s) {
      int64_t e = ids[IDX2(t, s, k)];
      swiglu_ffn(H, I, xt, wgu + e * 2 * I * H, wdn + e * H * I, g, u, hb, row);
      double ws = w[IDX2(t, s, k)];
      for (int64_t o = 0; o < H; ++o) acc[o] += ws * row[o];
      if (yr) memcpy(yr + IDX2(t * k + s, 0, H), row, sizeof(double) * (size_t)H);
    }
    swiglu_ffn(H, Is, xt, wsgu, wsdn, g, u, hb, row);
    for (int64_t o = 0; o < H; ++o) acc[o] += sig[t] * row[o];
    if (ys) memcpy(ys + IDX2(t, 0, H), row, sizeof(double) * (size_t)H);
    memcpy(y + IDX2(t, 0, H), acc, sizeof(double) * (size_t)H);
    free(scratch);
  }
}

/* ------------------------------------------------------------------ */
/* Backward, per token.  #503 commit message "Backward" and PR #557     */
/* "What": per-route input gradients are summed in ascending expert     */
/* order.  Then the shared expert, the router and the gate terms.       */
/* With L = sum_t dy_t . y_t:                                           */
/*   dw[t,s]    = dy_t . Y_{e_s}(x_t)           (route-weight grad)     */
/*   dlogit[t,s]= w_s (dw_s - sum_j w_j dw_j)   (softmax over the set)  */
/*   dsig[t]    = dy_t . Ys(x_t);  dz[t] = dsig sig (1 - sig)            */
/*   dx[t]      = sum_{routes, ascending e} J_e^T (w_s dy_t)            */
/*              + J_s^T (sig dy_t) + sum_s dlogit_s Wr[e_s] + dz w_sg   */
/* J^T v for the SwiGLU FFN: dh = Wdn^T v, dg = dh u silu'(g),          */
/* du = dh silu(g), dx = Wg^T dg + Wu^T du.                             */
/* ------------------------------------------------------------------ */
static void swiglu_vjp_x(int64_t H, int64_t I, const double *x,
                         const double *wgu, const double *wdn,
                         const double *v, double *g, double *u, double *dh,
                         double *dx_acc) {
  for (int64_t i = 0; i < I; ++i) {
    const double *wg = wgu + IDX2(i, 0, H);
    const double *wu = wgu + IDX2(I + i, 0, H);
    double ag = 0.0, au = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      ag += wg[h] * x[h];
      au += wu[h] * x[h];
    }
    g[i] = ag;
    u[i] = au;
  }
  for (int64_t i = 0; i < I; ++i) {
    double acc = 0.0;
    for (int64_t o = 0; o < H; ++o) acc += wdn[IDX2(o, i, I)] * v[o];
    dh[i] = acc;
  }
  /* dg_i = dh_i u_i silu'(g_i), du_i = dh_i silu(g_i); stored over g, u */
  for (int64_t i = 0; i < I; ++i) {
    double dgi = dh[i] * u[i] * silu_grad(g[i]);
    double dui = dh[i] * silu(g[i]);
    g[i] = dgi;
    u[i] = dui;
  }
  /* dx_acc[h] += sum_i dg_i Wg[i,h] + du_i Wu[i,h]: the vector product of
     this expert is formed first, then added to the running sum. */
  for (int64_t h = 0; h < H; ++h) {
    double acc = 0.0;
    for (int64_t i = 0; i < I; ++i)
      acc += g[i] * wgu[IDX2(i, h, H)] + u[i] * wgu[IDX2(I + i, h, H)];
    dx_acc[h] += acc;
  }
}

void oracle_moe_backward_tokens(int64_t T, int64_t H, int64_t E, int64_t k,
                                int64_t I, int64_t Is, const double *x,
                                const int32_t *ids, const double *w,
                                const double *sig, const double *wr,
                                const double *wsg, const double *wgu,
                                const double *wdn, const double *wsgu,
                                const double *wsdn, const double *dy,
                                double *dx, double *dw, double *dlogit,
                                double *dsig_out) {
  (void)E;
  int64_t Imax = I > Is ? I : Is;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t t = 0; t < T; ++t) {
    double *scr = (double *)malloc(sizeof(double) * (size_t)(4 * Imax + 3 * H + 2 * k));
    double *g = scr, *u = g + Imax, *hb = u + Imax, *dh = hb + Imax;
    double *row = dh + Imax, *v = row + H, *acc = v + H;
    double *dws = acc + H;
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
    const double *xt = x + IDX2(t, 0, H);
    const double *dyt = dy + IDX2(t, 0, H);
    const int32_t *id = ids + IDX2(t, 0, k);
    const double *wt = w + IDX2(t, 0, k);

    /* route-weight grads dw_s = dy . Y_e(x) */
    for (int64_t s = 0; s < k; ++s) {
      swiglu_ffn(H, I, xt, wgu + (int64_t)id[s] * 2 * I * H,
                 wdn + (int64_t)id[s] * H * I, g, u, hb, row);
      double a = 0.0;
      for (int64_t o = 0; o < H; ++o) a += dyt[o] * row[o];
      dws[s] = a;
    }
    /* softmax-over-the-set Jacobian */
    double wdw = 0.0;
    for (int64_t s = 0; s < k; ++s) wdw += wt[s] * dws[s];
    for (int64_t s = 0; s < k; ++s) dws[k + s] = wt[s] * (dws[s] - wdw);

    /* slots in ascending expert id (ids in a row are distinct) */
    for (int64_t s = 0; s < k; ++s) order[s] = (int32_t)s;
    for (int64_t a = 1; a < k; ++a) { /* insertion sort by expert id */
      int32_t cur = order[a];
      int64_t b = a - 1;
      while (b >= 0 && id[order[b]] > id[cur]) { order[b + 1] = order[b]; --b; }
      order[b + 1] = cur;
    }
    for (int64_t o = 0; o < H; ++o) acc[o] = 0.0;
    for (int64_t a = 0; a < k; ++a) {
      int64_t s = order[a];
      int64_t e = id[s];
      for (int64_t o = 0; o < H; ++o) v[o] = wt[s] * dyt[o];
      swiglu_vjp_x(H, I, xt, wgu + e * 2 * I * H, wdn + e * H * I, v, g, u, dh, acc);
    }
    /* shared expert */
    swiglu_ffn(H, Is, xt, wsgu, wsdn, g, u, hb, row);
    double dsig = 0.0;
    for (int64_t o = 0; o < H; ++o) dsig += dyt[o] * row[o];
    for (int64_t o = 0; o < H; ++o) v[o] = sig[t] * dyt[o];
    swiglu_vjp_x(H, Is, xt, wsgu, wsdn, v, g, u, dh, acc);
    /* router */
    for (int64_t o = 0; o < H; ++o) {
      double a = 0.0;
      for (int64_t s = 0; s < k; ++s) a += dws[k + s] * wr[IDX2(id[s], o, H)];
      acc[o] += a;
    }
    /* gate */
    double dz = dsig * sig[t] * (1.0 - sig[t]);
    for (int64_t o = 0; o < H; ++o) acc[o] += dz * wsg[o];

    memcpy(dx + IDX2(t, 0, H), acc, sizeof(double) * (size_t)H);
    if (dw) for (int64_t s = 0; s < k; ++s) dw[IDX2(t, s, k)] = dws[s];
    if (dlogit) for (int64_t s = 0; s < k; ++s) dlogit[IDX2(t, s, k)] = dws[k + s];
    if (dsig_out) dsig_out[t] = dsig;
    free(order);
    free(scr);
  }
}

/* ------------------------------------------------------------------ */
/* Expert weight gradients for experts e in [e0, e1).  #503 commit      */
/* message "Backward": per-expert GEMMs; sums over the expert's routes  */
/* in ascending (t, s) order.                                           */
/*   dWdn[e] = sum_routes (w_s dy_t) h^T          [H][I]                */
/*   dWg[e]  = sum_routes dg x_t^T, dWu[e] = sum du x_t^T  [2I][H]       */
/* Outputs hold experts e0..e1-1 only: dwgu[(e-e0)][2I][H], dwdn[(e-e0)][H][I]. */
/* ------------------------------------------------------------------ */
static void swiglu_weight_grads(int64_t H, int64_t I, const double *x,
                                const double *wgu, const double *wdn,
                                const double *v, double *g, double *u,
                                double *hb, double *dh, double *dwgu,
                                double *dwdn) {
  for (int64_t i = 0; i < I; ++i) {
    const double *wg = wgu + IDX2(i, 0, H);
    const double *wu = wgu + IDX2(I + i, 0, H);
    double ag = 0.0, au = 0.0;
    for (int64_t h = 0; h < H; ++h) {
      ag += wg[h] * x[h];
      au += wu[h] * x[h];
    }
    g[i] = ag;
    u[i] = au;
    hb[i] = silu(ag) * au;
  }
  for (int64_t i = 0; i < I; ++i) {
    double acc = 0.0;
    for (int64_t o = 0; o < H; ++o) acc += wdn[IDX2(o, i, I)] * v[o];
    dh[i] = acc;
  }
  for (int64_t o = 0; o < H; ++o)
    for (int64_t i = 0; i < I; ++i) dwdn[IDX2(o, i, I)] += v[o] * hb[i];
  for (int64_t i = 0; i < I; ++i) {
    double dg = dh[i] * u[i] * silu_grad(g[i]);
    double du = dh[i] * silu(g[i]);
    for (int64_t h = 0; h < H; ++h) {
      dwgu[IDX2(i, h, H)] += dg * x[h];
      dwgu[IDX2(I + i, h, H)] += du * x[h];
    }
  }
}

void oracle_moe_backward_expert_weights(int64_t T, int64_t H, int64_t E,
                                        int64_t k, int64_t I, const double *x,
                                        const int32_t *ids, const double *w,
                                        const double *dy, const double *wgu,
                                        const double *wdn, int64_t e0,
                                        int64_t e1, double *dwgu,
                                        double *dwdn) {
  (void)E;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t e = e0; e < e1; ++e) {
    double *scr = (double *)malloc(sizeof(double) * (size_t)(4 * I + H));
    double *g = scr, *u = g + I, *hb = u + I, *dh = hb + I, *v = dh + I;
    double *dge = dwgu + (e - e0) * 2 * I * H, *dde = dwdn + (e - e0) * H * I;
    memset(dge, 0, sizeof(double) * (size_t)(2 * I * H));
    memset(dde, 0, sizeof(double) * (size_t)(H * I));
    for (int64_t t = 0; t < T; ++t)
      for (int64_t s = 0; s < k; ++s) {
        if (ids[IDX2(t, s, k)] != e) continue;
        double ws = w[IDX2(t, s, k)];
        for (int64_t o = 0; o < H; ++o) v[o] = ws * dy[IDX2(t, o, H)];
        swiglu_weight_grads(H, I, x + IDX2(t, 0, H), wgu + e * 2 * I * H,
                            wdn + e * H * I, v, g, u, hb, dh, dge, dde);
      }
    free(scr);
  }
}

/* Shared-expert weight gradients: the same chain with v = sig[t] dy_t.   */
/* The per-token vectors h, dg, du are formed first (tokens independent), */
/* then every weight-gradient entry sums over tokens in ascending order.  */
void oracle_moe_backward_shared_weights(int64_t T, int64_t H, int64_t Is,
                                        const double *x, const double *sig,
                                        const double *dy, const double *wsgu,
                                        const double *wsdn, double *dwsgu,
                                        double *dwsdn) {
  double *hv = (double *)malloc(sizeof(double) * (size_t)(T * Is));
  double *dgv = (double *)malloc(sizeof(double) * (size_t)(T * Is));
  double *duv = (double *)malloc(sizeof(double) * (size_t)(T * Is));
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t t = 0; t < T; ++t) {
    const double *xt = x + IDX2(t, 0, H);
    for (int64_t i = 0; i < Is; ++i) {
      const double *wg = wsgu + IDX2(i, 0, H);
      const double *wu = wsgu + IDX2(Is + i, 0, H);
      double ag = 0.0, au = 0.0;
      for (int64_t h = 0; h < H; ++h) {
        ag += wg[h] * xt[h];
        au += wu[h] * xt[h];
      }
      double dh = 0.0;
      for (int64_t o = 0; o < H; ++o)
        dh += wsdn[IDX2(o, i, Is)] * (sig[t] * dy[IDX2(t, o, H)]);
      hv[IDX2(t, i, Is)] = silu(ag) * au;
      dgv[IDX2(t, i, Is)] = dh * au * silu_grad(ag);
      duv[IDX2(t, i, Is)] = dh * silu(ag);
    }
  }
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t o = 0; o < H; ++o)
    for (int64_t i = 0; i < Is; ++i) {
      double acc = 0.0;
      for (int64_t t = 0; t < T; ++t)
        acc += (sig[t] * dy[IDX2(t, o, H)]) * hv[IDX2(t, i, Is)];
      dwsdn[IDX2(o, i, Is)] = acc;
    }
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t i = 0; i < Is; ++i)
    for (int64_t h = 0; h < H; ++h) {
      double ag = 0.0, au = 0.0;
      for (int64_t t = 0; t < T; ++t) {
        ag += dgv[IDX2(t, i, Is)] * x[IDX2(t, h, H)];
        au += duv[IDX2(t, i, Is)] * x[IDX2(t, h, H)];
      }
      dwsgu[IDX2(i, h, H)] = ag;
      dwsgu[IDX2(Is + i, h, H)] = au;
    }
  free(hv);
  free(dgv);
  free(duv);
}

/* ------------------------------------------------------------------ */
/* Router and gate weight gradients:                                   */
/*   dWr[e,h]  = sum_t sum_{s: ids[t,s]=e} dlogit[t,s] x[t,h]           */
/*   dwsg[h]   = sum_t dz[t] x[t,h],  dz = dsig sig (1 - sig)            */
/* Tokens in ascending order.                                          */
/* ------------------------------------------------------------------ */
void oracle_moe_backward_router(int64_t T, int64_t H, int64_t E, int64_t k,
                                const double *x, const int32_t *ids,
                                const double *dlogit, const double *sig,
                                const double *dsig, double *dwr,
                                double *dwsg) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t e = 0; e < E; ++e) {
    double *row = dwr + IDX2(e, 0, H);
    for (int64_t h = 0; h < H; ++h) row[h] = 0.0;
    for (int64_t t = 0; t < T; ++t)
      for (int64_t s = 0; s < k; ++s) {
        if (ids[IDX2(t, s, k)] != e) continue;
        double d = dlogit[IDX2(t, s, k)];
        for (int64_t h = 0; h < H; ++h) row[h] += d * x[IDX2(t, h, H)];
      }
  }
  for (int64_t h = 0; h < H; ++h) dwsg[h] = 0.0;
  for (int64_t t = 0; t < T; ++t) {
    double dz = dsig[t] * sig[t] * (1.0 - sig[t]);
    for (int64_t h = 0; h < H; ++h) dwsg[h] += dz * x[IDX2(t, h, H)];
  }
}
