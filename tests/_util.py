"""Shared helpers of the test suite: cached seeded inputs, the near-tie routing
rule, per-token oracle evaluation at full size, and tolerance checks.

Tolerances (the layer's stated bar): bf16 configurations max |y - y64| <= 2e-2
and ||y - y64||_2 / ||y64||_2 <= 5e-3 per output tensor; the FP32 tiny
configuration max |y - y64| <= 1e-4.  Routes and the permutation are compared
bit for bit, except near-tie tokens: those where two adjacent logits among
the k+1 largest (which decide the selected set at the k-th/(k+1)-th boundary
and the slot order inside the set) are less than 1e-4 apart in either the
oracle's FP64 logits or the GPU's FP32 logits.  For those the oracle selects
and orders from the GPU's logits (ties to the lower id) and computes the
weights in FP64 on that ordered set.
"""
from __future__ import annotations

import ctypes
import functools
import os
import re
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np
import torch

import oracle
from top_routed_grouped_gb300 import inputs as I

TIE_GAP = 1e-4
BF16_MAX_ABS = 2e-2
BF16_REL_L2 = 5e-3
F32_MAX_ABS = 1e-4

# Every value comparison of the session: (tensor, precision, max_abs, scale,
# rel_l2, elements), printed as a per-tensor summary at the end of the run.
RECORDS: list[tuple] = []
_rec_lock = threading.Lock()


def record(what: str, kind: str, max_abs: float, scale: float, rel: float, n: int) -> None:
    name = re.split(r"[\s\[(,]", what.strip(), maxsplit=1)[0] or what
    with _rec_lock:
        RECORDS.append((name, kind, max_abs, scale, rel, n))


def summary_lines() -> list[str]:
    """Worst case per (tensor, precision) over the session's comparisons."""
    worst: dict = {}
    for name, kind, m, s, r, n in RECORDS:
        key = (kind, name)
        w = worst.setdefault(key, [0.0, 1.0, 0.0, 0, 0])
        if m / s >= w[0] / w[1]:
            w[0], w[1] = m, s
        w[2] = max(w[2], r)
        w[3] += n
        w[4] += 1
    lines = [f"{'tensor':<15}{'dtype':<6}{'max_abs':>10}{'scale':>8}{'rel_l2':>10}{'elements':>12}{'checks':>7}"]
    for (kind, name), (m, s, r, n, c) in sorted(worst.items()):
        lines.append(f"{name:<15}{kind:<6}{m:>10.2e}{s:>8.3g}{r:>10.2e}{n:>12d}{c:>7d}")
    return lines


def _omp_one_thread() -> None:
    """Limit the calling thread's OpenMP regions to one thread (the oracle's
    per-token calls then run side by side in a thread pool)."""
    try:
        ctypes.CDLL("libgomp.so.1").omp_set_num_threads(1)
    except OSError:  # pragma: no cover
        pass


def _pool_map(fn, items):
    n = max(1, min(16, len(os.sched_getaffinity(0))))
    with ThreadPoolExecutor(n, initializer=_omp_one_thread) as ex:
        return list(ex.map(fn, items))


@functools.lru_cache(maxsize=None)
def full_weights():
    """bf16 weights of the 512-expert layer (identical for every bf16 workload)."""
    cfg = I.CONFIGS["bf16_t1024"]
    d = I.make_inputs(cfg, T=1)
    return {k: v for k, v in d.items() if k not in ("x", "dy", "router_bias")}


@functools.lru_cache(maxsize=None)
def full_x(T: int):
    return I.normal((T, 2048), 0, I._STREAM["x"], 1.0, torch.bfloat16)


@functools.lru_cache(maxsize=None)
def full_dy(T: int):
    return I.normal((T, 2048), 2, I._STREAM["dy"], 1.0, torch.bfloat16)


def to_dev(d: dict, device="cuda") -> dict:
    return {k: (v.to(device) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}


def min_top_gap(logits: np.ndarray, k: int) -> np.ndarray:
    """Smallest gap between adjacent values among the k+1 largest logits of each row."""
    E = logits.shape[1]
    m = min(k + 1, E)
    top = -np.sort(-logits, axis=1)[:, :m]
    if m < 2:
        return np.full(logits.shape[0], np.inf)
    return np.min(top[:, :-1] - top[:, 1:], axis=1)


def oracle_routes(x, w_router, bias, k: int, gpu_logits: np.ndarray):
    """Oracle routes with the near-tie rule.  Returns (ids, w, near_mask, logits64)."""
    l64 = oracle.router_logits(x, w_router, bias)
    ids = oracle.topk_select(l64, k)
    gl = np.asarray(gpu_logits, dtype=np.float64)
    near = (min_top_gap(l64, k) < TIE_GAP) | (min_top_gap(gl, k) < TIE_GAP)
    if near.any():
        ids[near] = oracle.topk_select(gl[near], k)
    w = oracle.topk_weights(l64, ids)
    return ids, w, near, l64


def oracle_rows(x_rows, ids_rows, w_rows, sig_rows, W: dict, want_rows=False):
    """Oracle forward of a few tokens at full size, one token at a time with
    only its k experts widened to float64 (the experts are remapped to 0..k-1);
    the tokens run side by side in a thread pool."""
    def one(t):
        e = torch.as_tensor(np.asarray(ids_rows[t], dtype=np.int64))
        wgu = W["w_gate_up"].index_select(0, e.to(W["w_gate_up"].device)).cpu()
        wdn = W["w_down"].index_select(0, e.to(W["w_down"].device)).cpu()
        local = np.arange(len(e), dtype=np.int32)[None, :]
        return oracle.moe_forward(x_rows[t:t + 1], local, np.asarray(w_rows[t:t + 1]), np.asarray(sig_rows[t:t + 1]),
                                  wgu, wdn, W["ws_gate_up"].cpu(), W["ws_down"].cpu(), want_rows=want_rows)
    res = _pool_map(one, range(x_rows.shape[0]))
    if want_rows:
        return tuple(np.concatenate([r[i] for r in res]) for i in range(3))
    return np.concatenate(res)


def oracle_segment_rows(x_tokens, w_gate_up_e, w_down_e):
    """Oracle rows of one expert on the given token rows (its whole segment):
    the layer with that one expert, weight 1, and no shared expert."""
    n, H = x_tokens.shape
    ids = np.zeros((n, 1), np.int32)
    _, yr, _ = oracle.moe_forward(x_tokens, ids, np.ones((n, 1)), np.zeros(n), w_gate_up_e[None], w_down_e[None],
                                  np.zeros((0, H)), np.zeros((H, 0)), want_rows=True)
    return yr


def oracle_shared_rows(x_tokens, ws_gate_up, ws_down):
    """Oracle rows of the shared expert on the given token rows (no routes)."""
    n, H = x_tokens.shape
    _, _, ys = oracle.moe_forward(x_tokens, np.zeros((n, 0), np.int32), np.zeros((n, 0)), np.ones(n),
                                  np.zeros((1, 0, H)), np.zeros((1, H, 0)), ws_gate_up, ws_down, want_rows=True)
    return ys


def err_stats(got, ref) -> tuple[float, float]:
    g = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    max_abs = float(np.max(np.abs(g - r))) if g.size else 0.0
    den = float(np.linalg.norm(r))
    rel = float(np.linalg.norm(g - r) / den) if den > 0 else float(np.linalg.norm(g - r))
    return max_abs, rel


def assert_bf16_close(got, ref, what=""):
    m, r = err_stats(got, ref)
    record(what, "bf16", m, 1.0, r, int(np.asarray(ref).size))
    assert m <= BF16_MAX_ABS and r <= BF16_REL_L2, f"{what}: max_abs={m:.3e} rel_l2={r:.3e}"
    return m, r


def assert_f32_close(got, ref, what=""):
    m, r = err_stats(got, ref)
    record(what, "f32", m, 1.0, r, int(np.asarray(ref).size))
    assert m <= F32_MAX_ABS, f"{what}: max_abs={m:.3e}"
    return m, r


def bits(t: torch.Tensor) -> torch.Tensor:
    """Raw bit pattern (signed zeros and NaN payloads compare exactly)."""
    t = t.detach().contiguous()
    view = {torch.bfloat16: torch.int16, torch.float16: torch.int16, torch.float32: torch.int32,
            torch.int32: torch.int32}[t.dtype]
    return t.view(view).cpu()


# ---------------------------------------------------------------- backward
def grad_scale(ref) -> float:
    """Scale of a gradient tensor for its max-abs bar: max(1, max|ref|).

    Weight gradients are sums over up to T rows, so their entries grow like
    the square root of the row count; the layer's max-abs bar (stated for
    outputs of unit scale) is applied relative to that scale."""
    r = np.asarray(ref, np.float64)
    return max(1.0, float(np.max(np.abs(r)))) if r.size else 1.0


def assert_grad_close(got, ref, what="", f32=False):
    m, r = err_stats(got, ref)
    s = grad_scale(ref)
    record(what, "f32" if f32 else "bf16", m, s, r, int(np.asarray(ref).size))
    if f32:
        assert m <= F32_MAX_ABS * s, f"{what}: max_abs={m:.3e} scale={s:.3g}"
    else:
        assert m <= BF16_MAX_ABS * s and r <= BF16_REL_L2, f"{what}: max_abs={m:.3e} scale={s:.3g} rel_l2={r:.3e}"
    print(f"{what}: max_abs={m:.3e} scale={s:.3g} rel_l2={r:.3e}")
    return m, r


def oracle_bwd_rows(x_rows, ids_rows, w_rows, sig_rows, dy_rows, W: dict):
    """Oracle per-token backward (dx, dw, dlogit, dsig) of a few tokens at full
    size, one token at a time with only its k experts widened to float64;
    the tokens run side by side in a thread pool.  Local ids keep the
    ascending order of the global ids, so the oracle's ascending-expert sum
    of the routed input gradients is unchanged."""
    def one(t):
        e = np.asarray(ids_rows[t], dtype=np.int64)
        srt = np.sort(e)
        local = np.searchsorted(srt, e).astype(np.int32)[None, :]
        idx = torch.as_tensor(srt)
        g = lambda name: W[name].index_select(0, idx.to(W[name].device)).cpu()  # noqa: E731
        return oracle.backward_tokens(x_rows[t:t + 1], local, np.asarray(w_rows[t:t + 1]),
                                      np.asarray(sig_rows[t:t + 1]), g("w_router"), W["w_shared_gate"].cpu(),
                                      g("w_gate_up"), g("w_down"), W["ws_gate_up"].cpu(), W["ws_down"].cpu(),
                                      dy_rows[t:t + 1])
    res = _pool_map(one, range(x_rows.shape[0]))
    return tuple(np.concatenate([r[i] for r in res]) for i in range(4))


def small_layer(T, H, E, k, I_, Is, seed=11):
    """A small bf16 layer of the given shape (same recipe as the workloads)."""
    s = seed
    return {"x": I.normal((T, H), s, 0, 1.0, torch.bfloat16),
            "w_router": I.normal((E, H), s, 1, 0.02, torch.float32),
            "w_shared_gate": I.normal((H,), s, 2, 0.02, torch.bfloat16),
            "w_gate_up": I.normal((E, 2 * I_, H), s, 4, 0.02, torch.bfloat16),
            "w_down": I.normal((E, H, I_), s, 5, 0.02, torch.bfloat16),
            "ws_gate_up": I.normal((2 * Is, H), s, 6, 0.02, torch.bfloat16),
            "ws_down": I.normal((H, Is), s, 7, 0.02, torch.bfloat16),
            "dy": I.normal((T, H), s + 1, 8, 1.0, torch.bfloat16)}
