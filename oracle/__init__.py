"""FP64 CPU oracle of the batch-invariant MoE layer.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only ``tests/``, the smoke check in
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import this
package.  It shares no code with the CUDA path (``top_routed_grouped_gb300``)
and neither imports the other.

The arithmetic lives in ``moe_oracle.c`` (plain C loops in double precision,
OpenMP over independent tokens / experts).  This module only compiles it with
gcc, loads it with ctypes and marshals numpy arrays.  Every function states the
page passage it follows in the C source; in short:

* routing  -- RL-Kernel PR #557, #503 commit message "Routing": FP32 router
  GEMM, fixed-order softmax, stable descending top-k with ties to the lower
  expert id, renormalisation of the k selected weights;
* dispatch -- PR #557 "What": local selection; a stable counting sort of the
  routes by expert;
* experts  -- #503 "Experts": unweighted per-route SwiGLU rows, one writer;
* combine  -- #503 "Combine": k ordered weighted adds, then the sigmoid-gated
  shared expert;
* backward -- #503 "Backward": per-expert weight gradients, per-route input
  gradients summed in ascending expert order.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "moe_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off"]


def build(force: bool = False) -> str:
    """Compile ``moe_oracle.c`` into ``liboracle.so`` next to it (gcc)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, "-o", tmp, _SRC, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB)
            i64, dp, ip = ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p
            sigs = {
                "oracle_router_logits": ([i64, i64, i64, dp, dp, dp, dp], None),
                "oracle_topk_select": ([i64, i64, i64, dp, ip], i64),
                "oracle_topk_weights": ([i64, i64, i64, dp, ip, dp], None),
                "oracle_shared_gate": ([i64, i64, dp, dp, dp], None),
                "oracle_permute": ([i64, i64, i64, ip, ip, ip, ip], ctypes.c_int),
                "oracle_expert_ffn": ([i64, i64, dp, dp, dp, dp], None),
                "oracle_moe_forward": ([i64] * 6 + [dp, ip] + [dp] * 9, None),
                "oracle_moe_backward_tokens": ([i64] * 6 + [dp, ip] + [dp] * 13, None),
                "oracle_moe_backward_expert_weights": ([i64] * 5 + [dp, ip] + [dp] * 4 + [i64, i64, dp, dp], None),
                "oracle_moe_backward_shared_weights": ([i64] * 3 + [dp] * 7, None),
                "oracle_moe_backward_router": ([i64] * 4 + [dp, ip] + [dp] * 5, None),
            }
            for name, (args, res) in sigs.items():
                fn = getattr(lib, name)
                fn.argtypes = args
                fn.restype = res
            _lib = lib
    return _lib


def _f64(a) -> np.ndarray:
    """Exact widening to a C-contiguous float64 array (bf16/fp32 -> f64 is exact)."""
    if a is None:
        return None
    if hasattr(a, "detach"):  # torch tensor
        import torch

        a = a.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _i32(a) -> np.ndarray:
    if hasattr(a, "detach"):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


def _p(a):
    return None if a is None else a.ctypes.data


# ---------------------------------------------------------------- routing
def router_logits(x, w_router, bias=None) -> np.ndarray:
    """l[t,e] = x_t . Wr_e (+ bias_e), FP64.  x [T,H], Wr [E,H]."""
    x, wr, b = _f64(x), _f64(w_router), _f64(bias)
    T, H = x.shape
    E = wr.shape[0]
    out = np.empty((T, E), np.float64)
    _load().oracle_router_logits(T, H, E, _p(x), _p(wr), _p(b), _p(out))
    return out


def topk_select(logits, k: int) -> np.ndarray:
    """ids [T,k]: descending logit, ties to the lower expert id."""
    l = _f64(logits)
    T, E = l.shape
    ids = np.empty((T, k), np.int32)
    _load().oracle_topk_select(T, E, k, _p(l), _p(ids))
    return ids


def topk_weights(logits, ids) -> np.ndarray:
    """w [T,k]: softmax over the selected logits (= softmax then renormalise)."""
    l, ids = _f64(logits), _i32(ids)
    T, E = l.shape
    k = ids.shape[1]
    w = np.empty((T, k), np.float64)
    _load().oracle_topk_weights(T, E, k, _p(l), _p(ids), _p(w))
    return w


def shared_gate(x, w_shared_gate) -> np.ndarray:
    """sig [T] = sigmoid(x_t . w_sg)."""
    x, wsg = _f64(x), _f64(w_shared_gate)
    T, H = x.shape
    sig = np.empty((T,), np.float64)
    _load().oracle_shared_gate(T, H, _p(x), _p(wsg), _p(sig))
    return sig


def route(x, w_router, w_shared_gate, k: int, bias=None):
    """Full routing: (logits, ids, w, sig), FP64."""
    logits = router_logits(x, w_router, bias)
    ids = topk_select(logits, k)
    return logits, ids, topk_weights(logits, ids), shared_gate(x, w_shared_gate)


def permute(ids, E: int):
    """Stable counting sort of routes by expert: (offsets[E+1], sorted_route[R], route_pos[R])."""
    ids = _i32(ids)
    T, k = ids.shape
    R = T * k
    offsets = np.empty((E + 1,), np.int32)
    sorted_route = np.empty((R,), np.int32)
    route_pos = np.empty((R,), np.int32)
    rc = _load().oracle_permute(T, E, k, _p(ids), _p(offsets), _p(sorted_route), _p(route_pos))
    if rc != 0:
        raise ValueError("expert id outside [0, E)")
    return offsets, sorted_route, route_pos


# ---------------------------------------------------------------- experts
def expert_ffn(x_row, w_gate_up_e, w_down_e) -> np.ndarray:
    """One SwiGLU expert on one row: Wdn (silu(Wg x) * (Wu x))."""
    x, wgu, wdn = _f64(x_row), _f64(w_gate_up_e), _f64(w_down_e)
    H = x.shape[0]
    I = wgu.shape[0] // 2
    y = np.empty((H,), np.float64)
    _load().oracle_expert_ffn(H, I, _p(x), _p(wgu), _p(wdn), _p(y))
    return y


def moe_forward(x, ids, w, sig, w_gate_up, w_down, ws_gate_up, ws_down, want_rows: bool = False):
    """Layer output y [T,H] for given routes; optionally the unweighted rows.

    Returns y, or (y, yr [T*k,H], ys [T,H]) when ``want_rows``.
    """
    x, ids, w, sig = _f64(x), _i32(ids), _f64(w), _f64(sig)
    wgu, wdn, wsgu, wsdn = _f64(w_gate_up), _f64(w_down), _f64(ws_gate_up), _f64(ws_down)
    T, H = x.shape
    k = ids.shape[1]
    E, I2, _ = wgu.shape
    I, Is = I2 // 2, wsgu.shape[0] // 2
    y = np.empty((T, H), np.float64)
    yr = np.empty((T * k, H), np.float64) if want_rows else None
    ys = np.empty((T, H), np.float64) if want_rows else None
    _load().oracle_moe_forward(T, H, E, k, I, Is, _p(x), _p(ids), _p(w), _p(sig), _p(wgu), _p(wdn),
                               _p(wsgu), _p(wsdn), _p(yr), _p(ys), _p(y))
    return (y, yr, ys) if want_rows else y


def layer_forward(x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, k: int, bias=None):
    """Route, then experts and combine.  Returns dict with logits, ids, w, sig, y."""
    logits, ids, w, sig = route(x, w_router, w_shared_gate, k, bias)
    y = moe_forward(x, ids, w, sig, w_gate_up, w_down, ws_gate_up, ws_down)
    return {"logits": logits, "ids": ids, "w": w, "sig": sig, "y": y}


# ---------------------------------------------------------------- backward
def backward_tokens(x, ids, w, sig, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, dy):
    """Per-token backward: dx [T,H], dw [T,k], dlogit [T,k], dsig [T]."""
    x, ids, w, sig, dy = _f64(x), _i32(ids), _f64(w), _f64(sig), _f64(dy)
    wr, wsg = _f64(w_router), _f64(w_shared_gate)
    wgu, wdn, wsgu, wsdn = _f64(w_gate_up), _f64(w_down), _f64(ws_gate_up), _f64(ws_down)
    T, H = x.shape
    k = ids.shape[1]
    E, I2, _ = wgu.shape
    I, Is = I2 // 2, wsgu.shape[0] // 2
    dx = np.empty((T, H), np.float64)
    dw = np.empty((T, k), np.float64)
    dl = np.empty((T, k), np.float64)
    ds = np.empty((T,), np.float64)
    _load().oracle_moe_backward_tokens(T, H, E, k, I, Is, _p(x), _p(ids), _p(w), _p(sig), _p(wr), _p(wsg),
                                       _p(wgu), _p(wdn), _p(wsgu), _p(wsdn), _p(dy), _p(dx), _p(dw),
                                       _p(dl), _p(ds))
    return dx, dw, dl, ds


def backward_expert_weights(x, ids, w, dy, w_gate_up, w_down, e0: int = 0, e1: int | None = None):
    """dW_gate_up [e1-e0, 2I, H], dW_down [e1-e0, H, I] for experts e0..e1-1."""
    x, ids, w, dy = _f64(x), _i32(ids), _f64(w), _f64(dy)
    T, H = x.shape
    k = ids.shape[1]
    E = w_gate_up.shape[0]
    e1 = E if e1 is None else e1
    wgu, wdn = _f64(w_gate_up[e0:e1]), _f64(w_down[e0:e1])
    I = wgu.shape[1] // 2
    n = e1 - e0
    dwgu = np.empty((n, 2 * I, H), np.float64)
    dwdn = np.empty((n, H, I), np.float64)
    # Pass the slice with shifted ids: the C routine indexes weights by e - 0
    # over its own range, so shift the range to start at zero.
    ids_shift = np.where((ids >= e0) & (ids < e1), ids - e0, -1).astype(np.int32)
    _load().oracle_moe_backward_expert_weights(T, H, n, k, I, _p(x), _p(ids_shift), _p(w), _p(dy),
                                               _p(wgu), _p(wdn), 0, n, _p(dwgu), _p(dwdn))
    return dwgu, dwdn


def backward_shared_weights(x, sig, dy, ws_gate_up, ws_down):
    """dWs_gate_up [2Is, H], dWs_down [H, Is]."""
    x, sig, dy = _f64(x), _f64(sig), _f64(dy)
    wsgu, wsdn = _f64(ws_gate_up), _f64(ws_down)
    T, H = x.shape
    Is = wsgu.shape[0] // 2
    dwsgu = np.empty((2 * Is, H), np.float64)
    dwsdn = np.empty((H, Is), np.float64)
    _load().oracle_moe_backward_shared_weights(T, H, Is, _p(x), _p(sig), _p(dy), _p(wsgu), _p(wsdn),
                                               _p(dwsgu), _p(dwsdn))
    return dwsgu, dwsdn


def backward_router(x, ids, dlogit, sig, dsig, E: int):
    """dWr [E, H] and dw_sg [H]."""
    x, ids, dl, sig, ds = _f64(x), _i32(ids), _f64(dlogit), _f64(sig), _f64(dsig)
    T, H = x.shape
    k = ids.shape[1]
    dwr = np.empty((E, H), np.float64)
    dwsg = np.empty((H,), np.float64)
    _load().oracle_moe_backward_router(T, H, E, k, _p(x), _p(ids), _p(dl), _p(sig), _p(ds), _p(dwr), _p(dwsg))
    return dwr, dwsg


def layer_backward(x, ids, w, sig, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, dy):
    """All gradients of L = sum(dy * y) with the routes held fixed."""
    dx, dw, dl, ds = backward_tokens(x, ids, w, sig, w_router, w_shared_gate, w_gate_up, w_down,
                                     ws_gate_up, ws_down, dy)
    dwgu, dwdn = backward_expert_weights(x, ids, w, dy, w_gate_up, w_down)
    dwsgu, dwsdn = backward_shared_weights(x, sig, dy, ws_gate_up, ws_down)
    dwr, dwsg = backward_router(x, ids, dl, sig, ds, np.asarray(w_router.shape)[0])
    return {"dx": dx, "dw": dw, "dlogit": dl, "dsig": ds, "dw_gate_up": dwgu, "dw_down": dwdn,
            "dws_gate_up": dwsgu, "dws_down": dwsdn, "dw_router": dwr, "dw_shared_gate": dwsg}
