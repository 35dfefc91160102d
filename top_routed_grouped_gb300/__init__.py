"""Python binding of ``libmoe_gb300.so``, the batch-invariant MoE layer for GB300.

This module only marshals arguments: torch supplies device memory and the
stream, every step of the layer runs in the library's CUDA kernels.  The
functions named ``moe_*`` mirror the C entry points of ``include/moe.h`` one to
one (pointers in, status out, raising ``MoEError`` on a non-zero status); the
lower-case helpers (``route``, ``permute``, ``grouped_ffn``, ``combine``,
``forward``, ``backward``) allocate the outputs with torch and call them.

There is no fallback: if the library is missing, ``lib()`` raises.  Build it
with ``python -m top_routed_grouped_gb300.build`` (or ``__graft_entry__.build()``).

``MoELayer`` / ``MoEFunction`` (``layer.py``): the layer as a torch module
whose autograd Function calls ``moe_forward`` and ``moe_backward``.
"""
from __future__ import annotations

import ctypes
import os
import threading

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe_gb300.so")

MOE_F32, MOE_BF16 = 0, 1
OP = {"route": 0, "permute": 1, "grouped_ffn": 2, "combine": 3, "backward": 4, "forward": 5}
STATUS = {0: "MOE_OK", -1: "MOE_ERR_INVALID_ARG", -2: "MOE_ERR_UNSUPPORTED", -3: "MOE_ERR_WORKSPACE",
          -4: "MOE_ERR_CUDA", -5: "MOE_ERR_DEVICE"}
EXPORTED = ("moe_workspace_size", "moe_status_string", "moe_route", "moe_permute", "moe_grouped_ffn",
            "moe_combine", "moe_forward", "moe_backward", "moe_device_status", "moe_permute_noalloc",
            "moe_route_replay", "moe_grouped_ffn_ep", "moe_combine_sorted", "moe_router_logits",
            "moe_backward_ep", "moe_grouped_ffn_etp", "moe_etp_reduce", "moe_grouped_ffn_etp_fused")

_vp = ctypes.c_void_p


class Dims(ctypes.Structure):
    _fields_ = [("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32), ("k", ctypes.c_int32),
                ("I", ctypes.c_int32), ("Is", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class Saved(ctypes.Structure):
    _fields_ = [("gu", _vp), ("h", _vp), ("gu_shared", _vp), ("h_shared", _vp)]


class FwdArgs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("x", "w_router", "router_bias", "w_shared_gate", "w_gate_up", "w_down",
                                   "ws_gate_up", "ws_down", "y", "topk_ids", "topk_w", "shared_sig", "logits",
                                   "expert_offsets", "sorted_route", "route_pos", "y_routed", "y_shared")] + \
              [("saved", Saved), ("replay_ids", _vp)]


class BwdArgs(ctypes.Structure):
    _fields_ = [(n, _vp) for n in ("x", "w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up",
                                   "ws_down", "topk_ids", "topk_w", "shared_sig", "expert_offsets",
                                   "sorted_route", "route_pos", "y_routed", "y_shared")] + \
              [("saved", Saved)] + \
              [(n, _vp) for n in ("dy", "dx", "dw_gate_up", "dw_down", "dw_router", "dw_shared_gate",
                                  "dws_gate_up", "dws_down", "dlogit", "dz")]


class MoEError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn}: {STATUS.get(status, status)} ({status_string(status)})")


_lock = threading.Lock()
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded CUDA library.  Raises if it has not been built (no fallback)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                                   "`python -m top_routed_grouped_gb300.build`; there is no CPU fallback")
            L = ctypes.CDLL(LIB_PATH)
            D = ctypes.POINTER(Dims)
            sigs = {
                "moe_workspace_size": ([D, ctypes.c_int], ctypes.c_size_t),
                "moe_status_string": ([ctypes.c_int], ctypes.c_char_p),
                "moe_route": ([D] + [_vp] * 8 + [_vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_route_replay": ([D] + [_vp] * 8 + [_vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_router_logits": ([D, _vp, _vp, _vp, ctypes.c_int32, _vp, _vp, ctypes.c_size_t, _vp],
                                      ctypes.c_int),
                "moe_permute": ([D] + [_vp] * 4 + [_vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_grouped_ffn": ([D] + [_vp] * 9 + [ctypes.POINTER(Saved), _vp, ctypes.c_size_t, _vp],
                                    ctypes.c_int),
                "moe_combine": ([D] + [_vp] * 5 + [_vp], ctypes.c_int),
                "moe_grouped_ffn_ep": ([D, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32] + [_vp] * 9 +
                                       [ctypes.POINTER(Saved), _vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_combine_sorted": ([D] + [_vp] * 6 + [_vp], ctypes.c_int),
                "moe_grouped_ffn_etp": ([D] + [_vp] * 9 + [ctypes.POINTER(Saved), _vp, ctypes.c_size_t, _vp],
                                        ctypes.c_int),
                "moe_etp_reduce": ([D, ctypes.c_int32, _vp, _vp, _vp, _vp, _vp], ctypes.c_int),
                "moe_grouped_ffn_etp_fused": ([D] + [_vp] * 9 + [_vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_forward": ([D, ctypes.POINTER(FwdArgs), _vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_backward": ([D, ctypes.POINTER(BwdArgs), _vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_backward_ep": ([D, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, ctypes.POINTER(BwdArgs), _vp,
                                     _vp, ctypes.c_size_t, _vp], ctypes.c_int),
                "moe_device_status": ([ctypes.c_int, ctypes.POINTER(ctypes.c_int32)], ctypes.c_int),
                "moe_permute_noalloc": ([D] + [_vp] * 4 + [_vp], ctypes.c_int),
            }
            for name, (args, res) in sigs.items():
                fn = getattr(L, name)
                fn.argtypes = args
                fn.restype = res
            _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().moe_status_string(int(status)).decode()


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise MoEError(fn, rc)


def _p(t):
    """Device pointer of a tensor (None -> NULL)."""
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_dims(T, H, E, k, I, Is, dtype) -> Dims:
    import torch
    if isinstance(dtype, torch.dtype):
        dtype = {torch.float32: MOE_F32, torch.bfloat16: MOE_BF16}[dtype]
    return Dims(int(T), int(H), int(E), int(k), int(I), int(Is), int(dtype))


def dims_of(x, w_router, w_gate_up, ws_gate_up, k: int) -> Dims:
    T, H = x.shape
    return make_dims(T, H, w_router.shape[0], k, w_gate_up.shape[1] // 2, ws_gate_up.shape[0] // 2, x.dtype)


# ---------------------------------------------------------------- raw ABI
def moe_workspace_size(d: Dims, op) -> int:
    op = OP[op] if isinstance(op, str) else int(op)
    return int(lib().moe_workspace_size(ctypes.byref(d), op))


def moe_route(d, x, w_router, router_bias, w_shared_gate, topk_ids, topk_w, shared_sig, logits, ws, stream=None):
    _check("moe_route", lib().moe_route(ctypes.byref(d), _p(x), _p(w_router), _p(router_bias), _p(w_shared_gate),
                                        _p(topk_ids), _p(topk_w), _p(shared_sig), _p(logits), _p(ws),
                                        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_router_logits(d, x, w_router, router_bias, exact, logits, ws, stream=None):
    _check("moe_router_logits", lib().moe_router_logits(
        ctypes.byref(d), _p(x), _p(w_router), _p(router_bias), int(exact), _p(logits), _p(ws),
        0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def router_logits(x, w_router, router_bias=None, exact: bool = True, stream=None):
    """Router logits [T, E] float: exact FP32-equivalent (default) or the
    BF16-router ablation (weight rounded once to bf16)."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    d = make_dims(T, H, E, 1, 128, 128, x.dtype)  # k, I, Is unused
    out = torch.empty(T, E, dtype=torch.float32, device=x.device)
    moe_router_logits(d, x, w_router, router_bias, 1 if exact else 0, out, workspace(d, "route", x.device), stream)
    return out


def moe_route_replay(d, x, w_router, router_bias, w_shared_gate, topk_ids, topk_w, shared_sig, logits, ws,
                     stream=None):
    _check("moe_route_replay", lib().moe_route_replay(
        ctypes.byref(d), _p(x), _p(w_router), _p(router_bias), _p(w_shared_gate), _p(topk_ids), _p(topk_w),
        _p(shared_sig), _p(logits), _p(ws), 0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)))


def moe_permute(d, topk_ids, expert_offsets, sorted_route, route_pos, ws, stream=None):
    _check("moe_permute", lib().moe_permute(ctypes.byref(d), _p(topk_ids), _p(expert_offsets), _p(sorted_route),
                                            _p(route_pos), _p(ws), 0 if ws is None else ws.numel(),
                                            _stream(stream)))


def moe_permute_noalloc(d, topk_ids, expert_offsets, sorted_route, route_pos, stream=None):
    """moe_permute without a workspace: for callers that cannot allocate device
    memory (the scratch is a fixed array inside the library; see moe.h)."""
    _check("moe_permute_noalloc", lib().moe_permute_noalloc(ctypes.byref(d), _p(topk_ids), _p(expert_offsets),
                                                            _p(sorted_route), _p(route_pos), _stream(stream)))


def _saved(saved) -> Saved:
    saved = saved or {}
    return Saved(*(_p(saved.get(n)) for n in ("gu", "h", "gu_shared", "h_shared")))


def moe_grouped_ffn(d, x, expert_offsets, sorted_route, w_gate_up, w_down, ws_gate_up, ws_down, y_routed,
                    y_shared, saved, ws, stream=None):
    s = _saved(saved)
    _check("moe_grouped_ffn", lib().moe_grouped_ffn(
        ctypes.byref(d), _p(x), _p(expert_offsets), _p(sorted_route), _p(w_gate_up), _p(w_down), _p(ws_gate_up),
        _p(ws_down), _p(y_routed), _p(y_shared), ctypes.byref(s), _p(ws), 0 if ws is None else ws.numel(),
        _stream(stream)))


def moe_grouped_ffn_ep(d, e_begin, e_end, with_shared, x, expert_offsets, sorted_route, w_gate_up, w_down,
                       ws_gate_up, ws_down, y_sorted, y_shared, saved, ws, stream=None):
    """One rank's part of the expert-partitioned grouped FFN (see moe.h)."""
    sv = _saved(saved)
    _check("moe_grouped_ffn_ep", lib().moe_grouped_ffn_ep(
        ctypes.byref(d), int(e_begin), int(e_end), int(with_shared), _p(x), _p(expert_offsets), _p(sorted_route),
        _p(w_gate_up), _p(w_down), _p(ws_gate_up), _p(ws_down), _p(y_sorted), _p(y_shared), ctypes.byref(sv), _p(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def moe_grouped_ffn_etp(d, x, expert_offsets, sorted_route, w_gate_up, w_down, ws_gate_up, ws_down, yr_partial,
                        ys_partial, saved, ws, stream=None):
    """One rank's part of the expert-tensor-parallel grouped FFN (see moe.h):
    ``d`` carries the rank's slice widths; float partial rows out."""
    sv = _saved(saved)
    _check("moe_grouped_ffn_etp", lib().moe_grouped_ffn_etp(
        ctypes.byref(d), _p(x), _p(expert_offsets), _p(sorted_route), _p(w_gate_up), _p(w_down), _p(ws_gate_up),
        _p(ws_down), _p(yr_partial), _p(ys_partial), ctypes.byref(sv), _p(ws), 0 if ws is None else ws.numel(),
        _stream(stream)))


def moe_grouped_ffn_etp_fused(d, x, expert_offsets, sorted_route, w_gate_up, w_down, ws_gate_up, ws_down,
                              yr_partial, ys_partial, ws, stream=None):
    """moe_grouped_ffn_etp for a 128-feature slice with gate_up and down fused
    (h kept on chip; no saved activations), same partial rows bit for bit."""
    _check("moe_grouped_ffn_etp_fused", lib().moe_grouped_ffn_etp_fused(
        ctypes.byref(d), _p(x), _p(expert_offsets), _p(sorted_route), _p(w_gate_up), _p(w_down), _p(ws_gate_up),
        _p(ws_down), _p(yr_partial), _p(ys_partial), _p(ws), 0 if ws is None else ws.numel(), _stream(stream)))


def moe_etp_reduce(d, yr_parts, ys_parts, y_routed, y_shared, stream=None):
    """Rank-ordered FP32 sum of the partials, one rounding (see moe.h)."""
    n = len(yr_parts)
    if n != len(ys_parts):
        raise ValueError("one routed and one shared partial per rank")
    arr_r = (ctypes.c_void_p * max(n, 1))(*[_p(t) for t in yr_parts])
    arr_s = (ctypes.c_void_p * max(n, 1))(*[_p(t) for t in ys_parts])
    _check("moe_etp_reduce", lib().moe_etp_reduce(ctypes.byref(d), n, arr_r, arr_s, _p(y_routed), _p(y_shared),
                                                  _stream(stream)))


def moe_combine_sorted(d, y_sorted, route_pos, y_shared, topk_w, shared_sig, y, stream=None):
    _check("moe_combine_sorted", lib().moe_combine_sorted(ctypes.byref(d), _p(y_sorted), _p(route_pos), _p(y_shared),
                                                          _p(topk_w), _p(shared_sig), _p(y), _stream(stream)))


def moe_combine(d, y_routed, y_shared, topk_w, shared_sig, y, stream=None):
    _check("moe_combine", lib().moe_combine(ctypes.byref(d), _p(y_routed), _p(y_shared), _p(topk_w),
                                            _p(shared_sig), _p(y), _stream(stream)))


def moe_forward(d, args: dict, ws, stream=None):
    fa = FwdArgs()
    for name, _ in FwdArgs._fields_:
        if name != "saved":
            setattr(fa, name, _p(args.get(name)))  # replay_ids: NULL unless given
    fa.saved = _saved(args.get("saved"))
    _check("moe_forward", lib().moe_forward(ctypes.byref(d), ctypes.byref(fa), _p(ws),
                                            0 if ws is None else ws.numel(), _stream(stream)))


def _bwd_args(args: dict):
    ba = BwdArgs()
    for name, _ in BwdArgs._fields_:
        if name != "saved":
            setattr(ba, name, _p(args.get(name)))
    ba.saved = _saved(args.get("saved"))
    return ba


def moe_backward(d, args: dict, ws, stream=None):
    ba = _bwd_args(args)
    _check("moe_backward", lib().moe_backward(ctypes.byref(d), ctypes.byref(ba), _p(ws),
                                              0 if ws is None else ws.numel(), _stream(stream)))


def moe_backward_ep(d, e_begin, e_end, phase, args: dict, dxr_sorted, ws, stream=None):
    """One rank's part of the expert-partitioned backward (see moe.h): phase 1
    up to the rank's routed input-gradient rows, phase 2 dx, 3 both."""
    ba = _bwd_args(args)
    _check("moe_backward_ep", lib().moe_backward_ep(
        ctypes.byref(d), int(e_begin), int(e_end), int(phase), ctypes.byref(ba), _p(dxr_sorted), _p(ws),
        0 if ws is None else ws.numel(), _stream(stream)))


def moe_device_status(reset: bool = True) -> int:
    """Synchronise and return the device status code (0 = no failed device check)."""
    detail = ctypes.c_int32(0)
    rc = lib().moe_device_status(1 if reset else 0, ctypes.byref(detail))
    if rc not in (0, -5):
        raise MoEError("moe_device_status", rc)
    return int(detail.value)


# ---------------------------------------------------------------- helpers
def workspace(d: Dims, op, device="cuda"):
    import torch
    n = moe_workspace_size(d, op)
    return torch.empty(max(n, 256), dtype=torch.uint8, device=device)


def route(x, w_router, w_shared_gate, k: int, router_bias=None, E: int | None = None, want_logits=False,
          stream=None):
    """Returns dict(topk_ids [T,k] int32, topk_w [T,k] f32, shared_sig [T] f32, logits [T,E] f32 or None)."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    d = make_dims(T, H, E, k, 128, 128, x.dtype)  # I, Is unused by routing
    dev = x.device
    out = {"topk_ids": torch.empty(T, k, dtype=torch.int32, device=dev),
           "topk_w": torch.empty(T, k, dtype=torch.float32, device=dev),
           "shared_sig": torch.empty(T, dtype=torch.float32, device=dev),
           "logits": torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None}
    moe_route(d, x, w_router, router_bias, w_shared_gate, out["topk_ids"], out["topk_w"], out["shared_sig"],
              out["logits"], workspace(d, "route", dev), stream)
    return out


def route_replay(x, w_router, w_shared_gate, topk_ids, router_bias=None, want_logits=False, stream=None):
    """Route weights and shared gate for given expert ids [T,k] (router replay).
    Returns dict(topk_ids (the input), topk_w, shared_sig, logits or None)."""
    import torch
    T, H = x.shape
    k = topk_ids.shape[1]
    E = w_router.shape[0]
    d = make_dims(T, H, E, k, 128, 128, x.dtype)  # I, Is unused by routing
    dev = x.device
    out = {"topk_ids": topk_ids,
           "topk_w": torch.empty(T, k, dtype=torch.float32, device=dev),
           "shared_sig": torch.empty(T, dtype=torch.float32, device=dev),
           "logits": torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None}
    moe_route_replay(d, x, w_router, router_bias, w_shared_gate, topk_ids, out["topk_w"], out["shared_sig"],
                     out["logits"], workspace(d, "route", dev), stream)
    return out


def permute(topk_ids, E: int, stream=None):
    """Returns dict(expert_offsets [E+1], sorted_route [T*k], route_pos [T*k]), all int32."""
    import torch
    T, k = topk_ids.shape
    d = make_dims(T, 256, E, k, 128, 128, MOE_BF16)  # H, I, Is unused by the permutation
    dev = topk_ids.device
    out = {"expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
           "sorted_route": torch.empty(T * k, dtype=torch.int32, device=dev),
           "route_pos": torch.empty(T * k, dtype=torch.int32, device=dev)}
    moe_permute(d, topk_ids, out["expert_offsets"], out["sorted_route"], out["route_pos"],
                workspace(d, "permute", dev), stream)
    return out


def forward(x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, k: int, router_bias=None,
            save_for_backward: bool = False, want_logits: bool = False, replay_ids=None, stream=None, ws=None):
    """Full layer forward through ``moe_forward``.  Returns a dict with ``y`` and every intermediate.
    ``replay_ids`` [T,k] int32: route with these experts instead of the top-k (router replay).
    ``ws``: a caller-owned workspace (allocated here when None)."""
    import torch
    T, H = x.shape
    d = dims_of(x, w_router, w_gate_up, ws_gate_up, k)
    dev, dt = x.device, x.dtype
    R, E, I, Is = T * k, d.E, d.I, d.Is
    out = {
        "y": torch.empty(T, H, dtype=dt, device=dev),
        "topk_ids": torch.empty(T, k, dtype=torch.int32, device=dev),
        "topk_w": torch.empty(T, k, dtype=torch.float32, device=dev),
        "shared_sig": torch.empty(T, dtype=torch.float32, device=dev),
        "logits": torch.empty(T, E, dtype=torch.float32, device=dev) if want_logits else None,
        "expert_offsets": torch.empty(E + 1, dtype=torch.int32, device=dev),
        "sorted_route": torch.empty(R, dtype=torch.int32, device=dev),
        "route_pos": torch.empty(R, dtype=torch.int32, device=dev),
        "y_routed": torch.empty(R, H, dtype=dt, device=dev),
        "y_shared": torch.empty(T, H, dtype=dt, device=dev),
    }
    if save_for_backward:
        out["saved"] = {"gu": torch.empty(R, 2 * I, dtype=dt, device=dev),
                        "h": torch.empty(R, I, dtype=dt, device=dev),
                        "gu_shared": torch.empty(T, 2 * Is, dtype=dt, device=dev),
                        "h_shared": torch.empty(T, Is, dtype=dt, device=dev)}
    args = dict(out, x=x, w_router=w_router, router_bias=router_bias, w_shared_gate=w_shared_gate,
                w_gate_up=w_gate_up, w_down=w_down, ws_gate_up=ws_gate_up, ws_down=ws_down, replay_ids=replay_ids)
    moe_forward(d, args, workspace(d, "forward", dev) if ws is None else ws, stream)
    return out


def backward(fwd: dict, dy, x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, ws=None,
             stream=None):
    """Layer backward through ``moe_backward`` from the dict ``forward(..., save_for_backward=True)``
    returned.  Returns dx, the six weight gradients (float) and dlogit [T,k], dz [T].
    ``ws``: a caller-owned workspace (allocated here when None)."""
    import torch
    T, H = x.shape
    k = fwd["topk_ids"].shape[1]
    d = dims_of(x, w_router, w_gate_up, ws_gate_up, k)
    dev, f32 = x.device, torch.float32
    E, I, Is = d.E, d.I, d.Is
    out = {"dx": torch.empty(T, H, dtype=x.dtype, device=dev),
           "dw_gate_up": torch.empty(E, 2 * I, H, dtype=f32, device=dev),
           "dw_down": torch.empty(E, H, I, dtype=f32, device=dev),
           "dw_router": torch.empty(E, H, dtype=f32, device=dev),
           "dw_shared_gate": torch.empty(H, dtype=f32, device=dev),
           "dws_gate_up": torch.empty(2 * Is, H, dtype=f32, device=dev),
           "dws_down": torch.empty(H, Is, dtype=f32, device=dev),
           "dlogit": torch.empty(T, k, dtype=f32, device=dev),
           "dz": torch.empty(T, dtype=f32, device=dev)}
    args = dict(out, x=x, w_router=w_router, w_shared_gate=w_shared_gate, w_gate_up=w_gate_up, w_down=w_down,
                ws_gate_up=ws_gate_up, ws_down=ws_down, dy=dy, saved=fwd["saved"],
                **{n: fwd[n] for n in ("topk_ids", "topk_w", "shared_sig", "expert_offsets", "sorted_route",
                                       "route_pos", "y_routed", "y_shared")})
    moe_backward(d, args, workspace(d, "backward", dev) if ws is None else ws, stream)
    return out


def __getattr__(name):
    # The torch module lives in layer.py (imported on first use, so that this
    # binding itself does not import torch at load time).
    if name in ("MoELayer", "MoEFunction"):
        from . import layer
        return getattr(layer, name)
    raise AttributeError(name)
