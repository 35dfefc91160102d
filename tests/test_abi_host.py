"""Host-side checks of the C ABI (no GPU work): the library builds, loads and
exports every function include/moe.h declares; workspace sizes; fail-closed
argument validation (RL-Kernel PR #557 "What": a route slot owned by no rank
fails closed; here: bad arguments return an error and launch nothing)."""
import ctypes
import os
import re

import pytest

import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    build.build()
    return moe.lib()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "moe.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_]+)\s*\(", src)))


def test_header_declares_expected_entry_points():
    assert set(declared_functions()) == set(moe.EXPORTED)


def test_library_exports_every_declared_symbol(L):
    for name in declared_functions():
        assert hasattr(L, name), name
    out = os.popen(f"nm -D --defined-only {moe.LIB_PATH}").read()
    exported = set(re.findall(r" T (moe_\w+)", out))
    assert exported == set(declared_functions()), exported


def test_status_strings(L):
    for code in (0, -1, -2, -3, -4, -5):
        assert moe.status_string(code) != "unknown status"
    assert moe.status_string(7) == "unknown status"


def dims(**kw):
    base = dict(T=1024, H=2048, E=512, k=10, I=512, Is=512, dtype=moe.MOE_BF16)
    base.update(kw)
    return moe.make_dims(**base)


def test_workspace_sizes(L):
    d = dims()
    for op in moe.OP:
        n = moe.moe_workspace_size(d, op)
        assert n % 256 == 0
    assert moe.moe_workspace_size(d, "combine") == 0
    assert moe.moe_workspace_size(d, "forward") > moe.moe_workspace_size(d, "grouped_ffn")
    # invalid dims -> 0
    assert moe.moe_workspace_size(dims(k=17, E=32), "route") == 0
    assert moe.moe_workspace_size(dims(H=100), "route") == 0
    # monotone in T
    assert moe.moe_workspace_size(dims(T=2048), "forward") > moe.moe_workspace_size(d, "forward")


def call_route(d, ptr=16, ws_bytes=1 << 40):
    p = ctypes.c_void_p(ptr)
    return moe.lib().moe_route(ctypes.byref(d), p, p, None, p, p, p, p, None, p, ws_bytes, None)


@pytest.mark.parametrize("kw,expect", [
    (dict(k=0), -1), (dict(k=17, E=32), -1), (dict(k=5, E=4), -1), (dict(T=-1), -1), (dict(dtype=7), -1),
    (dict(H=0), -1), (dict(E=2048), -2), (dict(H=2000), -2), (dict(H=1920), -2), (dict(I=100), -2),
    (dict(I=192), -2), (dict(Is=64), -2),
    (dict(dtype=moe.MOE_F32, H=130), -2), (dict(T=300_000_000), -2),
])
def test_route_rejects_bad_dims(L, kw, expect):
    assert call_route(dims(**kw)) == expect


def test_route_rejects_null_and_misaligned(L):
    d = dims()
    assert call_route(d, ptr=0) == -1
    assert call_route(d, ptr=8) == -1  # not 16-byte aligned


def test_route_rejects_small_workspace(L):
    d = dims()
    need = moe.moe_workspace_size(d, "route")
    assert call_route(d, ws_bytes=need - 1) == -3


def test_null_dims_rejected(L):
    p = ctypes.c_void_p(16)
    assert L.moe_combine(None, p, p, p, p, p, None) == -1
    assert L.moe_forward(None, None, None, 0, None) == -1


def test_combine_zero_tokens_is_noop(L):
    d = dims(T=0)
    assert L.moe_combine(ctypes.byref(d), None, None, None, None, None, None) == 0


def test_permute_small_workspace(L):
    d = dims()
    p = ctypes.c_void_p(16)
    need = moe.moe_workspace_size(d, "permute")
    assert L.moe_permute(ctypes.byref(d), p, p, p, p, p, need - 256, None) == -3


def test_moe_layer_parameters_on_cpu():
    """MoELayer's parameters follow the library's layout (no GPU needed to
    construct it on the CPU)."""
    import torch
    import top_routed_grouped_gb300 as moe
    m = moe.MoELayer(256, 16, 4, 128, 128, dtype=torch.bfloat16, device="cpu")
    shapes = {n: (tuple(p.shape), p.dtype) for n, p in m.named_parameters()}
    assert shapes == {"w_router": ((16, 256), torch.float32), "w_shared_gate": ((256,), torch.bfloat16),
                      "w_gate_up": ((16, 256, 256), torch.bfloat16), "w_down": ((16, 256, 128), torch.bfloat16),
                      "ws_gate_up": ((256, 256), torch.bfloat16), "ws_down": ((256, 128), torch.bfloat16)}
    assert m.top_k == 4 and m.router_bias is None
