"""Expert-partitioned backward (moe_backward_ep), simulated on one GPU.

RL-Kernel PR #557 "What": experts in contiguous ranges across ranks, the
per-route input gradients written into one dense buffer and summed in
ascending expert order (#503 commit message "Backward"); here each rank
computes its experts' weight gradients (local) and its block of dXr rows,
one byte-copy exchange assembles dXr, and dx is local.  Bars: every rank's
dx and replicated gradients, and the expert weight gradients assembled from
the ranks' local arrays, equal the single-launch moe_backward bit for bit
(each value is computed by the same kernel with the same reduction order
whichever call computes it); one shape per GEMM path is also checked
against the FP64 oracle directly.
"""
import numpy as np
import pytest
import torch

import oracle
import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build, ep
from top_routed_grouped_gb300 import inputs as I

from _util import assert_grad_close, bits, full_dy, full_weights, full_x, small_layer, to_dev

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")
REPLICATED = ("dx", "dw_router", "dw_shared_gate", "dws_gate_up", "dws_down", "dlogit", "dz")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    moe.lib()
    moe.moe_device_status(reset=True)


def single_launch(d, dy, k, bias=None):
    args = [d[n] for n in WKEYS]
    f = moe.forward(d["x"], *args, k, router_bias=bias, save_for_backward=True)
    return f, moe.backward(f, dy, d["x"], *args)


def split(d, dy, k, world, ranges=None, bias=None):
    args = [d[n] for n in WKEYS]
    f = ep.forward_simulated(d["x"], *args, k, world, ranges=ranges, router_bias=bias, save_for_backward=True)
    return f, ep.backward_simulated(f, dy, d["x"], *args)


def assert_split_equals_single(d, dy, k, world, ranges=None, bias=None):
    f1, g1 = single_launch(d, dy, k, bias)
    fe, ge = split(d, dy, k, world, ranges, bias)
    assert torch.equal(bits(fe["y"]), bits(f1["y"]))
    assert torch.equal(bits(ge["dw_gate_up"]), bits(g1["dw_gate_up"]))
    assert torch.equal(bits(ge["dw_down"]), bits(g1["dw_down"]))
    for rank, out in enumerate(ge["ranks"]):
        for key in REPLICATED:
            assert torch.equal(bits(out[key]), bits(g1[key])), f"rank {rank}: {key}"
    assert moe.moe_device_status(reset=True) == 0
    return fe, ge


@pytest.mark.parametrize("world", [2, 4])
def test_bf16_ep_backward_equals_single_launch(world):
    W = to_dev(full_weights())
    T = 1024
    d = dict(W, x=full_x(T).cuda())
    assert_split_equals_single(d, full_dy(T).cuda(), 10, world)


def test_bf16_ep_backward_uneven_ranges_and_empty_rank():
    """Ranges of very different sizes, one empty, Zipf-skewed routing."""
    W = to_dev(full_weights())
    T = 2048
    d = dict(W, x=full_x(T).cuda())
    bias = I.zipf_bias(512).cuda()
    assert_split_equals_single(d, full_dy(T).cuda(), 10, 4, ranges=[(0, 5), (5, 5), (5, 300), (300, 512)],
                               bias=bias)


def test_f32_ep_backward_equals_single_launch():
    cfg = I.CONFIGS["tiny_f32"]
    d = to_dev(I.make_inputs(cfg, with_dy=True))
    assert_split_equals_single(d, d["dy"], cfg.k, 3)


@pytest.mark.parametrize("shape", [(600, 256, 4, 2, 256, 512), (77, 256, 16, 4, 128, 384)],
                         ids=["tensor-core", "cuda-core"])
def test_bf16_ep_backward_small_shapes_against_oracle(shape):
    """Both bf16 GEMM paths under a split, against the single launch and
    against the oracle's full backward (expert weight gradients from the
    ranks' local arrays, dx from every rank)."""
    T, H, E, k, I_, Is = shape
    c = small_layer(T, H, E, k, I_, Is)
    d = to_dev(c)
    fe, ge = assert_split_equals_single(d, d["dy"], k, 2)
    r = fe["route"]
    ids = r["topk_ids"].cpu().numpy()
    w = r["topk_w"].double().cpu().numpy()
    sig = r["shared_sig"].double().cpu().numpy()
    ref = oracle.layer_backward(c["x"], ids, w, sig, *[c[n] for n in WKEYS], c["dy"])
    assert_grad_close(ge["dw_gate_up"], ref["dw_gate_up"], "dw_gate_up")
    assert_grad_close(ge["dw_down"], ref["dw_down"], "dw_down")
    for out in ge["ranks"]:
        assert_grad_close(out["dx"], ref["dx"], "dx")


def test_ep_backward_dxr_blocks_are_disjoint():
    """Phase 1 of a rank writes exactly its block of dXr rows: rows outside
    [offsets[e_begin], offsets[e_end]) keep their previous contents."""
    cfg = I.CONFIGS["tiny_f32"]
    d = to_dev(I.make_inputs(cfg, with_dy=True))
    args = [d[n] for n in WKEYS]
    f = ep.forward_simulated(d["x"], *args, cfg.k, 2, save_for_backward=True)
    dm = moe.dims_of(d["x"], d["w_router"], d["w_gate_up"], d["ws_gate_up"], cfg.k)
    (b, e), _ = f["ranges"]
    off = f["permute"]["expert_offsets"].cpu().numpy()
    r0, r1 = ep.rank_rows(off, (b, e))
    R, H, E = cfg.T * cfg.k, cfg.H, cfg.E
    dxr = torch.full((R, H), float("nan"), device="cuda")
    f32 = torch.float32
    out = {"dx": torch.empty_like(d["x"]), "dw_router": torch.empty(E, H, dtype=f32, device="cuda"),
           "dw_shared_gate": torch.empty(H, dtype=f32, device="cuda"),
           "dws_gate_up": torch.empty_like(d["ws_gate_up"], dtype=f32),
           "dws_down": torch.empty_like(d["ws_down"], dtype=f32),
           "dw_gate_up": torch.empty_like(d["w_gate_up"][b:e], dtype=f32),
           "dw_down": torch.empty_like(d["w_down"][b:e], dtype=f32)}
    r, pm = f["route"], f["permute"]
    a = dict(out, x=d["x"], w_router=d["w_router"], w_shared_gate=d["w_shared_gate"], w_gate_up=d["w_gate_up"][b:e],
             w_down=d["w_down"][b:e], ws_gate_up=d["ws_gate_up"], ws_down=d["ws_down"], dy=d["dy"],
             saved=f["saved"], topk_ids=r["topk_ids"], topk_w=r["topk_w"], shared_sig=r["shared_sig"],
             expert_offsets=pm["expert_offsets"], sorted_route=pm["sorted_route"], route_pos=pm["route_pos"],
             y_routed=f["y_sorted"], y_shared=f["y_shared"])
    moe.moe_backward_ep(dm, b, e, 1, a, dxr, moe.workspace(dm, "backward", "cuda"))
    got = dxr.cpu()
    assert r1 > r0
    assert not torch.isnan(got[r0:r1]).any()
    assert torch.isnan(got[:r0]).all() and torch.isnan(got[r1:]).all()
    assert moe.moe_device_status(reset=True) == 0


def test_ep_backward_rejects_bad_range_and_phase():
    cfg = I.CONFIGS["tiny_f32"]
    d = to_dev(I.make_inputs(cfg, with_dy=True))
    dm = moe.dims_of(d["x"], d["w_router"], d["w_gate_up"], d["ws_gate_up"], cfg.k)
    dxr = torch.empty(cfg.T * cfg.k, cfg.H, device="cuda")
    ws = moe.workspace(dm, "backward", "cuda")
    for b, e, phase in [(4, 2, 1), (0, cfg.E + 1, 1), (-1, 3, 1), (0, cfg.E, 0), (0, cfg.E, 4)]:
        with pytest.raises(moe.MoEError):
            moe.moe_backward_ep(dm, b, e, phase, {}, dxr, ws)
    with pytest.raises(moe.MoEError):  # dXr buffer missing
        moe.moe_backward_ep(dm, 0, cfg.E, 1, {}, None, ws)
