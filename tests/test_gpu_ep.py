"""Expert partition (EP), simulated on one GPU.

RL-Kernel PR #557 "What": experts in contiguous ranges across ranks,
replicated routing, each rank runs only its experts' segments, one byte-copy
all_gather of the routed rows, a local ordered combine; a route slot owned by
no rank fails closed.  Bar: the layer output of every split equals the
single-launch moe_forward bit for bit (every row is computed by the same
arithmetic whichever call computes it; the combine order is unchanged).
"""
import numpy as np
import pytest
import torch

import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build, ep
from top_routed_grouped_gb300 import inputs as I

from _util import bits, full_weights, full_x, to_dev

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    moe.lib()
    moe.moe_device_status(reset=True)


def reference(d, k, bias=None):
    return moe.forward(d["x"], *[d[n] for n in WKEYS], k, router_bias=bias)


@pytest.mark.parametrize("world", [2, 3, 4])
def test_bf16_ep_split_equals_single_launch(world):
    W = to_dev(full_weights())
    x = full_x(1024).cuda()
    d = dict(W, x=x)
    ref = reference(d, 10)
    out = ep.forward_simulated(x, *[W[n] for n in WKEYS], 10, world)
    assert torch.equal(bits(out["y"]), bits(ref["y"]))
    # the sorted rows are the route-order rows permuted
    pos = out["permute"]["route_pos"].long()
    assert torch.equal(bits(out["y_sorted"][pos]), bits(ref["y_routed"]))
    assert moe.moe_device_status(reset=True) == 0


def test_bf16_ep_uneven_ranges_and_empty_rank():
    """Ranges of very different sizes, one of them empty, with Zipf-skewed routing."""
    W = to_dev(full_weights())
    x = full_x(2048).cuda()
    bias = I.zipf_bias(512).cuda()
    ranges = [(0, 5), (5, 5), (5, 300), (300, 512)]
    out = ep.forward_simulated(x, *[W[n] for n in WKEYS], 10, 4, ranges=ranges, router_bias=bias)
    ref = reference(dict(W, x=x), 10, bias)
    assert torch.equal(bits(out["y"]), bits(ref["y"]))


def test_f32_ep_split_equals_single_launch():
    cfg = I.CONFIGS["tiny_f32"]
    d = to_dev(I.make_inputs(cfg))
    ref = reference(d, cfg.k)
    out = ep.forward_simulated(d["x"], *[d[n] for n in WKEYS], cfg.k, 3)
    assert torch.equal(bits(out["y"]), bits(ref["y"]))


def test_ep_partition_fails_closed():
    with pytest.raises(ValueError):
        ep.check_partition([(0, 200), (256, 512)], 512)  # experts 200..255 unowned
    with pytest.raises(ValueError):
        ep.check_partition([(0, 300), (256, 512)], 512)  # overlap
    with pytest.raises(ValueError):
        ep.check_partition([(0, 256), (256, 500)], 512)  # tail unowned
    W = to_dev(full_weights())
    x = full_x(16).cuda()
    with pytest.raises(ValueError):
        ep.forward_simulated(x, *[W[n] for n in WKEYS], 10, 2, ranges=[(0, 100), (200, 512)])


def test_ep_api_rejects_bad_ranges():
    W = to_dev(full_weights())
    x = full_x(16).cuda()
    d = moe.dims_of(x, W["w_router"], W["w_gate_up"], W["ws_gate_up"], 10)
    r = moe.route(x, W["w_router"], W["w_shared_gate"], 10)
    pm = moe.permute(r["topk_ids"], 512)
    y_sorted = torch.empty(160, 2048, dtype=torch.bfloat16, device="cuda")
    ws = moe.workspace(d, "grouped_ffn")
    for b, e in [(-1, 4), (10, 5), (0, 513)]:
        with pytest.raises(moe.MoEError) as err:
            moe.moe_grouped_ffn_ep(d, b, e, 0, x, pm["expert_offsets"], pm["sorted_route"], W["w_gate_up"],
                                   W["w_down"], None, None, y_sorted, None, None, ws)
        assert err.value.status == -1
