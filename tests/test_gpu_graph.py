"""moe_forward and moe_backward captured into a CUDA graph.

moe_forward launches on the caller's stream and, above 2048 tokens (bf16),
on a second stream of the library that forks from the caller's stream and
joins back into it through events: after the router launch while the routed
GEMMs average fewer than 256 routes per expert, at the call otherwise.
Under stream capture the second stream joins the capture through those
events, so a captured forward replays the eager call bit for bit, on its
captured inputs and on new values written into the same buffers.  The
backward (one stream) is captured the same way.  Sizes: T = 1024 (one
stream), 8192 (fork after the router launch), 16384 with skewed routing
(fork at the call).
"""
import pytest
import torch

import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build
from top_routed_grouped_gb300 import inputs as I

from _util import bits, full_dy, full_weights, full_x

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")
FWD_OUT = ("y", "topk_ids", "topk_w", "shared_sig", "expert_offsets", "sorted_route", "route_pos", "y_routed",
           "y_shared")


def _same(a, b):
    return torch.equal(bits(a), bits(b)) if a.is_floating_point() else torch.equal(a, b)


@pytest.mark.parametrize("T,zipf", [(1024, False), (8192, False), (16384, True)])
def test_forward_graph_replay_is_bitwise(T, zipf):
    build.build()
    W = [v.cuda() for v in (full_weights()[n] for n in WKEYS)]
    x = full_x(T).cuda()
    x_new = full_x(2 * T)[T:].cuda()  # other token values, same shapes
    bias = I.zipf_bias(512).cuda() if zipf else None
    d = moe.dims_of(x, W[0], W[2], W[4], 10)
    ws = moe.workspace(d, "forward")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        ref = moe.forward(x, *W, 10, router_bias=bias, ws=ws)  # eager: the library's stream, kernel attributes
        ref_new = moe.forward(x_new, *W, 10, router_bias=bias, ws=ws)
    torch.cuda.synchronize()
    xin = x.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out = moe.forward(xin, *W, 10, router_bias=bias, ws=ws)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for key in FWD_OUT:
        assert _same(out[key], ref[key]), key
    xin.copy_(x_new)
    g.replay()
    torch.cuda.synchronize()
    for key in FWD_OUT:
        assert _same(out[key], ref_new[key]), key
    assert moe.moe_device_status(reset=True) == 0


def test_backward_graph_replay_is_bitwise():
    build.build()
    T = 1024
    W = [v.cuda() for v in (full_weights()[n] for n in WKEYS)]
    x = full_x(T).cuda()
    dy = full_dy(T).cuda()
    d = moe.dims_of(x, W[0], W[2], W[4], 10)
    wsb = moe.workspace(d, "backward")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        f = moe.forward(x, *W, 10, save_for_backward=True)
        ref = moe.backward(f, dy, x, *W, ws=wsb)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        out = moe.backward(f, dy, x, *W, ws=wsb)
    torch.cuda.synchronize()
    g.replay()
    torch.cuda.synchronize()
    for key, v in ref.items():
        assert _same(out[key], v), key
    assert moe.moe_device_status(reset=True) == 0
