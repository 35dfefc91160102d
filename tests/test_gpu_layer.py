"""MoELayer: the layer as a torch module whose autograd Function calls
moe_forward and moe_backward (#503 commit message, "Backward"; the layer's
boundary wraps the C ABI in an autograd Function on the current stream).

Bars: torch.autograd.grad through the module gives moe_backward's gradients
bit for bit (dx and the FP32 router gradient unchanged, the bf16 weights'
FP32 gradients rounded once to bf16 by autograd's cast to the parameter
dtype); y equals moe_forward's; dx of a token is bitwise independent of the
batch it runs in.
"""
import pytest
import torch

import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build
from top_routed_grouped_gb300 import inputs as I

from _util import bits, full_dy, full_weights, full_x

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")


@pytest.fixture(scope="module")
def layer():
    build.build()
    W = full_weights()
    m = moe.MoELayer(2048, 512, 10, 512, 512, dtype=torch.bfloat16, device="cuda")
    with torch.no_grad():
        for n in WKEYS:
            getattr(m, n).copy_(W[n])
    return m


def test_autograd_equals_moe_backward(layer):
    T = 1024
    x = full_x(T).cuda().requires_grad_(True)
    dy = full_dy(T).cuda()
    y = layer(x)
    grads = torch.autograd.grad(y, [x, *layer.weights()], grad_outputs=dy)
    W = [w.detach() for w in layer.weights()]
    f = moe.forward(x.detach(), *W, 10, save_for_backward=True)
    g = moe.backward(f, dy, x.detach(), *W)
    assert torch.equal(bits(y.detach()), bits(f["y"]))
    assert torch.equal(layer.last_routes["topk_ids"], f["topk_ids"])
    assert torch.equal(bits(grads[0]), bits(g["dx"]))
    for got, name, p in zip(grads[1:], ("dw_router", "dw_shared_gate", "dw_gate_up", "dw_down", "dws_gate_up",
                                        "dws_down"), W):
        assert got.dtype == p.dtype, name
        assert torch.equal(bits(got), bits(g[name].to(p.dtype))), name
    assert moe.moe_device_status(reset=True) == 0


def test_module_backward_accumulates_into_parameters(layer):
    """loss.backward() fills .grad of every parameter and of x; a second
    step accumulates (autograd's rule), the library itself overwrites."""
    T = 64
    x = full_x(T).cuda().requires_grad_(True)
    dy = full_dy(T).cuda()
    layer.zero_grad(set_to_none=True)
    (layer(x).float() * dy.float()).sum().backward()
    first = {n: getattr(layer, n).grad.clone() for n in WKEYS}
    assert all(torch.isfinite(v.float()).all() for v in first.values())
    assert x.grad is not None and x.grad.shape == x.shape
    (layer(x).float() * dy.float()).sum().backward()
    for n in WKEYS:
        # bf16 accumulation of two equal gradients doubles them exactly
        assert torch.equal(getattr(layer, n).grad, first[n] * 2), n


def test_module_dx_is_batch_invariant(layer):
    T = 256
    x = full_x(T).cuda()
    dy = full_dy(T).cuda()
    xf = x.clone().requires_grad_(True)
    dx_full, = torch.autograd.grad(layer(xf), [xf], grad_outputs=dy)
    perm = I.shuffled_order(T).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(T, device="cuda")
    for b in (1, 7, 256):
        parts = []
        for lo, hi in I.ragged_batches(T, b):
            sel = perm[lo:hi]
            xs = x[sel].clone().requires_grad_(True)
            dx, = torch.autograd.grad(layer(xs), [xs], grad_outputs=dy[sel])
            parts.append(dx)
        assert torch.equal(bits(torch.cat(parts)[inv]), bits(dx_full)), f"batch {b}"
    assert moe.moe_device_status(reset=True) == 0


def test_micro_batches_forwarded_before_backward(layer):
    """Gradient accumulation: two micro-batches of different sizes run their
    forwards first (the second one regrows the layer's workspace pair), then
    one backward over both.  The saved activations are per call, so the
    gradients equal the sum of the two calls' moe_backward results, and dx of
    each micro-batch equals its own moe_backward dx bit for bit."""
    layer._ws = None
    x1 = full_x(64).cuda().requires_grad_(True)
    x2 = full_x(1024)[64:1024].cuda().requires_grad_(True)
    dy1, dy2 = full_dy(64).cuda(), full_dy(1024)[64:1024].cuda()
    y1 = layer(x1)
    y2 = layer(x2)
    grads = torch.autograd.grad([y1, y2], [x1, x2, *layer.weights()], grad_outputs=[dy1, dy2])
    W = [w.detach() for w in layer.weights()]
    g1 = moe.backward(moe.forward(x1.detach(), *W, 10, save_for_backward=True), dy1, x1.detach(), *W)
    g2 = moe.backward(moe.forward(x2.detach(), *W, 10, save_for_backward=True), dy2, x2.detach(), *W)
    assert torch.equal(bits(grads[0]), bits(g1["dx"]))
    assert torch.equal(bits(grads[1]), bits(g2["dx"]))
    for got, name, p in zip(grads[2:], ("dw_router", "dw_shared_gate", "dw_gate_up", "dw_down", "dws_gate_up",
                                        "dws_down"), W):
        # autograd sums the two per-call gradients after casting each to the parameter dtype
        want = g1[name].to(p.dtype) + g2[name].to(p.dtype)
        assert torch.equal(bits(got), bits(want)), name
    assert moe.moe_device_status(reset=True) == 0


def test_f32_module_matches_library():
    """An FP32 module: the weight gradients reach the parameters unrounded,
    equal to moe_backward's FP32 outputs bit for bit."""
    build.build()
    cfg = I.CONFIGS["tiny_f32"]
    c = I.make_inputs(cfg, with_dy=True)
    m = moe.MoELayer(cfg.H, cfg.E, cfg.k, cfg.I, cfg.Is, dtype=torch.float32, device="cuda")
    with torch.no_grad():
        for n in WKEYS:
            getattr(m, n).copy_(c[n])
    x = c["x"].cuda().requires_grad_(True)
    dy = c["dy"].cuda()
    grads = torch.autograd.grad(m(x), [x, *m.weights()], grad_outputs=dy)
    W = [w.detach() for w in m.weights()]
    g = moe.backward(moe.forward(x.detach(), *W, cfg.k, save_for_backward=True), dy, x.detach(), *W)
    assert torch.equal(bits(grads[0]), bits(g["dx"]))
    for got, name in zip(grads[1:], ("dw_router", "dw_shared_gate", "dw_gate_up", "dw_down", "dws_gate_up",
                                     "dws_down")):
        assert got.dtype == torch.float32 and torch.equal(bits(got), bits(g[name])), name
    assert moe.moe_device_status(reset=True) == 0
