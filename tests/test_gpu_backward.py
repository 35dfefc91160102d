"""GPU parity of the backward against the FP64 oracle, through the C ABI.

RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503 commit
message "Backward": per-expert weight gradients, per-route input gradients
summed in ascending expert order; "Results (4 x H100)", footnote 1: every
reduction in a fixed order.  Bars: the layer's tolerances, with the max-abs
bar relative to max(1, max|ref|) for gradients (tests/_util.py); dx and the
logit / gate gradients of a token bitwise independent of the batch; weight
gradients bitwise repeatable.
"""
import numpy as np
import pytest
import torch

import oracle
import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build
from top_routed_grouped_gb300 import inputs as I

from _util import (assert_bf16_close, assert_grad_close, bits, full_dy, full_weights, full_x, oracle_bwd_rows,
                   oracle_routes, small_layer, to_dev)

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    moe.lib()
    moe.moe_device_status(reset=True)


def fwd_bwd(d, dy, k, bias=None):
    args = [d[n] for n in WKEYS]
    f = moe.forward(d["x"], *args, k, router_bias=bias, save_for_backward=True, want_logits=True)
    g = moe.backward(f, dy, d["x"], *args)
    return f, g


def checked_routes(f, x, W, bias, k):
    """Oracle routes (near-tie rule) after checking the GPU's against them."""
    ids, w, near, _ = oracle_routes(x, W["w_router"], bias, k, f["logits"].double().cpu().numpy())
    np.testing.assert_array_equal(f["topk_ids"].cpu().numpy(), ids)
    sig = oracle.shared_gate(x, W["w_shared_gate"])
    return ids, w, sig


def dz_of(dsig, sig):
    """Gradient of the gate pre-activation from that of sigmoid's output."""
    return dsig * sig * (1.0 - sig)


def test_tiny_f32_full_parity():
    cfg = I.CONFIGS["tiny_f32"]
    c = I.make_inputs(cfg, with_dy=True)
    d = to_dev(c)
    f, g = fwd_bwd(d, d["dy"], cfg.k)
    ids, w, sig = checked_routes(f, c["x"], c, None, cfg.k)
    ref = oracle.layer_backward(c["x"], ids, w, sig, *[c[n] for n in WKEYS], c["dy"])
    for key in ("dx", "dw_gate_up", "dw_down", "dws_gate_up", "dws_down", "dw_router", "dw_shared_gate",
                "dlogit"):
        assert_grad_close(g[key], ref[key], key, f32=True)
    assert_grad_close(g["dz"], dz_of(ref["dsig"], sig), "dz", f32=True)
    assert moe.moe_device_status(reset=True) == 0


def expert_chunks(E, n):
    return [(e0, min(E, e0 + n)) for e0 in range(0, E, n)]


@pytest.mark.parametrize("T", [37, 300])
def test_bf16_small_batches_full_parity(T):
    """Every gradient of the 512-expert layer (expert weight gradients in
    chunks of experts, all of them covered)."""
    W = full_weights()
    x, dy = full_x(4096)[:T].clone(), full_dy(4096)[:T].clone()
    d = to_dev(dict(W, x=x))
    f, g = fwd_bwd(d, dy.cuda(), 10)
    ids, w, sig = checked_routes(f, x, W, None, 10)
    dx, dw, dl, ds = oracle_bwd_rows(x, ids, w, sig, dy, W)
    assert_grad_close(g["dx"], dx, "dx")
    assert_grad_close(g["dlogit"], dl, "dlogit")
    assert_grad_close(g["dz"], dz_of(ds, sig), "dz")
    dwr, dwsg = oracle.backward_router(x, ids, dl, sig, ds, 512)
    assert_grad_close(g["dw_router"], dwr, "dw_router")
    assert_grad_close(g["dw_shared_gate"], dwsg, "dw_shared_gate")
    dwsgu, dwsdn = oracle.backward_shared_weights(x, sig, dy, W["ws_gate_up"], W["ws_down"])
    assert_grad_close(g["dws_gate_up"], dwsgu, "dws_gate_up")
    assert_grad_close(g["dws_down"], dwsdn, "dws_down")
    loads = np.bincount(ids.reshape(-1), minlength=512)
    chunks = expert_chunks(512, 32) if T <= 37 else [(e, e + 1) for e in
                                                     [int(np.argmax(loads)), int(np.argmin(loads)), 0, 511]]
    for e0, e1 in chunks:
        dwgu, dwdn = oracle.backward_expert_weights(x, ids, w, dy, W["w_gate_up"], W["w_down"], e0, e1)
        assert_grad_close(g["dw_gate_up"][e0:e1], dwgu, f"dw_gate_up[{e0}:{e1}]")
        assert_grad_close(g["dw_down"][e0:e1], dwdn, f"dw_down[{e0}:{e1}]")
    assert moe.moe_device_status(reset=True) == 0


def test_bf16_t4096_sampled():
    """The forward+backward workload at full size: the input, logit and gate
    gradients of 512 tokens (every token of the largest and of the smallest
    expert segment, the rest drawn at random) against the per-token oracle,
    the weight gradients of the largest, smallest and two more experts, and
    the router and gate weight gradients against the oracle's reduction of
    the GPU's (separately checked) logit and gate gradients."""
    W = full_weights()
    T = 4096
    x, dy = full_x(T), full_dy(T)
    d = to_dev(dict(W, x=x))
    f, g = fwd_bwd(d, dy.cuda(), 10)
    ids, w, sig = checked_routes(f, x, W, None, 10)
    rng = np.random.default_rng(5)
    loads = np.bincount(ids.reshape(-1), minlength=512)
    seg_tokens = np.flatnonzero((ids == int(np.argmax(loads))).any(1) | (ids == int(np.argmin(loads))).any(1))
    rest = np.setdiff1d(np.arange(T), seg_tokens)
    sample = np.unique(np.concatenate([[0, T - 1], seg_tokens,
                                       rng.choice(rest, 510 - len(seg_tokens), replace=False)]))
    assert len(sample) >= 500
    dx, dw, dl, ds = oracle_bwd_rows(x[sample], ids[sample], w[sample], sig[sample], dy[sample], W)
    st = torch.as_tensor(sample, device="cuda")
    assert_grad_close(g["dx"][st], dx, "dx sampled")
    assert_grad_close(g["dlogit"][st], dl, "dlogit sampled")
    assert_grad_close(g["dz"][st], dz_of(ds, sig[sample]), "dz sampled")
    # reductions over all routes, fed the GPU's per-route gradients (sig = 1/2
    # makes the oracle's dz equal to dsig / 4, exactly)
    gdl = g["dlogit"].double().cpu().numpy()
    gdz = g["dz"].double().cpu().numpy()
    dwr, dwsg = oracle.backward_router(x, ids, gdl, np.full(T, 0.5), 4.0 * gdz, 512)
    assert_grad_close(g["dw_router"], dwr, "dw_router")
    assert_grad_close(g["dw_shared_gate"], dwsg, "dw_shared_gate")
    for e in sorted({int(np.argmax(loads)), int(np.argmin(loads)), 0, 511}):
        dwgu, dwdn = oracle.backward_expert_weights(x, ids, w, dy, W["w_gate_up"], W["w_down"], e, e + 1)
        assert_grad_close(g["dw_gate_up"][e:e + 1], dwgu, f"dw_gate_up[{e}] ({loads[e]} routes)")
        assert_grad_close(g["dw_down"][e:e + 1], dwdn, f"dw_down[{e}]")
    assert moe.moe_device_status(reset=True) == 0


def test_backward_batch_invariance_and_repeatability():
    """dx, dlogit and dz rows of a shuffled 256-token batch, run in chunks of
    1, 7 and 256, equal the full run bit for bit; weight gradients repeat
    bit for bit."""
    W = to_dev(full_weights())
    T = 256
    x, dy = full_x(T).cuda(), full_dy(T).cuda()
    f, full = fwd_bwd(dict(W, x=x), dy, 10)
    perm = I.shuffled_order(T).cuda()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(T, device="cuda")
    for b in (1, 7, 256):
        parts = {"dx": [], "dlogit": [], "dz": []}
        for lo, hi in I.ragged_batches(T, b):
            sel = perm[lo:hi]
            _, g = fwd_bwd(dict(W, x=x[sel]), dy[sel], 10)
            for key in parts:
                parts[key].append(g[key])
        for key, v in parts.items():
            assert torch.equal(bits(torch.cat(v)[inv]), bits(full[key])), f"batch {b}: {key} differs"
    _, again = fwd_bwd(dict(W, x=x), dy, 10)
    for key in ("dx", "dw_gate_up", "dw_down", "dws_gate_up", "dws_down", "dw_router", "dw_shared_gate"):
        assert torch.equal(bits(again[key]), bits(full[key])), key


def test_backward_zero_tokens_zero_fills():
    W = to_dev(full_weights())
    x = torch.empty(0, 2048, dtype=torch.bfloat16, device="cuda")
    args = [W[n] for n in WKEYS]
    f = moe.forward(x, *args, 10, save_for_backward=True)
    g = moe.backward(f, torch.empty_like(x), x, *args)
    for key in ("dw_router", "dw_shared_gate", "dws_down"):
        assert torch.count_nonzero(g[key]) == 0, key
    assert torch.count_nonzero(g["dw_down"][:3]) == 0


def test_backward_rejects_missing_saved_and_small_workspace():
    W = to_dev(full_weights())
    x, dy = full_x(16).cuda(), full_dy(16).cuda()
    args = [W[n] for n in WKEYS]
    f = moe.forward(x, *args, 10, save_for_backward=True)
    f2 = dict(f, saved=dict(f["saved"], h=None))
    with pytest.raises(moe.MoEError) as e:
        moe.backward(f2, dy, x, *args)
    assert e.value.status == -1
    d = moe.dims_of(x, W["w_router"], W["w_gate_up"], W["ws_gate_up"], 10)
    need = moe.moe_workspace_size(d, "backward")
    with pytest.raises(moe.MoEError) as e:
        moe.backward(f, dy, x, *args, ws=torch.empty(need - 256, dtype=torch.uint8, device="cuda"))
    assert e.value.status == -3
    g = moe.backward(f, dy, x, *args, ws=torch.empty(need, dtype=torch.uint8, device="cuda"))
    assert torch.isfinite(g["dx"].float()).all()


def test_bf16_skewed_routing_t4096():
    """Zipf-biased routing (64 experts with no routes, the largest segment far
    above the mean): zero gradients for empty experts, long K loops for the
    large ones, sampled tokens against the oracle."""
    W = full_weights()
    T = 4096
    x, dy = full_x(T), full_dy(T)
    bias = I.zipf_bias(512)
    d = to_dev(dict(W, x=x))
    f, g = fwd_bwd(d, dy.cuda(), 10, bias=bias.cuda())
    ids, w, sig = checked_routes(f, x, W, bias, 10)
    loads = np.bincount(ids.reshape(-1), minlength=512)
    empty = np.flatnonzero(loads == 0)
    assert len(empty) >= 64
    et = torch.as_tensor(empty, device="cuda")
    for key in ("dw_gate_up", "dw_down", "dw_router"):
        assert torch.count_nonzero(g[key][et]) == 0, key
    rng = np.random.default_rng(6)
    sample = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 10, replace=False)]))
    dx, dw, dl, ds = oracle_bwd_rows(x[sample], ids[sample], w[sample], sig[sample], dy[sample], W)
    st = torch.as_tensor(sample, device="cuda")
    assert_grad_close(g["dx"][st], dx, "dx sampled")
    assert_grad_close(g["dlogit"][st], dl, "dlogit sampled")
    big = int(np.argmax(loads))
    assert loads[big] > 5 * loads.mean()
    for e in (big, int(np.argsort(loads)[len(loads) // 2])):
        dwgu, dwdn = oracle.backward_expert_weights(x, ids, w, dy, W["w_gate_up"], W["w_down"], e, e + 1)
        assert_grad_close(g["dw_gate_up"][e:e + 1], dwgu, f"dw_gate_up[{e}] ({loads[e]} routes)")
        assert_grad_close(g["dw_down"][e:e + 1], dwdn, f"dw_down[{e}]")
    assert moe.moe_device_status(reset=True) == 0


@pytest.mark.parametrize("shape", [(600, 256, 4, 2, 256, 512), (77, 256, 16, 4, 128, 384)],
                         ids=["tensor-core", "cuda-core"])
def test_bf16_small_shapes_every_gradient(shape):
    """Every gradient of a small bf16 layer against the oracle's full backward:
    one shape on the tensor-core GEMMs (H, I, Is multiples of 256, several
    row tiles per expert and ragged tails), one on the CUDA-core kernels
    (I, Is multiples of 128 only)."""
    T, H, E, k, I_, Is = shape
    c = small_layer(T, H, E, k, I_, Is)
    d = to_dev(c)
    f, g = fwd_bwd(d, d["dy"], k)
    ids, w, sig = checked_routes(f, c["x"], c, None, k)
    ref = oracle.layer_backward(c["x"], ids, w, sig, *[c[n] for n in WKEYS], c["dy"])
    for key in ("dx", "dw_gate_up", "dw_down", "dws_gate_up", "dws_down", "dw_router", "dw_shared_gate",
                "dlogit"):
        assert_grad_close(g[key], ref[key], key)
    assert_grad_close(g["dz"], dz_of(ref["dsig"], sig), "dz")
    assert moe.moe_device_status(reset=True) == 0


@pytest.mark.parametrize("shape", [(120, 768, 32, 1, 128, 128), (90, 1024, 64, 7, 256, 256),
                                   (64, 512, 32, 13, 128, 128)],
                         ids=["H768-k1", "H1024-k7", "H512-k13"])
def test_bf16_row_lengths_and_slot_counts(shape):
    """y and the gradients that the combine and its backward produce, for
    slot counts and row lengths the workloads do not reach: k = 1, 7 and 13
    (the combine keeps up to 2, 8 and 16 routed chunks per thread in flight)
    and rows of 768, 1024 and 512 features (the combine backward's loop form,
    and its register form with 4 and 2 chunks per lane)."""
    T, H, E, k, I_, Is = shape
    c = small_layer(T, H, E, k, I_, Is, seed=23)
    d = to_dev(c)
    f, g = fwd_bwd(d, d["dy"], k)
    ids, w, sig = checked_routes(f, c["x"], c, None, k)
    y = oracle.moe_forward(c["x"], ids, w, sig, c["w_gate_up"], c["w_down"], c["ws_gate_up"], c["ws_down"])
    assert_bf16_close(f["y"], y, f"y {shape}")
    ref = oracle.layer_backward(c["x"], ids, w, sig, *[c[n] for n in WKEYS], c["dy"])
    for key in ("dx", "dlogit", "dw_router", "dw_shared_gate"):
        assert_grad_close(g[key], ref[key], f"{key} {shape}")
    assert_grad_close(g["dz"], dz_of(ref["dsig"], sig), f"dz {shape}")
    assert moe.moe_device_status(reset=True) == 0
