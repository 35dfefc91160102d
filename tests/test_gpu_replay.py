"""Router replay (moe_route_replay, moe_forward with replay_ids) on the GPU.

SkyRL PR #2513, section "chunked_mlp fixes (#2532, merged)" (per-chunk router
replay) and SkyRL docs "Qwen3.8-Flash-Next", section "Example scripts"
(rollout routing replay): a later pass reuses the expert choices of an
earlier one.  Bars: with the ids moe_route chose, weights and gate equal
moe_route's bit for bit; for other ids, the weights are the softmax of the
given slots' logits (oracle in FP64, the route-weight bar of the forward
tests); the layer output and gradients with replayed routes match the
oracle; invalid ids fail closed with a device status code.
"""
import numpy as np
import pytest
import torch

import oracle
import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build
from top_routed_grouped_gb300 import inputs as I

from _util import (assert_bf16_close, assert_grad_close, bits, full_dy, full_weights, full_x, oracle_bwd_rows,
                   oracle_rows, to_dev)

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    moe.lib()
    moe.moe_device_status(reset=True)


def random_ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32)


@pytest.mark.parametrize("cfg_name,T", [("tiny_f32", 64), ("bf16_t1024", 1024)])
def test_replay_of_own_routes_is_bitwise(cfg_name, T):
    cfg = I.CONFIGS[cfg_name]
    d = to_dev(I.make_inputs(cfg, T=T))
    r = moe.route(d["x"], d["w_router"], d["w_shared_gate"], cfg.k, want_logits=True)
    p = moe.route_replay(d["x"], d["w_router"], d["w_shared_gate"], r["topk_ids"], want_logits=True)
    assert torch.equal(bits(p["topk_w"]), bits(r["topk_w"]))
    assert torch.equal(bits(p["shared_sig"]), bits(r["shared_sig"]))
    assert torch.equal(bits(p["logits"]), bits(r["logits"]))
    assert moe.moe_device_status(reset=True) == 0


def test_replay_of_other_routes_matches_oracle():
    """Arbitrary distinct ids in arbitrary slot order (not descending)."""
    W = full_weights()
    T, E, k = 300, 512, 10
    x = full_x(4096)[:T].clone()
    ids = random_ids(T, E, k, 7)
    d = to_dev(dict(W, x=x))
    p = moe.route_replay(d["x"], d["w_router"], d["w_shared_gate"], torch.as_tensor(ids, device="cuda"),
                         want_logits=True)
    assert moe.moe_device_status(reset=True) == 0
    l64 = oracle.router_logits(x, W["w_router"])
    gl = p["logits"].double().cpu().numpy()
    dl = float(np.max(np.abs(gl - l64)))
    assert dl < 5e-5, dl
    w64 = oracle.topk_weights(l64, ids)
    gw = p["topk_w"].double().cpu().numpy()
    assert np.all(np.abs(gw - w64) <= 2 * dl * w64 + 4e-7), float(np.max(np.abs(gw - w64)))
    np.testing.assert_allclose(gw.sum(axis=1), 1.0, atol=1e-6)
    sig = oracle.shared_gate(x, W["w_shared_gate"])
    np.testing.assert_allclose(p["shared_sig"].double().cpu().numpy(), sig, rtol=0, atol=1e-6)


def test_replayed_layer_forward_and_backward():
    """moe_forward with replay_ids, then moe_backward: sampled tokens against
    the oracle run on the same (replayed) routes."""
    W = full_weights()
    T, E, k = 256, 512, 10
    x, dy = full_x(T), full_dy(T)
    ids = random_ids(T, E, k, 11)
    d = to_dev(dict(W, x=x))
    args = [d[n] for n in WKEYS]
    ids_dev = torch.as_tensor(ids, device="cuda")
    f = moe.forward(d["x"], *args, k, save_for_backward=True, want_logits=True, replay_ids=ids_dev)
    assert torch.equal(f["topk_ids"], ids_dev)
    g = moe.backward(f, dy.cuda(), d["x"], *args)
    assert moe.moe_device_status(reset=True) == 0
    l64 = oracle.router_logits(x, W["w_router"])
    w = oracle.topk_weights(l64, ids)
    sig = oracle.shared_gate(x, W["w_shared_gate"])
    sample = np.array([0, 1, 77, 128, 255])
    st = torch.as_tensor(sample, device="cuda")
    y = oracle_rows(x[sample], ids[sample], w[sample], sig[sample], W)
    assert_bf16_close(f["y"][st], y, "y replayed")
    dx, _, dlg, _ = oracle_bwd_rows(x[sample], ids[sample], w[sample], sig[sample], dy[sample], W)
    assert_grad_close(g["dx"][st], dx, "dx replayed")
    assert_grad_close(g["dlogit"][st], dlg, "dlogit replayed")


def test_replay_batch_invariance():
    W = to_dev(full_weights())
    T = 64
    x = full_x(T).cuda()
    ids = torch.as_tensor(random_ids(T, 512, 10, 3), device="cuda")
    full = moe.route_replay(x, W["w_router"], W["w_shared_gate"], ids)
    for lo, hi in I.ragged_batches(T, 7):
        part = moe.route_replay(x[lo:hi], W["w_router"], W["w_shared_gate"], ids[lo:hi].clone())
        assert torch.equal(bits(part["topk_w"]), bits(full["topk_w"][lo:hi]))
        assert torch.equal(bits(part["shared_sig"]), bits(full["shared_sig"][lo:hi]))


@pytest.mark.parametrize("bad,code", [("range", 1), ("repeat", 4)])
def test_replay_invalid_ids_fail_closed(bad, code):
    W = to_dev(full_weights())
    T = 16
    x = full_x(T).cuda()
    ids = random_ids(T, 512, 10, 5)
    if bad == "range":
        ids[3, 4] = 512
    else:
        ids[3, 4] = ids[3, 0]
    moe.moe_device_status(reset=True)
    p = moe.route_replay(x, W["w_router"], W["w_shared_gate"], torch.as_tensor(ids, device="cuda"))
    assert moe.moe_device_status(reset=True) == code
    w = p["topk_w"].cpu()
    assert torch.count_nonzero(w[3]) == 0
    others = torch.cat([w[:3], w[4:]])
    assert torch.allclose(others.sum(dim=1), torch.ones(T - 1), atol=1e-6)


@pytest.mark.parametrize("T", [4096, 16384])
def test_replayed_forward_with_second_stream_is_bitwise(T):
    """Above 2048 tokens moe_forward runs the shared expert's GEMMs on a
    second stream, forked after the router launch (T = 4096: 80 routes per
    expert) or at the call (T = 16384: 320).  Replaying the call's own routes
    takes the replay gate instead of top-k at the fork point and gives the
    same rows and output bit for bit."""
    W = to_dev(full_weights())
    x = full_x(T).cuda()
    args = [W[n] for n in WKEYS]
    f = moe.forward(x, *args, 10)
    g = moe.forward(x, *args, 10, replay_ids=f["topk_ids"].clone())
    assert torch.equal(g["topk_ids"], f["topk_ids"])
    for key in ("y_routed", "y_shared", "y"):
        assert torch.equal(bits(g[key]), bits(f[key])), key
    assert moe.moe_device_status(reset=True) == 0
