"""Pins of the FP64 oracle against facts that do not come from the oracle.

Each test checks the oracle against something independent of its code:
a dense brute-force evaluation of every expert with a full-sort top-k,
closed forms (identical experts, k = E, k = 1, x = 0, shared expert only),
library routines (numpy's stable argsort / lexsort), the exact algebra of the
permutation (bijection, inverse, stability), and central finite differences
for the backward.  The layer definition is the one of RL-Kernel PR #557,
embedded #503 commit message ("Routing", "Experts", "Combine", "Backward").
"""
import math

import numpy as np
import pytest

import oracle
from top_routed_grouped_gb300 import inputs as I


def small(T, H, E, k, Iw, Is, seed=0, bias=False):
    """Small random layer in float64 numpy (weights N(0, 0.3) so FFNs matter)."""
    def n(shape, stream, std):
        return I.normal(shape, seed, stream, std).double().numpy()
    d = {
        "x": n((T, H), 11, 1.0),
        "w_router": n((E, H), 12, 0.5),
        "w_shared_gate": n((H,), 13, 0.5),
        "w_gate_up": n((E, 2 * Iw, H), 14, 0.3),
        "w_down": n((E, H, Iw), 15, 0.3),
        "ws_gate_up": n((2 * Is, H), 16, 0.3),
        "ws_down": n((H, Is), 17, 0.3),
        "router_bias": n((E,), 18, 0.2) if bias else None,
        "dy": n((T, H), 19, 1.0),
    }
    d["k"] = k
    return d


def silu(g):
    return g / (1.0 + np.exp(-g))


def sigmoid(z):
    return 1.0 / (1.0 + np.exp(-z))


def swiglu_np(x, wgu, wdn):
    """Textbook SwiGLU MLP: Wdn (silu(Wg x) * Wu x) for rows of x."""
    Iw = wgu.shape[0] // 2
    g = x @ wgu[:Iw].T
    u = x @ wgu[Iw:].T
    return (silu(g) * u) @ wdn.T


def brute_force(d):
    """Dense mixture: every expert on every token, full softmax, full-sort mask."""
    x, wr = d["x"], d["w_router"]
    T, H = x.shape
    E = wr.shape[0]
    k = d["k"]
    logits = x @ wr.T
    if d["router_bias"] is not None:
        logits = logits + d["router_bias"]
    p = np.exp(logits - logits.max(1, keepdims=True))
    p = p / p.sum(1, keepdims=True)
    mask = np.zeros_like(p)
    ids = np.zeros((T, k), np.int64)
    for t in range(T):
        order = np.lexsort((np.arange(E), -logits[t]))  # desc logit, then asc id
        mask[t, order[:k]] = 1.0
        ids[t] = order[:k]
    wf = p * mask
    wf = wf / wf.sum(1, keepdims=True)
    Y = np.stack([swiglu_np(x, d["w_gate_up"][e], d["w_down"][e]) for e in range(E)], 1)  # [T,E,H]
    sig = sigmoid(x @ d["w_shared_gate"])
    y = np.einsum("te,teh->th", wf, Y) + sig[:, None] * swiglu_np(x, d["ws_gate_up"], d["ws_down"])
    return {"logits": logits, "ids": ids, "wfull": wf, "sig": sig, "y": y}


def run_oracle(d):
    return oracle.layer_forward(d["x"], d["w_router"], d["w_shared_gate"], d["w_gate_up"], d["w_down"],
                                d["ws_gate_up"], d["ws_down"], d["k"], d["router_bias"])


@pytest.mark.parametrize("dims", [(64, 32, 16, 4, 8, 8), (17, 24, 8, 3, 4, 6), (5, 16, 6, 6, 4, 4),
                                  (9, 8, 5, 1, 3, 2)])
@pytest.mark.parametrize("bias", [False, True])
def test_oracle_vs_dense_bruteforce(dims, bias):
    d = small(*dims, bias=bias)
    o = run_oracle(d)
    b = brute_force(d)
    np.testing.assert_allclose(o["logits"], b["logits"], rtol=0, atol=1e-12)
    np.testing.assert_array_equal(o["ids"], b["ids"])
    T, k = o["ids"].shape
    for t in range(T):
        np.testing.assert_allclose(o["w"][t], b["wfull"][t, o["ids"][t]], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o["sig"], b["sig"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(o["y"], b["y"], rtol=0, atol=1e-12)


def test_oracle_tiny_config_vs_bruteforce():
    cfg = I.CONFIGS["tiny_f32"]
    t = I.make_inputs(cfg)
    d = {kk: (v.double().numpy() if v is not None else None) for kk, v in t.items()}
    d["k"] = cfg.k
    o = run_oracle(d)
    b = brute_force(d)
    np.testing.assert_array_equal(o["ids"], b["ids"])
    np.testing.assert_allclose(o["y"], b["y"], rtol=0, atol=1e-12)


def test_identical_experts_reduce_to_one_mlp():
    """All experts equal: sum_s w_s = 1, so y = FFN(x) + sig Ys for any routing."""
    d = small(12, 16, 7, 3, 5, 4)
    d["w_gate_up"][:] = d["w_gate_up"][2]
    d["w_down"][:] = d["w_down"][2]
    o = run_oracle(d)
    x = d["x"]
    ref = swiglu_np(x, d["w_gate_up"][0], d["w_down"][0]) + \
        sigmoid(x @ d["w_shared_gate"])[:, None] * swiglu_np(x, d["ws_gate_up"], d["ws_down"])
    np.testing.assert_allclose(o["y"], ref, rtol=0, atol=1e-12)


def test_k_equals_E_is_dense_softmax_mixture():
    d = small(10, 12, 5, 5, 4, 3)
    o = run_oracle(d)
    x = d["x"]
    l = x @ d["w_router"].T
    p = np.exp(l - l.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    Y = np.stack([swiglu_np(x, d["w_gate_up"][e], d["w_down"][e]) for e in range(5)], 1)
    ref = np.einsum("te,teh->th", p, Y) + \
        sigmoid(x @ d["w_shared_gate"])[:, None] * swiglu_np(x, d["ws_gate_up"], d["ws_down"])
    np.testing.assert_allclose(o["y"], ref, rtol=0, atol=1e-12)
    np.testing.assert_allclose(o["w"].sum(1), 1.0, rtol=0, atol=1e-15)


def test_k1_is_argmax_expert_mlp():
    d = small(10, 12, 6, 1, 4, 3)
    o = run_oracle(d)
    x = d["x"]
    am = np.argmax(x @ d["w_router"].T, axis=1)  # numpy: first occurrence on ties
    np.testing.assert_array_equal(o["ids"][:, 0], am)
    np.testing.assert_array_equal(o["w"], np.ones_like(o["w"]))
    for t in range(10):
        ref = swiglu_np(x[t:t + 1], d["w_gate_up"][am[t]], d["w_down"][am[t]])[0] + \
            sigmoid(x[t] @ d["w_shared_gate"]) * swiglu_np(x[t:t + 1], d["ws_gate_up"], d["ws_down"])[0]
        np.testing.assert_allclose(o["y"][t], ref, rtol=0, atol=1e-12)


def test_zero_input_pins_tie_break():
    """x = 0: every logit is 0, so the tie rule picks experts 0..k-1, w = 1/k, y = 0, sig = 1/2."""
    d = small(4, 8, 9, 4, 3, 3)
    d["x"][:] = 0.0
    o = run_oracle(d)
    np.testing.assert_array_equal(o["ids"], np.tile(np.arange(4), (4, 1)))
    np.testing.assert_array_equal(o["w"], np.full((4, 4), 0.25))
    np.testing.assert_array_equal(o["sig"], np.full(4, 0.5))
    np.testing.assert_array_equal(o["y"], np.zeros((4, 8)))


def test_shared_only_when_routed_down_is_zero():
    d = small(8, 12, 5, 2, 4, 3)
    d["w_down"][:] = 0.0
    o = run_oracle(d)
    x = d["x"]
    ref = sigmoid(x @ d["w_shared_gate"])[:, None] * swiglu_np(x, d["ws_gate_up"], d["ws_down"])
    np.testing.assert_allclose(o["y"], ref, rtol=0, atol=1e-13)


def test_hand_worked_example():
    """H=2, E=3, k=2, I=Is=1, worked by hand.

    x = (1, 0); router rows give logits (0.5, 0.2, 0.3) -> experts (0, 2) in
    that slot order, w = (sigmoid(0.2), sigmoid(-0.2)).  Expert e has gate row
    (a_e, 0), up row (1, 0) and down column (c_e, 0): Y_e = (c_e silu(a_e), 0).
    Shared: gate (1,0), up (2,0), down (1, 1): Ys = (2 silu(1), 2 silu(1)).
    Gate weight (0.4, 7): sig = sigmoid(0.4).
    """
    a = [0.7, -1.1, 2.0]
    c = [1.5, 3.0, -0.5]
    wgu = np.zeros((3, 2, 2))
    wdn = np.zeros((3, 2, 1))
    for e in range(3):
        wgu[e, 0, 0] = a[e]
        wgu[e, 1, 0] = 1.0
        wdn[e, 0, 0] = c[e]
    d = {"x": np.array([[1.0, 0.0]]), "w_router": np.array([[0.5, 9.0], [0.2, -3.0], [0.3, 1.0]]),
         "w_shared_gate": np.array([0.4, 7.0]), "w_gate_up": wgu, "w_down": wdn,
         "ws_gate_up": np.array([[1.0, 0.0], [2.0, 0.0]]), "ws_down": np.array([[1.0], [1.0]]),
         "router_bias": None, "k": 2}
    o = run_oracle(d)
    s = lambda z: 1.0 / (1.0 + math.exp(-z))
    sl = lambda g: g * s(g)
    assert o["ids"].tolist() == [[0, 2]]
    w0, w2 = s(0.2), s(-0.2)
    assert abs(o["w"][0, 0] - w0) < 1e-15 and abs(o["w"][0, 1] - w2) < 1e-15
    y0 = w0 * c[0] * sl(a[0]) + w2 * c[2] * sl(a[2]) + s(0.4) * 2 * sl(1.0)
    y1 = s(0.4) * 2 * sl(1.0)
    np.testing.assert_allclose(o["y"][0], [y0, y1], rtol=0, atol=1e-15)


def test_topk_ties_match_lexsort():
    rng = np.random.default_rng(5)
    l = rng.integers(-3, 4, size=(200, 13)).astype(np.float64)  # many exact ties
    ids = oracle.topk_select(l, 5)
    for t in range(200):
        ref = np.lexsort((np.arange(13), -l[t]))[:5]
        np.testing.assert_array_equal(ids[t], ref)


def test_topk_weights_are_softmax_of_selected():
    rng = np.random.default_rng(6)
    l = rng.normal(size=(50, 20)) * 3
    ids = oracle.topk_select(l, 6)
    w = oracle.topk_weights(l, ids)
    sel = np.take_along_axis(l, ids.astype(np.int64), 1)
    ref = np.exp(sel - sel.max(1, keepdims=True))
    ref /= ref.sum(1, keepdims=True)
    np.testing.assert_allclose(w, ref, rtol=1e-14, atol=0)
    full = np.exp(l - l.max(1, keepdims=True))
    full /= full.sum(1, keepdims=True)
    psel = np.take_along_axis(full, ids.astype(np.int64), 1)
    np.testing.assert_allclose(w, psel / psel.sum(1, keepdims=True), rtol=1e-13, atol=0)
    assert np.all(np.diff(sel, axis=1) <= 0)  # slot order = descending logit


@pytest.mark.parametrize("T,E,k", [(1, 4, 2), (37, 16, 4), (300, 64, 10), (0, 8, 2)])
def test_permute_invariants(T, E, k):
    rng = np.random.default_rng(T + E)
    ids = np.stack([rng.permutation(E)[:k] for _ in range(T)]) if T else np.zeros((0, k), np.int32)
    off, srt, pos = oracle.permute(ids, E)
    R = T * k
    flat = ids.reshape(-1)
    counts = np.bincount(flat, minlength=E) if R else np.zeros(E, np.int64)
    np.testing.assert_array_equal(off, np.concatenate([[0], np.cumsum(counts)]))
    assert off[-1] == R
    np.testing.assert_array_equal(np.sort(srt), np.arange(R))  # bijection
    np.testing.assert_array_equal(srt[pos], np.arange(R))  # inverse
    np.testing.assert_array_equal(srt, np.argsort(flat, kind="stable"))  # library routine
    for e in range(E):
        seg = srt[off[e]:off[e + 1]]
        assert np.all(flat[seg] == e)
        assert np.all(np.diff(seg) > 0)  # (t, s) ascending within a segment
    if R:  # every token appears in exactly k segments
        np.testing.assert_array_equal(np.bincount(srt // k, minlength=T), np.full(T, k))


def test_permute_rejects_bad_ids():
    with pytest.raises(ValueError):
        oracle.permute(np.array([[0, 5]], np.int32), 5)


def test_batch_independence():
    """Rows computed alone equal rows computed in a batch (the oracle is per token)."""
    d = small(20, 16, 8, 3, 4, 4)
    full = run_oracle(d)
    for t in (0, 7, 19):
        sub = dict(d)
        sub["x"] = d["x"][t:t + 1]
        one = run_oracle(sub)
        np.testing.assert_array_equal(one["y"][0], full["y"][t])
        np.testing.assert_array_equal(one["ids"][0], full["ids"][t])


# --------------------------------------------------------------------- backward
def loss_fixed_routes(d, ids):
    """L = sum(dy * y) with the selected set held fixed (the weights still move)."""
    x = d["x"]
    l = x @ d["w_router"].T
    w = oracle.topk_weights(l, ids)
    sig = oracle.shared_gate(x, d["w_shared_gate"])
    y = oracle.moe_forward(x, ids, w, sig, d["w_gate_up"], d["w_down"], d["ws_gate_up"], d["ws_down"])
    return float(np.sum(d["dy"] * y))


def test_backward_matches_finite_differences():
    d = small(6, 8, 5, 2, 4, 3)
    o = run_oracle(d)
    ids = o["ids"]
    g = oracle.layer_backward(d["x"], ids, o["w"], o["sig"], d["w_router"], d["w_shared_gate"],
                              d["w_gate_up"], d["w_down"], d["ws_gate_up"], d["ws_down"], d["dy"])
    eps = 1e-6
    rng = np.random.default_rng(0)

    def fd(name, idx):
        a = d[name]
        old = a[idx]
        a[idx] = old + eps
        lp = loss_fixed_routes(d, ids)
        a[idx] = old - eps
        lm = loss_fixed_routes(d, ids)
        a[idx] = old
        return (lp - lm) / (2 * eps)

    used = np.unique(ids)
    checks = [("x", "dx"), ("w_router", "dw_router"), ("w_shared_gate", "dw_shared_gate"),
              ("ws_gate_up", "dws_gate_up"), ("ws_down", "dws_down")]
    for pname, gname in checks:
        shape = d[pname].shape
        for _ in range(6):
            idx = tuple(int(rng.integers(0, s)) for s in shape)
            num, ana = fd(pname, idx), g[gname][idx]
            assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), (pname, idx, num, ana)
    for pname, gname in [("w_gate_up", "dw_gate_up"), ("w_down", "dw_down")]:
        shape = d[pname].shape
        for _ in range(8):
            e = int(rng.choice(used))
            idx = (e,) + tuple(int(rng.integers(0, s)) for s in shape[1:])
            num, ana = fd(pname, idx), g[gname][idx]
            assert abs(num - ana) <= 1e-6 * max(1.0, abs(num)), (pname, idx, num, ana)
    unused = [e for e in range(5) if e not in used]
    for e in unused:
        assert np.all(g["dw_gate_up"][e] == 0) and np.all(g["dw_down"][e] == 0)


def test_route_weight_grad_and_router_jacobian():
    """dw = dy . Yr and dlogit = J^T dw with J the softmax-over-the-set Jacobian."""
    d = small(7, 10, 6, 3, 4, 3)
    o = run_oracle(d)
    y, yr, ys = oracle.moe_forward(d["x"], o["ids"], o["w"], o["sig"], d["w_gate_up"], d["w_down"],
                                   d["ws_gate_up"], d["ws_down"], want_rows=True)
    dx, dw, dl, ds = oracle.backward_tokens(d["x"], o["ids"], o["w"], o["sig"], d["w_router"],
                                            d["w_shared_gate"], d["w_gate_up"], d["w_down"],
                                            d["ws_gate_up"], d["ws_down"], d["dy"])
    T, k = o["ids"].shape
    np.testing.assert_allclose(dw, np.einsum("th,tsh->ts", d["dy"], yr.reshape(T, k, -1)), atol=1e-13, rtol=0)
    np.testing.assert_allclose(ds, np.einsum("th,th->t", d["dy"], ys), atol=1e-13, rtol=0)
    for t in range(T):
        wv = o["w"][t]
        J = np.diag(wv) - np.outer(wv, wv)  # d softmax / d logits (symmetric)
        np.testing.assert_allclose(dl[t], J @ dw[t], atol=1e-14, rtol=0)
    np.testing.assert_allclose(dl.sum(1), 0.0, atol=1e-14)


def test_expert_weight_grad_range_matches_full():
    d = small(9, 8, 6, 2, 3, 3)
    o = run_oracle(d)
    full_gu, full_dn = oracle.backward_expert_weights(d["x"], o["ids"], o["w"], d["dy"], d["w_gate_up"], d["w_down"])
    part_gu, part_dn = oracle.backward_expert_weights(d["x"], o["ids"], o["w"], d["dy"], d["w_gate_up"],
                                                      d["w_down"], 2, 5)
    np.testing.assert_array_equal(part_gu, full_gu[2:5])
    np.testing.assert_array_equal(part_dn, full_dn[2:5])
