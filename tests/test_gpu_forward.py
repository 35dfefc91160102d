"""GPU parity of the forward path against the FP64 oracle, through the C ABI.

Layer: RL-Kernel PR #557 "EP4 distributed logprob parity", embedded #503
commit message ("Routing", "Experts", "Combine").  Bars: routes and the
permutation bit-exact (near-ties excepted, see tests/_util.py), values
within the stated tolerances, rows bitwise independent of the batch.
"""
import numpy as np
import pytest
import torch

import oracle
import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build
from top_routed_grouped_gb300 import inputs as I

from _util import (assert_bf16_close, assert_f32_close, bits, full_weights, full_x, oracle_routes, oracle_rows,
                   oracle_segment_rows, oracle_shared_rows, to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    moe.lib()
    moe.moe_device_status(reset=True)


def run_forward(d, k, want_logits=True):
    return moe.forward(d["x"], d["w_router"], d["w_shared_gate"], d["w_gate_up"], d["w_down"], d["ws_gate_up"],
                       d["ws_down"], k, router_bias=d.get("router_bias"), want_logits=want_logits)


def check_routes_and_permutation(out, x_cpu, wr_cpu, bias_cpu, k, E):
    gl = out["logits"].double().cpu().numpy()
    ids, w, near, l64 = oracle_routes(x_cpu, wr_cpu, bias_cpu, k, gl)
    dl = float(np.max(np.abs(gl - l64)))
    # The near-tie rule (gap < 1e-4 in either precision) is sound only while
    # 2 max|dl| < 1e-4: then every other token orders the same in both.
    assert dl < 5e-5, dl
    print(f"logit max|dl|={dl:.2e} near-tie tokens={int(near.sum())}/{len(near)}")
    gids = out["topk_ids"].cpu().numpy()
    np.testing.assert_array_equal(gids, ids)
    # w = softmax of the selected logits: |dw| <= 2 max|dl| w (+ FP32 rounding of the softmax)
    gw = out["topk_w"].double().cpu().numpy()
    assert np.all(np.abs(gw - w) <= 2 * dl * w + 4e-7), float(np.max(np.abs(gw - w)))
    off, srt, pos = oracle.permute(gids, E)
    np.testing.assert_array_equal(out["expert_offsets"].cpu().numpy(), off)
    np.testing.assert_array_equal(out["sorted_route"].cpu().numpy(), srt)
    np.testing.assert_array_equal(out["route_pos"].cpu().numpy(), pos)
    return ids, w, near


def test_tiny_f32_full_parity():
    cfg = I.CONFIGS["tiny_f32"]
    c = I.make_inputs(cfg)
    out = run_forward(to_dev(c), cfg.k)
    ids, w, near = check_routes_and_permutation(out, c["x"], c["w_router"], None, cfg.k, cfg.E)
    sig = oracle.shared_gate(c["x"], c["w_shared_gate"])
    np.testing.assert_allclose(out["shared_sig"].double().cpu().numpy(), sig, rtol=0, atol=1e-6)
    y, yr, ys = oracle.moe_forward(c["x"], ids, w, sig, c["w_gate_up"], c["w_down"], c["ws_gate_up"], c["ws_down"],
                                   want_rows=True)
    assert_f32_close(out["y_routed"], yr, "y_routed")
    assert_f32_close(out["y_shared"], ys, "y_shared")
    assert_f32_close(out["y"], y, "y")


@pytest.mark.parametrize("T", [1, 37, 300])
def test_bf16_small_batches_full_parity(T):
    W = full_weights()
    x = full_x(4096)[:T].clone()
    d = to_dev(dict(W, x=x))
    out = run_forward(d, 10)
    ids, w, near = check_routes_and_permutation(out, x, W["w_router"], None, 10, 512)
    sig = oracle.shared_gate(x, W["w_shared_gate"])
    np.testing.assert_allclose(out["shared_sig"].double().cpu().numpy(), sig, rtol=0, atol=1e-6)
    y, yr, ys = oracle_rows(x, ids, w, sig, W, want_rows=True)
    assert_bf16_close(out["y_routed"], yr, "y_routed")
    assert_bf16_close(out["y_shared"], ys, "y_shared")
    assert_bf16_close(out["y"], y, "y")


def pick_segments(off, T, k, zipf):
    """Expert segments to compare whole: the largest, the smallest non-empty,
    one whose length leaves a ragged tail in its last 256-row pair item, and
    (skewed routing) the largest two spanning several pair items besides it."""
    n = off[1:] - off[:-1]
    nz = np.flatnonzero(n > 0)
    order = nz[np.argsort(n[nz], kind="stable")]
    pick = [int(order[-1]), int(order[0])]
    ragged = [int(e) for e in order[::-1] if n[e] % 32 not in (0, 16) and int(e) not in pick]
    pick += ragged[:1]
    if zipf:
        multi = [int(e) for e in order[::-1] if n[e] > 256 and int(e) not in pick]
        pick += multi[:2]
        pick += [e for e in ragged if n[e] > 256 and e not in pick][:1]
    return pick


@pytest.mark.parametrize("T,zipf", [(1024, False), (8192, False), (16384, True)])
def test_bf16_full_size(T, zipf):
    """Full workload sizes: routes and permutation of every token; values of
    sampled tokens; at T >= 8192 also the unweighted rows of whole expert
    segments (the largest, the smallest, ragged tails, segments over several
    256-row pair items) and 512 shared-expert rows, element by element."""
    W = full_weights()
    x = full_x(16384)[:T].clone()
    bias = I.zipf_bias(512) if zipf else None
    d = to_dev(dict(W, x=x, router_bias=bias))
    out = run_forward(d, 10)
    ids, w, near = check_routes_and_permutation(out, x, W["w_router"], bias, 10, 512)
    rng = np.random.default_rng(T)
    sample = np.unique(np.concatenate([[0, T - 1], rng.choice(T, 14, replace=False)]))
    sig = oracle.shared_gate(x[sample], W["w_shared_gate"])
    y = oracle_rows(x[sample], ids[sample], w[sample], sig, W)
    assert_bf16_close(out["y"][torch.as_tensor(sample, device="cuda")], y, f"y T={T}")
    if zipf:
        import json, os
        ref = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "zipf_bias.json")))
        loads = np.bincount(out["topk_ids"].cpu().numpy().reshape(-1), minlength=512)
        assert int((loads == 0).sum()) == ref["empty_experts"]
        assert abs(int(loads.max()) - ref["max_load"]) <= 2
    if T < 8192:
        return
    off = out["expert_offsets"].cpu().numpy()
    srt = out["sorted_route"].cpu().numpy()
    segs = pick_segments(off, T, 10, zipf)
    if zipf:
        assert max(off[e + 1] - off[e] for e in segs) > 6000
    for e in segs:
        routes = srt[off[e]:off[e + 1]]
        yr = oracle_segment_rows(x[torch.as_tensor(routes // 10)], W["w_gate_up"][e], W["w_down"][e])
        assert_bf16_close(out["y_routed"][torch.as_tensor(routes, device="cuda", dtype=torch.int64)], yr,
                          f"y_routed segment e={e} ({len(routes)} rows)")
    rows = np.unique(np.concatenate([rng.choice(T, 510, replace=False), [0, T - 1]]))
    ys = oracle_shared_rows(x[torch.as_tensor(rows)], W["ws_gate_up"], W["ws_down"])
    assert_bf16_close(out["y_shared"][torch.as_tensor(rows, device="cuda")], ys, f"y_shared {len(rows)} rows")


def test_batch_invariance_bits():
    """Rows of a shuffled 8192-token batch, run in chunks of 1, 7, 256 and 8192,
    equal the full run bit for bit (output and every per-token intermediate)."""
    W = full_weights()
    T = 8192
    x = full_x(T).cuda()
    Wd = to_dev(W)
    full = run_forward(dict(Wd, x=x), 10)
    perm = I.shuffled_order(T).cuda()
    xs = x[perm]
    for b in (1, 7, 256, 8192):
        ys, ids, ws = [], [], []
        for lo, hi in I.ragged_batches(T, b):
            o = run_forward(dict(Wd, x=xs[lo:hi]), 10, want_logits=False)
            ys.append(o["y"]); ids.append(o["topk_ids"]); ws.append(o["topk_w"])
        inv = torch.empty_like(perm)
        inv[perm] = torch.arange(T, device="cuda")
        y = torch.cat(ys)[inv]
        assert torch.equal(bits(y), bits(full["y"])), f"batch {b}: y differs"
        assert torch.equal(torch.cat(ids)[inv].cpu(), full["topk_ids"].cpu()), f"batch {b}: ids differ"
        assert torch.equal(bits(torch.cat(ws)[inv]), bits(full["topk_w"])), f"batch {b}: w differs"


def test_repeat_launch_determinism():
    W = to_dev(full_weights())
    x = full_x(1024).cuda()
    ref = run_forward(dict(W, x=x), 10)
    for _ in range(20):
        o = run_forward(dict(W, x=x), 10)
        for key in ("y", "y_routed", "y_shared", "topk_w", "shared_sig", "logits"):
            assert torch.equal(bits(o[key]), bits(ref[key])), key
        for key in ("topk_ids", "expert_offsets", "sorted_route", "route_pos"):
            assert torch.equal(o[key], ref[key]), key


def test_zero_tokens():
    W = to_dev(full_weights())
    x = torch.empty(0, 2048, dtype=torch.bfloat16, device="cuda")
    out = run_forward(dict(W, x=x), 10)
    assert out["y"].shape == (0, 2048)
    assert out["expert_offsets"].cpu().tolist() == [0] * 513


def test_one_expert_takes_every_token_and_empty_experts():
    """A bias that sends every token to experts 5 and 9: 510 empty segments,
    two segments of T rows each (tiles over several row blocks, ragged tail)."""
    W = full_weights()
    T = 333
    x = full_x(T)
    bias = torch.full((512,), -100.0)
    bias[5] = 50.0
    bias[9] = 40.0
    d = to_dev(dict(W, x=x, router_bias=bias))
    out = moe.forward(d["x"], d["w_router"], d["w_shared_gate"], d["w_gate_up"], d["w_down"], d["ws_gate_up"],
                      d["ws_down"], 2, router_bias=d["router_bias"], want_logits=True)
    ids, w, near = check_routes_and_permutation(out, x, W["w_router"], bias, 2, 512)
    assert (ids[:, 0] == 5).all() and (ids[:, 1] == 9).all()
    sig = oracle.shared_gate(x, W["w_shared_gate"])
    sample = np.array([0, 1, 100, 331, 332])
    y = oracle_rows(x[sample], ids[sample], w[sample], sig[sample], W)
    assert_bf16_close(out["y"][torch.as_tensor(sample, device="cuda")], y, "y")


def test_permute_bad_ids_reported_on_device():
    ids = torch.tensor([[0, 3], [7, 1]], dtype=torch.int32, device="cuda")
    moe.moe_device_status(reset=True)
    moe.permute(ids, 4)
    assert moe.moe_device_status(reset=True) == 1
    moe.permute(ids.clamp(max=3), 4)
    assert moe.moe_device_status(reset=True) == 0


def check_permute(ids, E):
    out = moe.permute(torch.as_tensor(ids, device="cuda"), E)
    off, srt, pos = oracle.permute(ids, E)
    np.testing.assert_array_equal(out["expert_offsets"].cpu().numpy(), off)
    np.testing.assert_array_equal(out["sorted_route"].cpu().numpy(), srt)
    np.testing.assert_array_equal(out["route_pos"].cpu().numpy(), pos)


def test_permute_matches_oracle_random_ids():
    """Distinct ids per token (uniform ids with repeats for the largest case).
    Up to 2^20 routes the sort is one launch on a cluster of sixteen CTAs;
    110,000 x 10 routes take the four-kernel sort."""
    rng = np.random.default_rng(0)
    for T, E, k in [(1, 512, 10), (999, 512, 10), (5000, 64, 8), (70, 1024, 16), (8192, 512, 10)]:
        ids = np.argsort(rng.random((T, E)), axis=1)[:, :k].astype(np.int32)
        check_permute(ids, E)
    check_permute(rng.integers(0, 512, size=(110_000, 10), dtype=np.int32), 512)


def test_permute_skewed_ids_with_repeats():
    """The counting sort does not need distinct ids: heavily skewed ids with
    repeats inside a token, every chunk and warp boundary crossed by equal
    ids, an expert count that is not a multiple of 32, routes not a multiple
    of 32."""
    rng = np.random.default_rng(1)
    for T, E, k in [(4096, 16, 4), (333, 7, 3), (20_000, 1000, 10), (1, 1, 1), (3, 1024, 16)]:
        p = 1.0 / np.arange(1, E + 1) ** 1.5
        ids = rng.choice(E, size=(T, k), p=p / p.sum()).astype(np.int32)
        check_permute(ids, E)
    check_permute(np.zeros((5000, 8), np.int32), 512)  # every route to expert 0


@pytest.mark.parametrize("T,zipf", [(333, False), (1024, False), (4096, True), (6144, True), (8192, False),
                                    (16384, True)])
def test_forward_equals_step_by_step_calls(T, zipf):
    """moe_forward (the one-launch sort also writes the grouped GEMMs' item
    tables; above 2048 tokens the shared expert's GEMMs run on a second
    stream, forked after the router launch below 256 routes per expert and
    at the call from there on, i.e. T = 16384) equals moe_route,
    moe_permute, moe_grouped_ffn (which builds its own tables, shared expert
    included) and moe_combine called one by one, bit for bit."""
    W = to_dev(full_weights())
    x = full_x(T).cuda()
    bias = I.zipf_bias(512).cuda() if zipf else None
    ref = moe.forward(x, W["w_router"], W["w_shared_gate"], W["w_gate_up"], W["w_down"], W["ws_gate_up"],
                      W["ws_down"], 10, router_bias=bias, save_for_backward=True)
    r = moe.route(x, W["w_router"], W["w_shared_gate"], 10, router_bias=bias)
    pm = moe.permute(r["topk_ids"], 512)
    d = moe.dims_of(x, W["w_router"], W["w_gate_up"], W["ws_gate_up"], 10)
    yr = torch.empty(T * 10, 2048, dtype=x.dtype, device="cuda")
    ys = torch.empty(T, 2048, dtype=x.dtype, device="cuda")
    saved = {n: torch.empty_like(v) for n, v in ref["saved"].items()}  # the training activations too
    moe.moe_grouped_ffn(d, x, pm["expert_offsets"], pm["sorted_route"], W["w_gate_up"], W["w_down"],
                        W["ws_gate_up"], W["ws_down"], yr, ys, saved, moe.workspace(d, "grouped_ffn"))
    for key, v in saved.items():
        assert torch.equal(bits(v), bits(ref["saved"][key])), key
    y = torch.empty(T, 2048, dtype=x.dtype, device="cuda")
    moe.moe_combine(d, yr, ys, r["topk_w"], r["shared_sig"], y)
    for key in ("expert_offsets", "sorted_route", "route_pos"):
        assert torch.equal(pm[key], ref[key]), key
    assert torch.equal(bits(yr), bits(ref["y_routed"]))
    assert torch.equal(bits(ys), bits(ref["y_shared"]))
    assert torch.equal(bits(y), bits(ref["y"]))
    assert moe.moe_device_status(reset=True) == 0


def test_api_errors_on_device_buffers():
    W = to_dev(full_weights())
    x = full_x(16).cuda()
    d = moe.dims_of(x, W["w_router"], W["w_gate_up"], W["ws_gate_up"], 10)
    ids = torch.empty(16, 10, dtype=torch.int32, device="cuda")
    wt = torch.empty(16, 10, dtype=torch.float32, device="cuda")
    sig = torch.empty(16, dtype=torch.float32, device="cuda")
    ws = moe.workspace(d, "route")
    with pytest.raises(moe.MoEError) as e:  # misaligned x
        moe.moe_route(d, x.view(-1)[1:].view(-1)[:16 * 2048 - 8], W["w_router"], None, W["w_shared_gate"], ids, wt,
                      sig, None, ws)
    assert e.value.status == -1
    with pytest.raises(moe.MoEError) as e:
        moe.moe_route(d, x, W["w_router"], None, W["w_shared_gate"], ids, wt, sig, None, ws[:256])
    assert e.value.status == -3


def test_pair_and_single_sm_gemms_agree_bitwise(tmp_path):
    """The router and the grouped GEMMs on CTA pairs (two SMs per M = 256
    MMA) and on single SMs give the same bits: each output is one MMA chain
    over K in the same order either way (router logits, routes and training
    activations included).  The library reads its form switch (MOE_TC_PAIR)
    once per process, so the single-SM forms run in a child process."""
    import os
    import subprocess
    import sys
    from _forms_child import KEYS, SAVED, run
    if "MOE_TC_PAIR" in os.environ:
        pytest.skip("this process runs a forced GEMM form")
    Ts = (37, 300, 2048, 8192)
    out = tmp_path / "single_sm.pt"
    env = dict(os.environ, MOE_TC_PAIR="0")
    child = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_forms_child.py")
    subprocess.run([sys.executable, child, str(out)] + [str(T) for T in Ts], env=env, check=True, timeout=900)
    single = torch.load(out)
    for T in Ts:
        pair = run(T)
        for key in KEYS:
            assert torch.equal(bits(pair[key]), bits(single[T][key])), (T, key)
        for key in SAVED:
            assert torch.equal(bits(pair["saved_" + key]), bits(single[T]["saved_" + key])), (T, key)
