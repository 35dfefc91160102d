"""Expert tensor parallelism (ETP), simulated on one GPU.

RL-Kernel PR #557 "What", bullet "Fail closed" (EP 1 = every expert
expert-tensor-parallel over 4 ranks) and #503 "TP4 block" (partials reduced
across ranks).  Bars: with one rank the split path equals moe_grouped_ffn
bit for bit (the unrounded partial rounded once is the same FP32
accumulator); with 2 or 4 ranks the layer output matches the FP64 oracle
within the layer's tolerances and is bitwise repeatable and batch
invariant; the reduction sums in rank order (a case where the order changes
the FP32 result pins it).
"""
import numpy as np
import pytest
import torch

import oracle
import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build, etp
from top_routed_grouped_gb300 import inputs as I

from _util import assert_bf16_close, assert_f32_close, bits, full_weights, full_x, oracle_rows, to_dev

pytestmark = pytest.mark.gpu

WKEYS = ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")


@pytest.fixture(scope="module", autouse=True)
def built():
    build.build()
    moe.lib()
    moe.moe_device_status(reset=True)


def run(d, k, world, bias=None):
    return etp.forward_simulated(d["x"], *[d[n] for n in WKEYS], k, world, router_bias=bias)


def test_one_rank_equals_single_launch():
    W = to_dev(full_weights())
    d = dict(W, x=full_x(1024).cuda())
    ref = moe.forward(d["x"], *[d[n] for n in WKEYS], 10)
    out = run(d, 10, 1)
    for key in ("y", "y_routed", "y_shared"):
        assert torch.equal(bits(out[key]), bits(ref[key])), key
    assert moe.moe_device_status(reset=True) == 0


@pytest.mark.parametrize("world", [2, 4])
def test_bf16_split_matches_oracle(world):
    W = full_weights()
    T = 1024
    x = full_x(T)
    d = to_dev(dict(W, x=x))
    out = run(d, 10, world)
    assert moe.moe_device_status(reset=True) == 0
    r = out["route"]
    sample = np.array([0, 1, 2, 100, 511, 777, 1023])
    st = torch.as_tensor(sample, device="cuda")
    ids = r["topk_ids"].cpu().numpy()[sample]
    w = r["topk_w"].double().cpu().numpy()[sample]
    sig = r["shared_sig"].double().cpu().numpy()[sample]
    y64 = oracle_rows(x[sample], ids, w, sig, W)
    assert_bf16_close(out["y"][st], y64, f"y, {world} ranks")
    # the split changes only rounding: against the single launch, within the same bar
    ref = moe.forward(d["x"], *[d[n] for n in WKEYS], 10)
    assert_bf16_close(out["y_routed"], ref["y_routed"].double().cpu().numpy(), "y_routed vs single launch")


def test_split_repeatable_and_batch_invariant():
    W = to_dev(full_weights())
    T, world = 300, 4
    x = full_x(T).cuda()
    d = dict(W, x=x)
    ref = run(d, 10, world)
    again = run(d, 10, world)
    for key in ("y", "y_routed", "y_shared"):
        assert torch.equal(bits(again[key]), bits(ref[key])), key
    for lo, hi in I.ragged_batches(T, 5):
        part = run(dict(W, x=x[lo:hi].clone()), 10, world)
        assert torch.equal(bits(part["y"]), bits(ref["y"][lo:hi]))


@pytest.mark.parametrize("world", [2, 4])
def test_f32_split_full_parity(world):
    cfg = I.CONFIGS["tiny_f32"]
    c = I.make_inputs(cfg)
    d = to_dev(c)
    out = run(d, cfg.k, world)
    r = out["route"]
    ids = r["topk_ids"].cpu().numpy()
    w = r["topk_w"].double().cpu().numpy()
    sig = r["shared_sig"].double().cpu().numpy()
    y64 = oracle.moe_forward(c["x"], ids, w, sig, c["w_gate_up"], c["w_down"], c["ws_gate_up"], c["ws_down"])
    assert_f32_close(out["y"], y64, f"y, {world} ranks")


def test_reduce_sums_in_rank_order():
    """FP32 partials 1, 2^-24, 2^-24: in rank order each addition rounds back
    to 1 (ties to even); any other order gives 1 + 2^-23."""
    dims = moe.make_dims(1, 4, 2, 1, 4, 4, torch.float32)
    one, eps = 1.0, 2.0 ** -24
    parts_r = [torch.full((1, 4), v, device="cuda") for v in (one, eps, eps)]
    parts_s = [torch.full((1, 4), v, device="cuda") for v in (eps, eps, one)]
    yr = torch.empty(1, 4, device="cuda")
    ys = torch.empty(1, 4, device="cuda")
    moe.moe_etp_reduce(dims, parts_r, parts_s, yr, ys)
    assert torch.all(yr == 1.0)
    assert torch.all(ys == 1.0 + 2.0 ** -23)


def test_reduce_rejects_bad_part_counts():
    dims = moe.make_dims(1, 4, 2, 1, 4, 4, torch.float32)
    y = torch.empty(1, 4, device="cuda")
    for n in (0, 17):
        parts = [torch.zeros(1, 4, device="cuda") for _ in range(n)]
        with pytest.raises(moe.MoEError):
            moe.moe_etp_reduce(dims, parts, parts, y, y)


def rank_partials(d, k, rng, rng_sh, bias=None, fused=False):
    """One rank's FP32 partial rows through moe_grouped_ffn_etp(_fused)."""
    x = d["x"]
    T, H = x.shape
    E = d["w_router"].shape[0]
    r = moe.route(x, d["w_router"], d["w_shared_gate"], k, router_bias=bias)
    pm = moe.permute(r["topk_ids"], E)
    wg, wd, wsg, wsd = etp.rank_weights(d["w_gate_up"], d["w_down"], d["ws_gate_up"], d["ws_down"], rng, rng_sh)
    dims = moe.make_dims(T, H, E, k, rng[1] - rng[0], rng_sh[1] - rng_sh[0], x.dtype)
    pr = torch.full((T * k, H), float("nan"), device="cuda")
    ps = torch.full((T, H), float("nan"), device="cuda")
    ws = moe.workspace(dims, "grouped_ffn")
    if fused:
        moe.moe_grouped_ffn_etp_fused(dims, x, pm["expert_offsets"], pm["sorted_route"], wg, wd, wsg, wsd, pr, ps, ws)
    else:
        moe.moe_grouped_ffn_etp(dims, x, pm["expert_offsets"], pm["sorted_route"], wg, wd, wsg, wsd, pr, ps, None, ws)
    return pr, ps


@pytest.mark.parametrize("T,zipf", [(37, False), (1024, False), (8192, False), (4096, True)])
def test_fused_slice_equals_two_kernel_slice(T, zipf):
    """The fused gate_up -> down of a 128-feature slice (h kept in shared
    memory) gives the two-kernel path's FP32 partial rows bit for bit, for
    every rank of a four-way split: ragged row tiles (T = 37), one item per
    expert (T = 1024), about 160 rows per expert (T = 8192), and long skewed
    segments of many 128-row items (Zipf routing)."""
    W = to_dev(full_weights())
    d = dict(W, x=full_x(T).cuda())
    bias = I.zipf_bias(512).cuda() if zipf else None
    ranges, ranges_sh = etp.feature_ranges(512, 4), etp.feature_ranges(512, 4)
    for rank, (rng, rng_sh) in enumerate(zip(ranges, ranges_sh)):
        ref_r, ref_s = rank_partials(d, 10, rng, rng_sh, bias)
        got_r, got_s = rank_partials(d, 10, rng, rng_sh, bias, fused=True)
        assert torch.equal(bits(got_r), bits(ref_r)), f"rank {rank}: routed partials"
        assert torch.equal(bits(got_s), bits(ref_s)), f"rank {rank}: shared partials"
    assert moe.moe_device_status(reset=True) == 0


def test_fused_split_matches_oracle():
    W = full_weights()
    T = 1024
    x = full_x(T)
    d = to_dev(dict(W, x=x))
    out = etp.forward_simulated(d["x"], *[d[n] for n in WKEYS], 10, 4, fused=True)
    assert moe.moe_device_status(reset=True) == 0
    ref = run(d, 10, 4)
    for key in ("y", "y_routed", "y_shared"):
        assert torch.equal(bits(out[key]), bits(ref[key])), key
    r = out["route"]
    sample = np.array([0, 1, 2, 100, 511, 777, 1023])
    st = torch.as_tensor(sample, device="cuda")
    ids = r["topk_ids"].cpu().numpy()[sample]
    w = r["topk_w"].double().cpu().numpy()[sample]
    sig = r["shared_sig"].double().cpu().numpy()[sample]
    assert_bf16_close(out["y"][st], oracle_rows(x[sample], ids, w, sig, W), "y, 4 ranks (fused slices)")


def test_fused_rejects_other_slice_widths():
    W = to_dev(full_weights())
    d = dict(W, x=full_x(64).cuda())
    with pytest.raises(moe.MoEError) as e:  # two ranks: 256-feature slices
        rank_partials(d, 10, (0, 256), (0, 256), fused=True)
    assert e.value.status == -2
