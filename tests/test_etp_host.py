"""Expert tensor parallelism on the host: feature slicing against the oracle,
and the partial-sum exchange across two processes (gloo, CPU).

RL-Kernel PR #557 "What", bullet "Fail closed" (EP 1 = experts
expert-tensor-parallel over 4 ranks) and #503 "TP4 block" (partials reduced
across ranks).  Since Yr = sum_i h_i W_down[:, i] over the features i, the
oracle's expert FFN on a rank's weight slices is that rank's partial sum:
the partials of a split sum to the unsplit rows (FP64, up to reordering).
A slice that took the wrong up rows or down columns fails that.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from top_routed_grouped_gb300 import etp
from top_routed_grouped_gb300 import inputs as I


def test_feature_ranges_cover_and_balance():
    for width, world in [(512, 1), (512, 2), (512, 3), (512, 4), (1024, 3)]:
        rs = etp.feature_ranges(width, world)
        etp.check_ranges(rs, width)
        sizes = [b - a for a, b in rs]
        assert max(sizes) - min(sizes) <= etp.GRANULE and all(s % etp.GRANULE == 0 for s in sizes)
    with pytest.raises(ValueError):
        etp.feature_ranges(512, 5)  # fewer than 5 slices of 128
    with pytest.raises(ValueError):
        etp.feature_ranges(500, 2)
    with pytest.raises(ValueError):
        etp.check_ranges([(0, 128), (256, 512)], 512)  # features 128..255 unowned
    with pytest.raises(ValueError):
        etp.check_ranges([(0, 256), (128, 512)], 512)  # overlap


def _tiny():
    cfg = I.CONFIGS["tiny_f32"]
    return cfg, I.make_inputs(cfg)


def _partial_rows(c, e, rows, rng, rng_sh, shared=False):
    """Oracle rows of expert e (or the shared expert) on its slice weights."""
    if shared:
        wg, wd = etp.slice_gate_up(c["ws_gate_up"], *rng_sh), etp.slice_down(c["ws_down"], *rng_sh)
    else:
        wg, wd = etp.slice_gate_up(c["w_gate_up"][e], *rng), etp.slice_down(c["w_down"][e], *rng)
    return np.stack([oracle.expert_ffn(c["x"][t].double().numpy(), wg.double().numpy(), wd.double().numpy())
                     for t in rows])


@pytest.mark.parametrize("world,granule", [(2, 32), (4, 32), (3, 4)])
def test_slice_partials_sum_to_full_rows(world, granule):
    cfg, c = _tiny()
    rs = etp.feature_ranges(cfg.I, world, granule)
    rs_sh = etp.feature_ranges(cfg.Is, world, granule)
    rows = [0, 5, 63]
    for e in (0, 7, cfg.E - 1):
        full = _partial_rows(c, e, rows, (0, cfg.I), (0, cfg.Is))
        parts = sum(_partial_rows(c, e, rows, rng, rs_sh[0]) for rng in rs)
        np.testing.assert_allclose(parts, full, rtol=1e-12, atol=1e-14)
    full_sh = _partial_rows(c, 0, rows, (0, cfg.I), (0, cfg.Is), shared=True)
    parts_sh = sum(_partial_rows(c, 0, rows, rs[0], rng_sh, shared=True) for rng_sh in rs_sh)
    np.testing.assert_allclose(parts_sh, full_sh, rtol=1e-12, atol=1e-14)


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, c = _tiny()
        rs = etp.feature_ranges(cfg.I, world, 32)
        rows = list(range(0, cfg.T, 9))
        mine = torch.from_numpy(_partial_rows(c, 3, rows, rs[rank], (0, cfg.Is)))
        parts = etp.exchange_partials(mine)
        total = parts[0].clone()
        for p in parts[1:]:
            total += p  # rank order
        q.put((rank, total.numpy().tobytes()))
    finally:
        dist.destroy_process_group()


def test_partial_exchange_over_gloo():
    oracle.build()
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg, c = _tiny()
    rows = list(range(0, cfg.T, 9))
    full = _partial_rows(c, 3, rows, (0, cfg.I), (0, cfg.Is))
    a = np.frombuffer(got[0], dtype=np.float64).reshape(full.shape)
    b = np.frombuffer(got[1], dtype=np.float64).reshape(full.shape)
    assert np.array_equal(a, b)  # every rank reduces the same bytes in the same order
    np.testing.assert_allclose(a, full, rtol=1e-12, atol=1e-14)
