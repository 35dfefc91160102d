"""The expert-partition exchange across two processes (gloo, CPU).

RL-Kernel PR #557 "What": each rank computes the routed rows of its own
experts, one all_gather of the rows (a byte copy) gives every rank all of
them, the combine is local.  Here each rank computes its rows with the FP64
oracle on the tiny workload, ep.exchange_rows exchanges them over a gloo
process group, and every rank's assembled rows and combined output must
equal the single-process oracle bit for bit.  No GPU is used.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from top_routed_grouped_gb300 import ep
from top_routed_grouped_gb300 import inputs as I


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _layer():
    cfg = I.CONFIGS["tiny_f32"]
    c = I.make_inputs(cfg)
    _, ids, w, sig = oracle.route(c["x"], c["w_router"], c["w_shared_gate"], cfg.k)
    r = {"ids": ids, "w": w, "sig": sig}
    off, srt, pos = oracle.permute(ids, cfg.E)
    return cfg, c, r, off, srt, pos


def _rows_of(c, r, srt, k, rows):
    """Oracle routed rows for the given sorted rows (route sorted_route[j])."""
    out = {}
    for j in rows:
        route = int(srt[j])
        t, s = divmod(route, k)
        e = int(r["ids"][t, s])
        out[j] = oracle.expert_ffn(c["x"][t].double().numpy(), c["w_gate_up"][e].double().numpy(),
                                   c["w_down"][e].double().numpy())
    return out


def _worker(rank, world, port, result_q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        cfg, c, r, off, srt, pos = _layer()
        ranges = ep.expert_ranges(cfg.E, world)
        R = cfg.T * cfg.k
        y_sorted = torch.full((R, cfg.H), float("nan"), dtype=torch.float64)
        r0, r1 = ep.rank_rows(off, ranges[rank])
        for j, row in _rows_of(c, r, srt, cfg.k, range(r0, r1)).items():
            y_sorted[j] = torch.from_numpy(row)
        ep.exchange_rows(y_sorted, off, ranges)
        result_q.put((rank, y_sorted.numpy().tobytes()))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2])
def test_exchange_assembles_every_row_on_every_rank(world):
    oracle.build()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(rank, world, port, q)) for rank in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=300) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg, c, r, off, srt, pos = _layer()
    R = cfg.T * cfg.k
    ref = np.stack([_rows_of(c, r, srt, cfg.k, [j])[j] for j in range(R)])
    for rank in range(world):
        rows = np.frombuffer(got[rank], dtype=np.float64).reshape(R, cfg.H)
        np.testing.assert_array_equal(rows, ref)
        # in route order, the assembled rows are the oracle layer's routed rows
        _, yr64, _ = oracle.moe_forward(c["x"], r["ids"], r["w"], r["sig"], c["w_gate_up"], c["w_down"],
                                        c["ws_gate_up"], c["ws_down"], want_rows=True)
        np.testing.assert_array_equal(rows[pos], yr64)


def test_expert_ranges_cover_and_balance():
    for E, world in [(16, 2), (512, 3), (7, 4), (512, 8)]:
        ranges = ep.expert_ranges(E, world)
        ep.check_partition(ranges, E)
        sizes = [t - b for b, t in ranges]
        assert max(sizes) - min(sizes) <= 1
        assert [ep.owner_of(e, ranges) for e in range(E)] == sorted(ep.owner_of(e, ranges) for e in range(E))
