"""bench.py's multi-rank plumbing on CPU (gloo, two processes): the timed
value is the maximum over the ranks on every rank, the barrier returns, and
under torchrun the reference arm runs on rank 0 only (the other ranks exit 0
without work).  No GPU is used."""
import os
import socket
import subprocess
import sys

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        q.put((rank, bench.max_over_ranks(1.5 + rank, world)))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_barrier_over_gloo():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got == {0: 2.5, 1: 2.5}


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny_f32"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_roofline_denominators_match_the_buffers():
    """The layer roofline's algorithmic bytes are the sizes of the buffers the
    layer touches once: every expert weight (all 512 experts are active at
    T=8192), the shared expert, the FP32 router weight and the shared gate, x
    read and y written; the backward adds a gradient buffer per weight in FP32
    and reads dy, writes dx.  FLOPs are 2 M N K per GEMM: per route a gate/up
    product (M = 2I, K = H) and a down product (M = H, K = I), per token the
    same with the shared expert's Is; the backward runs twice that."""
    sys.path.insert(0, ROOT)
    import bench
    from top_routed_grouped_gb300 import inputs as I
    cfg = I.CONFIGS["bf16_t8192"]
    T, H, E, k, Iw, Is = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.Is
    w = I.make_inputs(cfg, T=1)
    names = ("w_gate_up", "w_down", "ws_gate_up", "ws_down", "w_router", "w_shared_gate")
    weight_bytes = sum(w[n].numel() * w[n].element_size() for n in names)
    act = T * H * 2  # one bf16 [T, H] tensor
    fwd = bench.layer_bytes_flops(T, H, E, k, Iw, Is, E)
    assert fwd["bytes"] == weight_bytes + 2 * act
    gemm = lambda m, n, kk: 2 * m * n * kk
    flops = T * k * (gemm(2 * Iw, 1, H) + gemm(H, 1, Iw)) + T * (gemm(2 * Is, 1, H) + gemm(H, 1, Is))
    assert fwd["flops"] == flops
    bwd = bench.bwd_bytes_flops(T, H, E, k, Iw, Is)
    grad_bytes = sum(w[n].numel() * 4 for n in names)
    assert bwd["bytes"] == weight_bytes + grad_bytes + 3 * act
    assert bwd["flops"] == 2 * flops


def test_reference_arm_line_on_cpu():
    """The reference arm (the FP64 oracle on the host cores) prints one JSON
    line with the contract's keys: its cpu_baseline value is the line's
    value, its e2e moves no bytes, and its config has the same keys as the
    GPU arm's (workload_config)."""
    import json
    sys.path.insert(0, ROOT)
    import bench
    from top_routed_grouped_gb300 import inputs as I
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "tiny_f32", "--steps", "2", "--warmup", "3"], env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["steps"] == 2 and line["warmup"] == 3 and line["n_gpus"] == 1
    assert line["value"] > 0 and line["unit"] == "tokens/s" and line["higher_is_better"] is True
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] >= 1 and cb["value"] == line["value"] and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}
    cfg = I.CONFIGS["tiny_f32"]
    assert set(line["config"]) == set(bench.workload_config(cfg, cfg.E, 1))
    assert line["config"]["workload"] == "tiny_f32" and line["config"]["T"] == cfg.T


def test_launch_counts_follow_the_forward_structure():
    """gpu_launches: seven launches on the caller's stream, the router's
    chunk sum where T * E / 256 <= 4096, the shared expert's four on the
    second stream above 2048 tokens (the ncu launch lists in profiles/ show
    11 per forward at T = 8192 and at T = 4096, 23 per forward + backward)."""
    sys.path.insert(0, ROOT)
    import bench
    assert bench.launches_per_forward(8192, 512) == 11
    assert bench.launches_per_forward(4096, 512) == 11
    assert bench.launches_per_forward(2048, 512) == 8
    assert bench.launches_per_forward(1024, 512) == 8
    assert bench.launches_per_forward(16384, 512) == 11
