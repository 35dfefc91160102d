"""Benchmark of the batch-invariant MoE layer on GB300.

One step = one forward of the layer over one batch of T tokens (router,
top-k and gate, dispatch permute, grouped SwiGLU experts with the shared
expert, ordered combine) through the C ABI's moe_forward, inputs resident in
HBM.  The
default workload is bf16_t8192 (T=8192, H=2048, 512 experts top-10, I=Is=512);
the expert weights (3.2 GB) exceed L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  Keys beyond the basic contract:
  e2e          same metric through moe_forward with pinned host buffers and
               the host<->device copies of x and y inside the timed region
               (copies on their own streams, two alternating buffers, so a
               step's copies overlap its neighbours' compute)
  roofline     the dominant operation (moe_grouped_ffn) against measured HBM,
               its launches timed by CUDA events in a second loop of K steps
               that calls the four steps one by one (step_by_step)
  layer_roofline  the whole step against max(bytes/HBM, FLOPs/tensor peak)
  cpu_baseline the FP64 oracle on the host cores, on a bounded token sample
  clocks       nvidia-smi samples taken during the timed region
  fwd_bwd      forward (activations saved) + backward at T=4096
               (bf16_t4096_fwdbwd) through moe_forward / moe_backward, with
               its own layer roofline (forward and backward bytes and FLOPs)
  step_ms      p10 / p50 / p90 of the per-step times (also in fwd_bwd)
  extra_forward  the forward at T=1024 and at T=16384 with Zipf-skewed
               routing (same layer), reported beside the headline
  etp_slice    one expert-tensor-parallel rank's grouped FFN (128-feature
               slices) at T=8192: two kernels with h through HBM against
               the fused kernel that keeps h in shared memory

--impl reference times the oracle itself (the reference arm) on the host.
Multi-GPU (torchrun): every rank runs its own replica of the workload
(tokens shard with no exchange), value = all ranks' tokens / max rank time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
METRIC = "MoE layer tokens/sec (fwd, fwd+bwd) on 1 GB300; % of layer roofline"
# Kernels one forward step (moe_forward, bf16) launches: router weight split,
# router (and, for T * E / 256 <= 4096, the sum of its K-chunk planes),
# top-k/gate; the permute (one launch on a cluster of sixteen CTAs, which also
# writes the grouped GEMMs' item tables); gate_up, down; combine; above 2048
# tokens the shared expert on the second stream: its item tables (two
# launches), gate_up, down.


def launches_per_forward(T: int, E: int) -> int:
    return 7 + (1 if T * (E // 256) <= 4096 else 0) + (4 if T > 2048 else 0)


# The same forward as four separate calls: moe_grouped_ffn builds its own
# item tables (2 more launches).
LAUNCHES_PER_STEP_BY_STEP = 9


def load_peaks() -> tuple[dict, str]:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return json.load(f), "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def cpu_model() -> str:
    """The host CPU's model name (lscpu), for the oracle timing record."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.processor() or platform.machine()


def percentiles(vals) -> dict:
    """p10 / p50 / p90 of per-step times in ms."""
    v = sorted(vals)
    pick = lambda q: v[min(len(v) - 1, int(round(q * (len(v) - 1))))]  # noqa: E731
    return {"p10": pick(0.1), "p50": pick(0.5), "p90": pick(0.9), "n": len(v)}


def max_over_ranks(value: float, world: int) -> float:
    """Largest value over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


class _Nvml:
    """Read-only NVML queries through ctypes (the driver's libnvidia-ml):
    current and maximum SM clock, clock-event reasons and power draw."""
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown", 0x4: "sw_power_cap"}

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h)) != 0:
            raise OSError("no NVML handle")
        self.reasons_fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self.lib.nvmlDeviceGetCurrentClocksThrottleReasons
        self.max_sm = self._clock(self.lib.nvmlDeviceGetMaxClockInfo)

    def _clock(self, fn) -> int | None:
        v = self.ct.c_uint(0)
        return int(v.value) if fn(self.h, self.ct.c_int(1), self.ct.byref(v)) == 0 else None  # 1 = SM clock

    def sample(self) -> tuple:
        r = self.ct.c_ulonglong(0)
        reasons = int(r.value) if self.reasons_fn(self.h, self.ct.byref(r)) == 0 else 0
        mw = self.ct.c_uint(0)
        power = mw.value / 1000.0 if self.lib.nvmlDeviceGetPowerUsage(self.h, self.ct.byref(mw)) == 0 else None
        return self._clock(self.lib.nvmlDeviceGetClockInfo), self.max_sm, reasons, power


class ClockSampler:
    """SM clock and throttle reasons during a region.

    Preferred source: NVML polled every millisecond from a thread (read-only
    queries), so that a region of a few milliseconds still gets samples;
    fallback: nvidia-smi every 50 ms.  start() returns once sampling runs,
    and only samples taken between begin() and end() count."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, period_ms: int = 50, nvml_period_s: float = 0.001):
        self.idx, self.period, self.nvml_period = gpu_index, period_ms, nvml_period_s
        self.proc, self.lines, self.t0, self.t1 = None, [], None, None
        self.nvml, self.samples, self.stop_flag, self.thread = None, [], False, None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line))

    def _poll(self):
        while not self.stop_flag:
            self.samples.append((time.perf_counter(), self.nvml.sample()))
            time.sleep(self.nvml_period)

    def start(self):
        import threading
        try:
            self.nvml = _Nvml(self.idx)
            self.thread = threading.Thread(target=self._poll, daemon=True)
            self.thread.start()
            return
        except (OSError, AttributeError):
            self.nvml = None
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(self.period)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        threading.Thread(target=self._read, daemon=True).start()
        deadline = time.perf_counter() + 5.0
        while not self.lines and time.perf_counter() < deadline and self.proc.poll() is None:
            time.sleep(0.01)

    def begin(self):
        self.t0 = time.perf_counter()

    def end(self):
        self.t1 = time.perf_counter()

    def _inside(self, ts) -> bool:
        return self.t0 is None or self.t0 <= ts <= (self.t1 or ts)

    def stop(self) -> dict:
        sm, mx, reasons, power = [], [], set(), []
        if self.nvml is not None:
            self.stop_flag = True
            self.thread.join(timeout=5)
            for ts, (clk, cmax, bits, pw) in list(self.samples):
                if not self._inside(ts) or clk is None:
                    continue
                sm.append(float(clk))
                if cmax is not None:
                    mx.append(float(cmax))
                if pw is not None:
                    power.append(pw)
                reasons.update(n for b, n in _Nvml.REASONS.items() if bits & b)
            src = "nvml, 1 ms"
        elif self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            for ts, line in list(self.lines):
                if not self._inside(ts):
                    continue
                f = [x.strip() for x in line.split(",")]
                if len(f) < 8:
                    continue
                try:
                    sm.append(float(f[0]))
                    mx.append(float(f[1]))
                except ValueError:
                    continue
                for n, v in zip(self.NAMES, f[4:8]):
                    if v.lower().startswith("active"):
                        reasons.add(n)
            src = f"nvidia-smi, {self.period} ms"
        else:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm), "source": src,
                "power_w_max": max(power) if power else None}


# DRAM bytes (read + write) of one moe_grouped_ffn call (gate_up + down) at
# bf16_t8192: dram__bytes_read.sum + dram__bytes_write.sum of the two kernels
# in the first timed step-by-step call (the launch pair that the roofline
# times; the forward steps before it launch four pair GEMMs each, the shared
# expert's on the second stream) of
#   ncu --metrics dram__bytes_read.sum,dram__bytes_write.sum --clock-control none \
#       -k regex:tc_pair_kernel -s 30 -c 2 \
#       python bench.py --steps 3 --warmup 3 --no-cpu-baseline --no-fwd-bwd --no-extra
# (one pass per launch), valid only for the kernel sources it was taken on
# (hash below); otherwise null.
FFN_TRAFFIC = {"sources": "74736556d040a5f5", "workload": "bf16_t8192",
               "bytes": 2_188_150_272 + 73_008_384 + 1_186_576_640 + 317_780_224}


def kernel_sources_hash() -> str:
    """Hash of the grouped-FFN kernel sources with comments and white space
    removed: changes when the code changes, not when a comment does."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "top_routed_grouped_gb300", "csrc")
    per = []
    for n in ("gemm_tc.cu", "umma.cuh", "common.cuh"):
        src = open(os.path.join(csrc, n)).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        src = re.sub(r"//[^\n]*", "", src)
        per.append(hashlib.sha256("".join(src.split()).encode()).hexdigest())
    return hashlib.sha256("".join(per).encode()).hexdigest()[:16]


def layer_bytes_flops(T, H, E, k, I, Is, active_experts, es=2) -> dict:
    """Algorithmic bytes and FLOPs of one layer forward.

    FLOPs: 6 H I per route + 6 H Is per token (the router is not counted).
    Bytes: weights of every expert with >= 1 route, the shared expert, the fp32
    router weight and the shared gate, x read once and y written once.
    """
    weights = active_experts * 3 * H * I * es + 3 * H * Is * es + E * H * 4 + H * es
    return {"bytes": weights + 2 * T * H * es, "flops": 6 * H * I * T * k + 6 * H * Is * T, "weight_bytes": weights}


def ffn_bytes_flops(T, H, k, I, Is, active_experts, es=2) -> dict:
    """Algorithmic bytes / FLOPs of moe_grouped_ffn: weights of active experts
    and the shared expert read once, x read once, the unweighted rows written
    once, and the intermediate h written and read once."""
    R = T * k
    w = active_experts * 3 * H * I * es + 3 * H * Is * es
    b = w + T * H * es + (R + T) * H * es + 2 * (R * I + T * Is) * es
    return {"bytes": b, "flops": 6 * H * I * R + 6 * H * Is * T}


def bwd_bytes_flops(T, H, E, k, I, Is, es=2) -> dict:
    """Algorithmic bytes and FLOPs of one layer backward.

    FLOPs: twice the forward's (input and weight gradients): 12 H I per route
    + 12 H Is per token (the router and gate gradients are not counted).
    Bytes: every expert weight read once, every weight gradient written once
    in FP32 (all E experts: empty ones are written as zeros), the router
    weight read and its gradient written, x and dy read, dx written.
    """
    weights = E * 3 * H * I * es + 3 * H * Is * es + E * H * 4 + H * es
    grads = (E * 3 * H * I + 3 * H * Is + E * H + H) * 4
    return {"bytes": weights + grads + 3 * T * H * es, "flops": 12 * H * I * T * k + 12 * H * Is * T}


def fwd_bwd_bench(cfg, dev_w, steps: int, warmup: int, world: int, peaks: dict) -> dict:
    """Forward (activations saved) + backward of the layer through moe_forward
    and moe_backward, inputs and upstream gradient resident in HBM."""
    import torch
    import top_routed_grouped_gb300 as moe
    from top_routed_grouped_gb300 import inputs as I
    T, H, E, k, Iw, Is = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.Is
    x = I.normal((T, H), 0, I._STREAM["x"], 1.0, cfg.torch_dtype).cuda()
    dy = I.normal((T, H), 2, I._STREAM["dy"], 1.0, cfg.torch_dtype).cuda()
    wargs = [dev_w[n] for n in ("w_router", "w_shared_gate", "w_gate_up", "w_down", "ws_gate_up", "ws_down")]
    d = moe.make_dims(T, H, E, k, Iw, Is, cfg.torch_dtype)
    bws = moe.workspace(d, "backward")
    stream = torch.cuda.current_stream()

    def step(ev=None):
        if ev: ev[0].record(stream)
        f = moe.forward(x, *wargs, k, save_for_backward=True, stream=stream)
        if ev: ev[1].record(stream)
        moe.backward(f, dy, x, *wargs, ws=bws, stream=stream)
        if ev: ev[2].record(stream)

    for _ in range(warmup):
        step()
    torch.cuda.synchronize()
    moe.moe_device_status(reset=True)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(steps):
        step(evs[i])
    torch.cuda.synchronize()
    barrier(world)
    if moe.moe_device_status(reset=True) != 0:
        raise RuntimeError("a kernel recorded a failed device-side check during the fwd+bwd region")
    ms = max_over_ranks(statistics.mean(e[0].elapsed_time(e[2]) for e in evs), world)
    fwd_ms = statistics.mean(e[0].elapsed_time(e[1]) for e in evs)
    bwd_ms = statistics.mean(e[1].elapsed_time(e[2]) for e in evs)
    hbm, tf = float(peaks["hbm_gbs"]), float(peaks["bf16_tflops"])
    fb = layer_bytes_flops(T, H, E, k, Iw, Is, E)
    bb = bwd_bytes_flops(T, H, E, k, Iw, Is)
    roof = lambda b: max(b["bytes"] / (hbm * 1e9), b["flops"] / (tf * 1e12)) * 1e3
    t_roof = roof(fb) + roof(bb)
    return {"workload": cfg.name, "T": T, "value": T * world / (ms * 1e-3), "unit": "tokens/s",
            "ms_per_step": ms, "fwd_ms": fwd_ms, "bwd_ms": bwd_ms, "steps": steps, "warmup": warmup,
            "step_ms": percentiles([e[0].elapsed_time(e[2]) for e in evs]),
            "api": "moe_forward (activations saved) + moe_backward",
            # moe_forward (launches_per_forward); moe_backward: combine bwd, item tables (2), down
            # dgrad, gate_up dgrad, x gather, down wgrad, gate_up wgrad, tile table, router/gate
            # partial sums and reduction, dx (12)
            "gpu_launches_per_step": launches_per_forward(T, E) + 12,
            "layer_roofline": {"fwd_bytes": fb["bytes"], "fwd_flops": fb["flops"], "bwd_bytes": bb["bytes"],
                               "bwd_flops": bb["flops"], "roofline_ms": t_roof, "frac": t_roof / ms,
                               "bwd_roofline_ms": roof(bb), "bwd_frac": roof(bb) / bwd_ms}}


def extra_forward(name: str, dev_w: dict, steps: int, warmup: int, peaks: dict) -> dict:
    """The forward at another configuration of the same layer (reported beside
    the headline, not instead of it): per-step times through moe_forward
    (consecutive step starts, inputs resident), tokens/s at the median and
    the layer-roofline fraction."""
    import torch
    import top_routed_grouped_gb300 as moe
    from top_routed_grouped_gb300 import inputs as I
    cfg = I.CONFIGS[name]
    T, H, E, k, Iw, Is = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.Is
    # The weights of every configuration of this layer are the same draw; x and the bias are per configuration.
    dv = dict(dev_w, x=I.normal((T, H), 0, I._STREAM["x"], 1.0, cfg.torch_dtype).cuda(),
              router_bias=I.zipf_bias(E, cfg.zipf_beta, n_empty=cfg.zipf_empty).cuda() if cfg.zipf else None)
    d = moe.make_dims(T, H, E, k, Iw, Is, cfg.torch_dtype)
    off = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    fargs = {n: dv[n] for n in ("x", "w_router", "router_bias", "w_shared_gate", "w_gate_up", "w_down",
                                "ws_gate_up", "ws_down")}
    fargs.update(y=torch.empty(T, H, dtype=cfg.torch_dtype, device="cuda"), expert_offsets=off)
    fws = moe.workspace(d, "forward")
    stream = torch.cuda.current_stream()
    for _ in range(warmup):
        moe.moe_forward(d, fargs, fws, stream)
    torch.cuda.synchronize()
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    for i in range(steps):
        evs[i].record(stream)
        moe.moe_forward(d, fargs, fws, stream)
    evs[steps].record(stream)
    torch.cuda.synchronize()
    if moe.moe_device_status(reset=True) != 0:
        raise RuntimeError(f"a kernel recorded a failed device-side check ({name})")
    pc = percentiles([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)])
    active = int((off[1:] - off[:-1] > 0).sum().item())
    lb = layer_bytes_flops(T, H, E, k, Iw, Is, active)
    roof = max(lb["bytes"] / (float(peaks["hbm_gbs"]) * 1e9), lb["flops"] / (float(peaks["bf16_tflops"]) * 1e12))
    return {"workload": name, "T": T, "active_experts": active, "step_ms": pc,
            "tokens_per_s": T / (pc["p50"] * 1e-3), "layer_roofline_ms": roof * 1e3,
            "layer_roofline_frac": roof * 1e3 / pc["p50"], "api": "moe_forward"}


def widen(W_cpu: dict) -> dict:
    """The weights widened to float64 once (exact), as the oracle reads them."""
    import torch
    return {k: v.to(torch.float64).numpy() for k, v in W_cpu.items()}


def etp_slice_bench(dev_w: dict, steps: int, warmup: int, T: int = 8192, world: int = 4) -> dict:
    """One expert-tensor-parallel rank's FFN (rank 0 of `world`, 128-feature
    slices of I and Is) at T tokens: the two grouped GEMMs with h through
    device memory (moe_grouped_ffn_etp) against the fused form that keeps h
    in shared memory (moe_grouped_ffn_etp_fused), CUDA events, same inputs
    and routes; the partial rows must agree bit for bit."""
    import torch
    import top_routed_grouped_gb300 as moe
    from top_routed_grouped_gb300 import etp
    from top_routed_grouped_gb300 import inputs as I
    E, H, k = dev_w["w_router"].shape[0], dev_w["w_router"].shape[1], 10
    I_full, Is_full = dev_w["w_down"].shape[-1], dev_w["ws_down"].shape[-1]
    x = I.normal((T, H), 0, I._STREAM["x"], 1.0, torch.bfloat16).cuda()
    r = moe.route(x, dev_w["w_router"], dev_w["w_shared_gate"], k)
    pm = moe.permute(r["topk_ids"], E)
    rng, rng_sh = etp.feature_ranges(I_full, world)[0], etp.feature_ranges(Is_full, world)[0]
    wg, wd, wsg, wsd = etp.rank_weights(dev_w["w_gate_up"], dev_w["w_down"], dev_w["ws_gate_up"], dev_w["ws_down"],
                                        rng, rng_sh)
    d = moe.make_dims(T, H, E, k, rng[1] - rng[0], rng_sh[1] - rng_sh[0], torch.bfloat16)
    ws = moe.workspace(d, "grouped_ffn")
    outs = {}
    res = {"workload": f"rank 0 of {world}: I and Is slices of {rng[1] - rng[0]} features, T={T}, k={k}, E={E}",
           "api": "moe_grouped_ffn_etp vs moe_grouped_ffn_etp_fused"}
    for name, fused in (("two_kernels", False), ("fused", True)):
        pr = torch.empty(T * k, H, dtype=torch.float32, device="cuda")
        ps = torch.empty(T, H, dtype=torch.float32, device="cuda")

        def call():
            if fused:
                moe.moe_grouped_ffn_etp_fused(d, x, pm["expert_offsets"], pm["sorted_route"], wg, wd, wsg, wsd, pr,
                                              ps, ws)
            else:
                moe.moe_grouped_ffn_etp(d, x, pm["expert_offsets"], pm["sorted_route"], wg, wd, wsg, wsd, pr, ps,
                                        None, ws)
        for _ in range(warmup):
            call()
        evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
        stream = torch.cuda.current_stream()
        for i in range(steps):
            evs[i].record(stream)
            call()
        evs[steps].record(stream)
        torch.cuda.synchronize()
        res[name + "_ms"] = percentiles([evs[i].elapsed_time(evs[i + 1]) for i in range(steps)])["p50"]
        outs[name] = (pr, ps)
    if moe.moe_device_status(reset=True) != 0:
        raise RuntimeError("a kernel recorded a failed device-side check (ETP slice)")
    res["bitwise_equal"] = bool(torch.equal(outs["fused"][0], outs["two_kernels"][0]) and
                                torch.equal(outs["fused"][1], outs["two_kernels"][1]))
    res["fused_gain"] = 1.0 - res["fused_ms"] / res["two_kernels_ms"]
    return res


def cpu_oracle_baseline(cfg, x_cpu, W_cpu, bias, budget_s: float = 20.0, max_tokens: int | None = None,
                        f64: dict | None = None) -> dict:
    """Time the FP64 oracle (routing + experts + combine) on the first tokens
    of the workload (all of them by default), in blocks of 32 tokens until
    `budget_s` has elapsed.  `f64`: the weights already widened (else widened
    here, outside the timed blocks)."""
    if max_tokens is None:
        max_tokens = cfg.T
    os.environ.setdefault("OMP_NUM_THREADS", str(host_cores()))
    import numpy as np
    import oracle
    import torch

    if f64 is None:
        f64 = widen(W_cpu)
    b64 = None if bias is None else bias.to(torch.float64).numpy()
    oracle.build()
    done, elapsed = 0, 0.0
    while elapsed < budget_s and done < max_tokens:
        xs = x_cpu[done:done + 32].to(torch.float64).numpy()
        t0 = time.perf_counter()
        r = oracle.layer_forward(xs, f64["w_router"], f64["w_shared_gate"], f64["w_gate_up"], f64["w_down"],
                                 f64["ws_gate_up"], f64["ws_down"], cfg.k, b64)
        elapsed += time.perf_counter() - t0
        done += xs.shape[0]
        assert np.isfinite(r["y"]).all()
    return {"value": done / elapsed, "unit": "tokens/s", "cores": int(os.environ["OMP_NUM_THREADS"]),
            "cpu_model": cpu_model(), "kind": "oracle", "tokens": done, "oracle_s": elapsed,
            "sample": f"first {done} tokens of {cfg.name} (FP64 route + experts + combine), "
                      f"{elapsed:.1f} s of oracle time"}


def workload_config(cfg, active: int, world: int) -> dict:
    """The `config` object of both arms' lines (same keys and values)."""
    es = 2 if cfg.dtype == "bf16" else 4
    wb = cfg.E * 3 * cfg.H * cfg.I * es
    l2 = (f"no flush: expert weights ({wb / 1e9:.1f} GB) exceed the 129 MB L2" if wb > 129e6 else
          f"expert weights ({wb / 1e6:.1f} MB) fit in L2; no flush")
    return {"workload": cfg.name, "T": cfg.T, "H": cfg.H, "E": cfg.E, "k": cfg.k, "I": cfg.I, "Is": cfg.Is,
            "step": "forward", "active_experts": active, "l2": l2, "parallelism": f"replicas x{world}"}


def run_reference(args, cfg, rank: int) -> None:
    """Reference arm: the oracle, as it stands, on the host cores.  A step is
    a bounded sample of the workload (the first tokens, as many as the
    oracle finishes in a few seconds); value = tokens / oracle time over all
    steps, ms_per_step = the measured time of one such step."""
    if rank != 0:
        return
    import numpy as np
    import oracle
    from top_routed_grouped_gb300 import inputs as I
    d = I.make_inputs(cfg)
    W = {k: v for k, v in d.items() if k not in ("x", "dy", "router_bias")}
    # active experts of the whole workload, from the oracle's own routing
    ids = oracle.topk_select(oracle.router_logits(d["x"], W["w_router"], d["router_bias"]), cfg.k)
    active = int((np.bincount(ids.reshape(-1), minlength=cfg.E) > 0).sum())
    budget = max(2.0, min(20.0, 60.0 / max(1, args.steps + args.warmup)))
    f64 = widen(W)
    for _ in range(args.warmup):
        cpu_oracle_baseline(cfg, d["x"], W, d["router_bias"], budget_s=0.5, max_tokens=32, f64=f64)
    tokens, secs, per_step = 0, 0.0, []
    cb = None
    for _ in range(args.steps):
        t0 = time.perf_counter()
        cb = cpu_oracle_baseline(cfg, d["x"], W, d["router_bias"], budget_s=budget, f64=f64)
        per_step.append(time.perf_counter() - t0)
        tokens += cb["tokens"]
        secs += cb["oracle_s"]
    v = tokens / secs
    cb = dict(cb, value=v, sample=f"{args.steps} steps, each the first {tokens // args.steps} tokens of "
                                  f"{cfg.name} (FP64 route + experts + combine, {budget:.1f} s budget per step)")
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000.0 * statistics.mean(per_step),
            "tokens_per_step": tokens // args.steps,
            "ms_per_workload_scaled": {"value": 1000.0 * cfg.T / v, "note": f"scaled: the oracle's rate applied to "
                                       f"all {cfg.T} tokens of the workload, not measured"},
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(cfg, active, args.gpus),
            "cpu_baseline": cb, "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                                        "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def route_only_bench(cfg, steps: int, warmup: int) -> dict:
    """moe_route alone on the workload's x, router weight and gate: CUDA
    events around `steps` back-to-back calls after `warmup` calls."""
    import torch
    import top_routed_grouped_gb300 as moe
    from top_routed_grouped_gb300 import inputs as I
    cpu = I.make_inputs(cfg)
    x, wr, wsg = cpu["x"].cuda(), cpu["w_router"].cuda(), cpu["w_shared_gate"].cuda()
    bias = cpu["router_bias"].cuda() if cpu.get("router_bias") is not None else None
    for _ in range(warmup):
        moe.route(x, wr, wsg, cfg.k, router_bias=bias)
    s = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(s)
    for _ in range(steps):
        moe.route(x, wr, wsg, cfg.k, router_bias=bias)
    e1.record(s)
    torch.cuda.synchronize()
    if moe.moe_device_status(reset=True) != 0:
        raise RuntimeError("a kernel recorded a failed device-side check")
    return {"workload": cfg.name, "T": cfg.T, "E": cfg.E, "k": cfg.k, "steps": steps,
            "ms_per_call": e0.elapsed_time(e1) / max(steps, 1), "api": "moe_route"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=400)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="bf16_t8192")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-fwd-bwd", action="store_true", help="skip the forward+backward measurement")
    ap.add_argument("--no-extra", action="store_true",
                    help="skip the forward at the 1024-token and 16384-token Zipf configurations")
    ap.add_argument("--fwd-bwd-workload", default="bf16_t4096_fwdbwd",
                    help="workload of the forward+backward measurement (same layer shape as --workload)")
    ap.add_argument("--etp-only", action="store_true",
                    help="only the expert-tensor-parallel slice comparison (two kernels vs fused) on the layer of "
                         "--workload at --etp-tokens tokens, printed as one JSON object (a profiling case)")
    ap.add_argument("--etp-tokens", type=int, default=8192)
    ap.add_argument("--route-only", action="store_true",
                    help="only moe_route (router weight split, router, top-k and gate) on --workload, --steps "
                         "back-to-back calls after --warmup, printed as one JSON object (a profiling case that "
                         "holds x, the router weight and the logits only)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    from top_routed_grouped_gb300 import inputs as I
    cfg = I.CONFIGS[args.workload]
    if args.impl == "reference":
        run_reference(args, cfg, rank)
        return

    import torch
    import top_routed_grouped_gb300 as moe
    from top_routed_grouped_gb300 import build as B
    if rank == 0 or not B.up_to_date():
        B.build()
    torch.cuda.set_device(local)
    if args.etp_only:
        w = {k: v.cuda() for k, v in I.make_inputs(cfg, T=1).items() if k not in ("x", "dy", "router_bias")}
        print(json.dumps({"etp_slice": etp_slice_bench(w, args.steps, args.warmup, T=args.etp_tokens)}), flush=True)
        return
    if args.route_only:
        print(json.dumps({"route_only": route_only_bench(cfg, args.steps, args.warmup)}), flush=True)
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    # ---- inputs (seeded, made on the host, copied once) ----
    cpu = I.make_inputs(cfg)
    dev = {k: (v.cuda() if v is not None else None) for k, v in cpu.items()}
    T, H, E, k, Iw, Is = cfg.T, cfg.H, cfg.E, cfg.k, cfg.I, cfg.Is
    R = T * k
    dt = cfg.torch_dtype
    d = moe.make_dims(T, H, E, k, Iw, Is, dt)
    o = {"ids": torch.empty(T, k, dtype=torch.int32, device="cuda"),
         "w": torch.empty(T, k, dtype=torch.float32, device="cuda"),
         "sig": torch.empty(T, dtype=torch.float32, device="cuda"),
         "off": torch.empty(E + 1, dtype=torch.int32, device="cuda"),
         "srt": torch.empty(R, dtype=torch.int32, device="cuda"),
         "pos": torch.empty(R, dtype=torch.int32, device="cuda"),
         "yr": torch.empty(R, H, dtype=dt, device="cuda"),
         "ys": torch.empty(T, H, dtype=dt, device="cuda"),
         "y": torch.empty(T, H, dtype=dt, device="cuda")}
    ws = torch.empty(max(moe.moe_workspace_size(d, op) for op in ("route", "permute", "grouped_ffn")),
                     dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    fws = moe.workspace(d, "forward")
    f_out = {"x": dev["x"], "w_router": dev["w_router"], "router_bias": dev["router_bias"],
             "w_shared_gate": dev["w_shared_gate"], "w_gate_up": dev["w_gate_up"], "w_down": dev["w_down"],
             "ws_gate_up": dev["ws_gate_up"], "ws_down": dev["ws_down"], "y": o["y"], "topk_ids": o["ids"],
             "topk_w": o["w"], "shared_sig": o["sig"], "expert_offsets": o["off"], "sorted_route": o["srt"],
             "route_pos": o["pos"], "y_routed": o["yr"], "y_shared": o["ys"]}

    def step():
        """One layer forward: moe_forward (router weight split, router, top-k
        and gate, permute with the item tables, gate_up, down, combine)."""
        moe.moe_forward(d, f_out, fws, stream)

    def step_by_step(ev):
        """The same forward as the four calls one by one, with events around
        moe_grouped_ffn (the dominant operation's launches)."""
        moe.moe_route(d, dev["x"], dev["w_router"], dev["router_bias"], dev["w_shared_gate"], o["ids"], o["w"],
                      o["sig"], None, ws, stream)
        moe.moe_permute(d, o["ids"], o["off"], o["srt"], o["pos"], ws, stream)
        ev[0].record(stream)
        moe.moe_grouped_ffn(d, dev["x"], o["off"], o["srt"], dev["w_gate_up"], dev["w_down"], dev["ws_gate_up"],
                            dev["ws_down"], o["yr"], o["ys"], None, ws, stream)
        ev[1].record(stream)
        moe.moe_combine(d, o["yr"], o["ys"], o["w"], o["sig"], o["y"], stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    moe.moe_device_status(reset=True)
    active = int((o["off"][1:] - o["off"][:-1] > 0).sum().item())

    # ---- device-timed region: K forward steps through moe_forward ----
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps + 1)]
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    clocks.begin()
    for i in range(args.steps):
        evs[i].record(stream)
        step()
    evs[args.steps].record(stream)
    torch.cuda.synchronize()
    clocks.end()
    clk = clocks.stop()
    barrier(world)
    ms_local = evs[0].elapsed_time(evs[args.steps]) / args.steps
    ms = max_over_ranks(ms_local, world)
    if moe.moe_device_status(reset=True) != 0:
        raise RuntimeError("a kernel recorded a failed device-side check during the timed region")
    y_ref = o["y"].clone()

    # ---- the dominant operation: K steps of the step-by-step calls, events around moe_grouped_ffn ----
    for _ in range(args.warmup):
        step_by_step([torch.cuda.Event(enable_timing=True) for _ in range(2)])
    fevs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s0.record(stream)
    for i in range(args.steps):
        step_by_step(fevs[i])
    s1.record(stream)
    torch.cuda.synchronize()
    ffn_ms = statistics.mean(fevs[i][0].elapsed_time(fevs[i][1]) for i in range(args.steps))
    sbs_ms = s0.elapsed_time(s1) / args.steps
    if not torch.equal(o["y"], y_ref):
        raise RuntimeError("the step-by-step forward differs from moe_forward")

    # ---- end to end: pinned host x -> device, moe_forward, y -> pinned host ----
    # Every step copies its x in and its y out through pinned host memory.
    # As a serving loop runs it, the copies go on their own streams into two
    # alternating device buffers, so step i's copies overlap the compute of
    # steps i - 1 and i + 1; the timed region spans the first copy in to the
    # last copy out.
    x_host = cpu["x"].pin_memory()
    y_host = [torch.empty(T, H, dtype=dt).pin_memory() for _ in range(2)]
    x_buf = [torch.empty_like(dev["x"]) for _ in range(2)]
    y_buf = [torch.empty_like(o["y"]) for _ in range(2)]
    h2d, d2h = torch.cuda.Stream(), torch.cuda.Stream()
    fargs = [{"x": x_buf[b], "w_router": dev["w_router"], "router_bias": dev["router_bias"],
              "w_shared_gate": dev["w_shared_gate"], "w_gate_up": dev["w_gate_up"], "w_down": dev["w_down"],
              "ws_gate_up": dev["ws_gate_up"], "ws_down": dev["ws_down"], "y": y_buf[b]} for b in range(2)]
    ev = lambda: torch.cuda.Event()  # noqa: E731
    x_ready, x_free, y_ready, y_free = ([ev() for _ in range(2)] for _ in range(4))
    for b in range(2):  # both buffers start free
        x_free[b].record(stream)
        y_free[b].record(stream)

    def e2e_step(i):
        b = i & 1
        h2d.wait_event(x_free[b])
        with torch.cuda.stream(h2d):
            x_buf[b].copy_(x_host, non_blocking=True)
        x_ready[b].record(h2d)
        stream.wait_event(x_ready[b])
        stream.wait_event(y_free[b])
        moe.moe_forward(d, fargs[b], fws, stream)
        x_free[b].record(stream)
        y_ready[b].record(stream)
        d2h.wait_event(y_ready[b])
        with torch.cuda.stream(d2h):
            y_host[b].copy_(y_buf[b], non_blocking=True)
        y_free[b].record(d2h)

    for i in range(args.warmup):
        e2e_step(i)
    barrier(world)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    h2d.wait_event(e0)
    for i in range(args.steps):
        e2e_step(i)
    stream.wait_stream(d2h)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, world)
    if not torch.equal(y_buf[0], y_ref):
        raise RuntimeError("the end-to-end forward differs from the device-timed forward")

    peaks, peak_src = load_peaks()
    lb = layer_bytes_flops(T, H, E, k, Iw, Is, active)
    fb = ffn_bytes_flops(T, H, k, Iw, Is, active)
    hbm = float(peaks["hbm_gbs"])
    tf_sus = float(peaks.get("bf16_tflops_sustained", peaks["bf16_tflops"]))
    t_roof_ms = max(lb["bytes"] / (hbm * 1e9), lb["flops"] / (float(peaks["bf16_tflops"]) * 1e12)) * 1e3
    achieved = fb["bytes"] / (ffn_ms * 1e-3) / 1e9
    tokens_all = T * world
    line = {
        "metric": METRIC, "value": tokens_all / (ms * 1e-3), "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16" if cfg.dtype == "bf16" else "f32",
        "data": "synthetic (seeded N(0,1) inputs, N(0,0.02) weights)",
        "config": workload_config(cfg, active, world),
        "e2e": {"value": tokens_all / (e2e_ms * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2, "api": "moe_forward"},
        "gpu_launches": launches_per_forward(T, E) * args.steps,
        "roofline": {"kernel": "moe_grouped_ffn (gate_up+SwiGLU, down)", "bound": "hbm", "achieved": achieved,
                     "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "traffic": FFN_TRAFFIC["bytes"] if (kernel_sources_hash() == FFN_TRAFFIC["sources"] and
                                                        cfg.name == FFN_TRAFFIC["workload"]) else None,
                     "peak_source": peak_src, "ms_per_launch": ffn_ms,
                     "algorithmic_bytes": fb["bytes"]},
        "layer_roofline": {"bytes": lb["bytes"], "flops": lb["flops"], "roofline_ms": t_roof_ms,
                           "frac": t_roof_ms / ms, "peak_hbm_gbs": hbm, "peak_bf16_tflops": peaks["bf16_tflops"],
                           "peak_source": peak_src},
        "clocks": clk,
        "step_ms": percentiles([evs[i].elapsed_time(evs[i + 1]) for i in range(args.steps)]),
        "step_by_step": {"ms_per_step": sbs_ms, "api": "moe_route, moe_permute, moe_grouped_ffn, moe_combine",
                         "launches_per_step": LAUNCHES_PER_STEP_BY_STEP,
                         "note": "the timed loop of the roofline's moe_grouped_ffn launches"},
    }
    if not args.no_fwd_bwd and cfg.dtype == "bf16":
        del o, ws, fws
        torch.cuda.empty_cache()
        fb_cfg = I.CONFIGS[args.fwd_bwd_workload]
        assert (fb_cfg.H, fb_cfg.E, fb_cfg.I, fb_cfg.Is) == (H, E, Iw, Is), "fwd+bwd workload must share the layer"
        line["fwd_bwd"] = fwd_bwd_bench(fb_cfg, dev, args.steps, args.warmup, world, peaks)
    if world == 1 and not args.no_extra and cfg.name == "bf16_t8192":
        line["extra_forward"] = [extra_forward(n, dev, 50, 5, peaks) for n in ("bf16_t1024", "bf16_t16384_zipf")]
        line["etp_slice"] = etp_slice_bench(dev, 50, 5)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        W = {kk: v for kk, v in cpu.items() if kk not in ("x", "dy", "router_bias")}
        line["cpu_baseline"] = cpu_oracle_baseline(cfg, cpu["x"], W, cpu["router_bias"])
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
