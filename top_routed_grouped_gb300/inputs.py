"""Seeded synthetic inputs for the MoE layer.

This module holds no arithmetic of the layer itself: it only draws the
inputs (activations, weights, upstream gradient, router logit bias) from
fixed seeds, so that the CUDA path, the tests and the CPU oracle all read the
same bits.  Normals come from numpy's PCG64 generator in fixed-size chunks,
each chunk with its own ``SeedSequence`` spawn key, so the values do not
depend on the number of threads or on the machine (x86-64 and AArch64 give
identical arrays).  fp32 draws are rounded to bf16 with round-to-nearest-even.

Workloads (the layer of SkyRL PR #2513 "What": 512 routed experts, top-10,
plus a shared expert; hidden and intermediate sizes are this build's choice):

=====================  ======  ====  ===  ==  ===  ===  =====  ====================
name                   T       H     E    k   I    Is   dtype  notes
=====================  ======  ====  ===  ==  ===  ===  =====  ====================
tiny_f32               64      256   16   4   128  128  f32    FP32 throughout
bf16_t1024             1024    2048  512  10  512  512  bf16   near-uniform routing
bf16_t8192             8192    2048  512  10  512  512  bf16   one 8K packed sequence
bf16_t16384_zipf       16384   2048  512  10  512  512  bf16   Zipf(1.1) logit bias
bf16_t4096_fwdbwd      4096    2048  512  10  512  512  bf16   forward + backward
bf16_e64_t512          512     2048  64   10  512  512  bf16   small profiling case:
                                                               80 routes per expert
                                                               as at T=4096, ~1 GB
bf16_smoke             300     256   256  4   256  512  bf16   smallest shape on every
                                                               tensor-core kernel
                                                               (forward and backward)
bf16_e64_zipf_t4096    4096    2048  64   10  512  512  bf16   small profiling case of
                                                               long skewed segments:
                                                               Zipf bias over 64 experts
                                                               (8 empty, beta 0.3: the
                                                               largest gets 2304 rows)
=====================  ======  ====  ===  ==  ===  ===  =====  ====================

Distributions: x ~ N(0,1); every weight ~ N(0, 0.02) (the router weight is
kept in fp32 for every dtype); upstream gradient dy ~ N(0,1).  Seeds: 0 for
inputs and weights, 2 for dy, 3 for the random expert order of the Zipf bias.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, replace

import numpy as np
import torch

# Stream ids: one independent random stream per tensor.
_STREAM = {"x": 1, "w_router": 2, "w_shared_gate": 3, "w_gate_up": 4, "w_down": 5,
           "ws_gate_up": 6, "ws_down": 7, "dy": 8}
_CHUNK = 1 << 22
WEIGHT_STD = 0.02

# Zipf bias strength for bf16_t16384_zipf.  Chosen by bisection so that the
# busiest expert receives about 20x the mean load R/E; the script
# tests/golden/make_zipf_bias.py recomputes it with the oracle's routing and
# records the realised loads in tests/golden/zipf_bias.json.
ZIPF_S = 1.1
ZIPF_EMPTY = 64
ZIPF_BETA = 0.3065471947193146


@dataclass(frozen=True)
class MoEConfig:
    name: str
    T: int
    H: int
    E: int
    k: int
    I: int
    Is: int
    dtype: str  # "f32" or "bf16"
    zipf: bool = False
    backward: bool = False
    zipf_beta: float = 0.3065471947193146  # ZIPF_BETA
    zipf_empty: int = 64                   # ZIPF_EMPTY

    @property
    def R(self) -> int:
        return self.T * self.k

    @property
    def torch_dtype(self) -> torch.dtype:
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    def with_tokens(self, T: int) -> "MoEConfig":
        return replace(self, T=T)


CONFIGS = {
    "tiny_f32": MoEConfig("tiny_f32", 64, 256, 16, 4, 128, 128, "f32"),
    "bf16_t1024": MoEConfig("bf16_t1024", 1024, 2048, 512, 10, 512, 512, "bf16"),
    "bf16_t8192": MoEConfig("bf16_t8192", 8192, 2048, 512, 10, 512, 512, "bf16"),
    "bf16_t16384_zipf": MoEConfig("bf16_t16384_zipf", 16384, 2048, 512, 10, 512, 512, "bf16", zipf=True),
    "bf16_t4096_fwdbwd": MoEConfig("bf16_t4096_fwdbwd", 4096, 2048, 512, 10, 512, 512, "bf16", backward=True),
    "bf16_e64_t512": MoEConfig("bf16_e64_t512", 512, 2048, 64, 10, 512, 512, "bf16", backward=True),
    "bf16_smoke": MoEConfig("bf16_smoke", 300, 256, 256, 4, 256, 512, "bf16", backward=True),
    "bf16_e64_zipf_t4096": MoEConfig("bf16_e64_zipf_t4096", 4096, 2048, 64, 10, 512, 512, "bf16", zipf=True,
                                     zipf_beta=0.3, zipf_empty=8),
}


def _threads() -> int:
    try:
        return max(1, min(32, len(os.sched_getaffinity(0))))
    except AttributeError:  # pragma: no cover
        return max(1, min(32, os.cpu_count() or 1))


def normal(shape, seed: int, stream: int, std: float = 1.0, dtype: torch.dtype = torch.float32) -> torch.Tensor:
    """N(0, std^2) tensor on the CPU, drawn chunk by chunk from fixed seeds."""
    n = int(np.prod(shape)) if len(shape) else 1
    out = torch.empty(n, dtype=dtype)
    n_chunks = (n + _CHUNK - 1) // _CHUNK

    def fill(c: int) -> None:
        lo, hi = c * _CHUNK, min(n, (c + 1) * _CHUNK)
        ss = np.random.SeedSequence(entropy=seed, spawn_key=(stream, c))
        a = np.random.Generator(np.random.PCG64(ss)).standard_normal(hi - lo, dtype=np.float32)
        if std != 1.0:
            a *= np.float32(std)
        out[lo:hi] = torch.from_numpy(a).to(dtype)

    if n_chunks <= 1:
        for c in range(n_chunks):
            fill(c)
    else:
        with ThreadPoolExecutor(min(_threads(), n_chunks)) as ex:
            list(ex.map(fill, range(n_chunks)))
    return out.reshape(shape)


def zipf_bias(E: int, beta: float = ZIPF_BETA, s: float = ZIPF_S, n_empty: int = ZIPF_EMPTY,
              seed: int = 3) -> torch.Tensor:
    """Per-expert router logit bias (fp32).

    A random expert order is drawn (seed 3).  The first ``n_empty`` experts in
    that order get -30 (never selected).  The remaining ones, ranked r = 1, 2,
    ..., get beta * ln(r^-s), so lower ranks are preferred in a Zipf-like way.
    """
    order = np.random.default_rng(seed).permutation(E)
    b = np.empty(E, np.float64)
    b[order[:n_empty]] = -30.0
    ranks = np.arange(1, E - n_empty + 1, dtype=np.float64)
    b[order[n_empty:]] = -s * beta * np.log(ranks)
    return torch.from_numpy(b.astype(np.float32))


def make_inputs(cfg: MoEConfig, seed: int = 0, T: int | None = None, device: str | torch.device = "cpu",
                with_dy: bool | None = None, beta: float | None = None) -> dict:
    """All layer inputs for ``cfg`` (``T`` overrides the token count).

    Weights do not depend on T, and x / dy for T rows are the leading T rows
    of the draw for any larger T (chunks are laid out by element index).
    """
    T = cfg.T if T is None else T
    dt = cfg.torch_dtype
    H, E, I, Is = cfg.H, cfg.E, cfg.I, cfg.Is
    d = {
        "x": normal((T, H), seed, _STREAM["x"], 1.0, dt),
        "w_router": normal((E, H), seed, _STREAM["w_router"], WEIGHT_STD, torch.float32),
        "w_shared_gate": normal((H,), seed, _STREAM["w_shared_gate"], WEIGHT_STD, dt),
        "w_gate_up": normal((E, 2 * I, H), seed, _STREAM["w_gate_up"], WEIGHT_STD, dt),
        "w_down": normal((E, H, I), seed, _STREAM["w_down"], WEIGHT_STD, dt),
        "ws_gate_up": normal((2 * Is, H), seed, _STREAM["ws_gate_up"], WEIGHT_STD, dt),
        "ws_down": normal((H, Is), seed, _STREAM["ws_down"], WEIGHT_STD, dt),
        "router_bias": zipf_bias(E, cfg.zipf_beta if beta is None else beta, n_empty=cfg.zipf_empty)
        if cfg.zipf else None,
    }
    if with_dy or (with_dy is None and cfg.backward):
        d["dy"] = normal((T, H), 2, _STREAM["dy"], 1.0, dt)
    if str(device) != "cpu":
        d = {key: (v.to(device) if v is not None else None) for key, v in d.items()}
    return d


def shuffled_order(T: int, seed: int = 1) -> torch.Tensor:
    """Seeded permutation of the T rows (batch-invariance check)."""
    return torch.from_numpy(np.random.default_rng(seed).permutation(T).astype(np.int64))


def ragged_batches(T: int, b: int) -> list[tuple[int, int]]:
    """Consecutive [lo, hi) chunks of size b; the last one may be shorter."""
    return [(lo, min(T, lo + b)) for lo in range(0, T, b)]
