"""Expert tensor parallelism (ETP): the intermediate dimension split across ranks.

RL-Kernel PR #557 "What", bullet "Fail closed" (EP 1 runs every expert
expert-tensor-parallel over 4 ranks) and the embedded #503 commit message,
bullet "TP4 block" (every expert on every rank, partial results reduced
across ranks).  Rank r holds, for every expert, the gate and up rows of its
feature slice [i0, i1) of I and the matching columns of W_down, and the same
slice layout for the shared expert's Is.  Routing and the permutation are
replicated.  Because Yr = sum_i h_i W_down[:, i], each rank's down
projection is a partial sum of every row (``moe_grouped_ffn_etp``, FP32,
unrounded).  The partials are exchanged by a byte-copy all_gather (as PR
#557 "What" exchanges rows) and every rank sums them in rank order with one
rounding (``moe_etp_reduce``), then combines locally.

``forward_simulated`` runs the ranks one after another on one GPU;
``exchange_partials`` is the gather for a real process group.
"""
from __future__ import annotations

from typing import Sequence

import top_routed_grouped_gb300 as moe

GRANULE = 128  # feature-slice granularity of the bf16 kernels (their tile of I)


def feature_ranges(width: int, world: int, granule: int = GRANULE) -> list[tuple[int, int]]:
    """Contiguous, balanced slices [i0, i1) of `width` features, each a
    multiple of `granule` wide; every rank gets at least one granule."""
    if world <= 0 or width <= 0 or granule <= 0:
        raise ValueError("need width, world and granule > 0")
    if width % granule:
        raise ValueError(f"width {width} is not a multiple of {granule}")
    units = width // granule
    if units < world:
        raise ValueError(f"{width} features give fewer than {world} slices of {granule}")
    q, r = divmod(units, world)
    out, i = [], 0
    for rank in range(world):
        n = (q + (1 if rank < r else 0)) * granule
        out.append((i, i + n))
        i += n
    return out


def slice_gate_up(w, i0: int, i1: int):
    """[..., 2I, H] gate/up weight (gate rows first) -> [..., 2 (i1 - i0), H]
    holding gate rows i0..i1-1 then up rows i0..i1-1."""
    import torch
    I2 = w.shape[-2]
    I = I2 // 2
    if I2 % 2 or not 0 <= i0 < i1 <= I:
        raise ValueError("bad feature slice")
    return torch.cat([w[..., i0:i1, :], w[..., I + i0:I + i1, :]], dim=-2).contiguous()


def slice_down(w, i0: int, i1: int):
    """[..., H, I] down weight -> its columns i0..i1-1."""
    if not 0 <= i0 < i1 <= w.shape[-1]:
        raise ValueError("bad feature slice")
    return w[..., i0:i1].contiguous()


def rank_weights(w_gate_up, w_down, ws_gate_up, ws_down, rng, rng_sh):
    """The weights rank (rng, rng_sh) holds: routed experts' slice rng of I,
    the shared expert's slice rng_sh of Is."""
    return (slice_gate_up(w_gate_up, *rng), slice_down(w_down, *rng), slice_gate_up(ws_gate_up, *rng_sh),
            slice_down(ws_down, *rng_sh))


def forward_simulated(x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, k: int, world: int,
                      router_bias=None, stream=None, fused: bool = False):
    """The layer forward with I (and Is) split over `world` ranks, run on one
    GPU: replicated routing and permutation; per rank, its weight slices and
    one moe_grouped_ffn_etp call (FP32 partials; ``fused``: the
    moe_grouped_ffn_etp_fused form, for 128-feature slices); the rank-ordered
    reduction; the combine.  Returns dict(y, y_routed, y_shared, parts, ranges)."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    I, Is = w_down.shape[-1], ws_down.shape[-1]
    granule = 4 if x.dtype == torch.float32 else GRANULE  # the FP32 kernels take any multiple of 4
    ranges, ranges_sh = feature_ranges(I, world, granule), feature_ranges(Is, world, granule)
    r = moe.route(x, w_router, w_shared_gate, k, router_bias=router_bias, stream=stream)
    pm = moe.permute(r["topk_ids"], E, stream=stream)
    parts_r, parts_s = [], []
    for rng, rng_sh in zip(ranges, ranges_sh):
        wg, wd, wsg, wsd = rank_weights(w_gate_up, w_down, ws_gate_up, ws_down, rng, rng_sh)
        d = moe.make_dims(T, H, E, k, rng[1] - rng[0], rng_sh[1] - rng_sh[0], x.dtype)
        pr = torch.empty(T * k, H, dtype=torch.float32, device=x.device)
        ps = torch.empty(T, H, dtype=torch.float32, device=x.device)
        if fused:
            moe.moe_grouped_ffn_etp_fused(d, x, pm["expert_offsets"], pm["sorted_route"], wg, wd, wsg, wsd, pr, ps,
                                          moe.workspace(d, "grouped_ffn", x.device), stream)
        else:
            moe.moe_grouped_ffn_etp(d, x, pm["expert_offsets"], pm["sorted_route"], wg, wd, wsg, wsd, pr, ps, None,
                                    moe.workspace(d, "grouped_ffn", x.device), stream)
        parts_r.append(pr)
        parts_s.append(ps)
    d = moe.make_dims(T, H, E, k, I, Is, x.dtype)
    y_routed = torch.empty(T * k, H, dtype=x.dtype, device=x.device)
    y_shared = torch.empty(T, H, dtype=x.dtype, device=x.device)
    moe.moe_etp_reduce(d, parts_r, parts_s, y_routed, y_shared, stream)
    y = torch.empty(T, H, dtype=x.dtype, device=x.device)
    moe.moe_combine(d, y_routed, y_shared, r["topk_w"], r["shared_sig"], y, stream)
    return {"y": y, "y_routed": y_routed, "y_shared": y_shared, "parts": (parts_r, parts_s),
            "ranges": (ranges, ranges_sh), "route": r}


def exchange_partials(partial, group=None) -> list:
    """All-gather of one equally shaped partial per rank (a byte copy):
    returns every rank's partial, in rank order."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = [torch.empty_like(partial) for _ in range(world)]
    dist.all_gather(out, partial.contiguous(), group=group)
    return out


def check_ranges(ranges: Sequence[tuple[int, int]], width: int, granule: int = GRANULE) -> None:
    """Fail closed unless the slices are contiguous, ordered, granule-aligned
    and cover [0, width): every feature must belong to exactly one rank."""
    i = 0
    for rank, (a, b) in enumerate(ranges):
        if a != i or b <= a or a % granule or b % granule:
            raise ValueError(f"rank {rank}: slice [{a}, {b}) does not continue at {i} in steps of {granule}")
        i = b
    if i != width:
        raise ValueError(f"features [{i}, {width}) have no owner")
