"""Expert partition (EP) of the MoE layer.

RL-Kernel PR #557 "EP4 distributed logprob parity", section "What": the
experts are split into contiguous ranges, one per rank; every rank computes
the same routes (the router and the permutation are replicated), runs the
grouped FFN only for the segments of its own experts, and one all_gather of
the routed rows (a byte copy) gives every rank all rows; the ordered combine
is then local.  A route slot whose expert no rank owns fails closed.

Here the routed rows of one rank are one contiguous block of the sorted row
order (``moe_grouped_ffn_ep`` writes sorted order), so the exchange copies
one block per rank.  The shared expert is replicated: every rank computes it
for all tokens.

The backward mirrors it (``moe_backward_ep``): every rank computes the
replicated parts (combine backward, shared expert, router and gate
gradients), the weight gradients of its own experts (they stay local) and
the routed input gradients dXr of its rows, one contiguous block of the
sorted order; the same exchange of dXr blocks gives every rank all rows,
and dx (summed in ascending expert order) is again local.

``forward_simulated`` and ``backward_simulated`` run the ranks one after
another on one GPU (their blocks are disjoint rows of one buffer, which is
what the exchange would assemble); ``exchange_rows`` is the exchange for a
real process group (any row type: routed outputs or their gradients).
"""
from __future__ import annotations

from typing import Sequence

import top_routed_grouped_gb300 as moe


def expert_ranges(E: int, world: int) -> list[tuple[int, int]]:
    """Contiguous, balanced expert ranges [e_begin, e_end) of the ranks."""
    if world <= 0 or E <= 0:
        raise ValueError("need E > 0 and world > 0")
    q, r = divmod(E, world)
    out, e = [], 0
    for rank in range(world):
        n = q + (1 if rank < r else 0)
        out.append((e, e + n))
        e += n
    return out


def check_partition(ranges: Sequence[tuple[int, int]], E: int) -> None:
    """Fail closed unless the ranges are contiguous, ordered, disjoint and
    cover [0, E): every route slot must have exactly one owner."""
    e = 0
    for rank, (b, t) in enumerate(ranges):
        if b != e or t < b:
            raise ValueError(f"rank {rank}: range [{b}, {t}) leaves experts [{e}, {b}) without an owner"
                             if b > e else f"rank {rank}: range [{b}, {t}) overlaps or is reversed")
        e = t
    if e != E:
        raise ValueError(f"experts [{e}, {E}) have no owner")


def owner_of(expert: int, ranges: Sequence[tuple[int, int]]) -> int:
    for rank, (b, t) in enumerate(ranges):
        if b <= expert < t:
            return rank
    raise ValueError(f"expert {expert} has no owner")


def rank_rows(offsets_host: Sequence[int], rng: tuple[int, int]) -> tuple[int, int]:
    """Sorted rows [r0, r1) that the rank owning experts `rng` produces."""
    return int(offsets_host[rng[0]]), int(offsets_host[rng[1]])


def forward_simulated(x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down, k: int, world: int,
                      ranges=None, router_bias=None, stream=None, save_for_backward: bool = False):
    """The layer forward with the experts split over `world` ranks, run on one
    GPU: replicated routing and permutation, one moe_grouped_ffn_ep call per
    rank with only that rank's expert weights, the shared expert on every
    rank (identical), and the local ordered combine.  Returns dict(y,
    y_sorted, y_shared, ranges, route, permute) and, with `save_for_backward`, the
    activations the backward needs (`saved`; each rank writes the rows of its
    own experts)."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    ranges = expert_ranges(E, world) if ranges is None else list(ranges)
    check_partition(ranges, E)
    r = moe.route(x, w_router, w_shared_gate, k, router_bias=router_bias, stream=stream)
    pm = moe.permute(r["topk_ids"], E, stream=stream)
    d = moe.dims_of(x, w_router, w_gate_up, ws_gate_up, k)
    y_sorted = torch.empty(T * k, H, dtype=x.dtype, device=x.device)
    y_shared = torch.empty(T, H, dtype=x.dtype, device=x.device)
    saved = None
    if save_for_backward:
        R, dt, dev = T * k, x.dtype, x.device
        saved = {"gu": torch.empty(R, 2 * d.I, dtype=dt, device=dev), "h": torch.empty(R, d.I, dtype=dt, device=dev),
                 "gu_shared": torch.empty(T, 2 * d.Is, dtype=dt, device=dev),
                 "h_shared": torch.empty(T, d.Is, dtype=dt, device=dev)}
    ws = moe.workspace(d, "grouped_ffn", x.device)
    for rank, (b, e) in enumerate(ranges):
        # Each rank holds only its experts' weights (views of the full arrays here).
        moe.moe_grouped_ffn_ep(d, b, e, 1, x, pm["expert_offsets"], pm["sorted_route"],
                               w_gate_up[b:e] if e > b else None, w_down[b:e] if e > b else None, ws_gate_up,
                               ws_down, y_sorted, y_shared, saved, ws, stream)
    y = torch.empty(T, H, dtype=x.dtype, device=x.device)
    moe.moe_combine_sorted(d, y_sorted, pm["route_pos"], y_shared, r["topk_w"], r["shared_sig"], y, stream)
    return {"y": y, "y_sorted": y_sorted, "y_shared": y_shared, "ranges": ranges, "route": r, "permute": pm,
            "saved": saved}


def backward_simulated(fwd: dict, dy, x, w_router, w_shared_gate, w_gate_up, w_down, ws_gate_up, ws_down,
                       stream=None):
    """The expert-partitioned backward, run on one GPU from the dict
    ``forward_simulated(..., save_for_backward=True)`` returned: every rank
    runs phase 1 of ``moe_backward_ep`` with its own workspace, expert weights
    and weight-gradient arrays; the ranks' row blocks of dXr land in one
    buffer (what ``exchange_rows`` would assemble); then every rank runs phase
    2.  Returns, per rank, its dx and its replicated gradients, plus the
    expert weight gradients assembled from the ranks' local arrays."""
    import torch
    T, H = x.shape
    E = w_router.shape[0]
    k = fwd["route"]["topk_ids"].shape[1]
    d = moe.dims_of(x, w_router, w_gate_up, ws_gate_up, k)
    dev, f32 = x.device, torch.float32
    I, Is = d.I, d.Is
    r, pm = fwd["route"], fwd["permute"]
    dw_gate_up = torch.empty(E, 2 * I, H, dtype=f32, device=dev)
    dw_down = torch.empty(E, H, I, dtype=f32, device=dev)
    dxr = torch.empty(T * k, H, dtype=f32, device=dev)
    ranks = []
    for b, e in fwd["ranges"]:
        out = {"dx": torch.empty(T, H, dtype=x.dtype, device=dev),
               "dw_router": torch.empty(E, H, dtype=f32, device=dev),
               "dw_shared_gate": torch.empty(H, dtype=f32, device=dev),
               "dws_gate_up": torch.empty(2 * Is, H, dtype=f32, device=dev),
               "dws_down": torch.empty(H, Is, dtype=f32, device=dev),
               "dlogit": torch.empty(T, k, dtype=f32, device=dev),
               "dz": torch.empty(T, dtype=f32, device=dev)}
        local = dict(w_gate_up=w_gate_up[b:e] if e > b else None, w_down=w_down[b:e] if e > b else None,
                     dw_gate_up=dw_gate_up[b:e] if e > b else None, dw_down=dw_down[b:e] if e > b else None)
        args = dict(out, **local, x=x, w_router=w_router, w_shared_gate=w_shared_gate, ws_gate_up=ws_gate_up,
                    ws_down=ws_down, dy=dy, saved=fwd["saved"], topk_ids=r["topk_ids"], topk_w=r["topk_w"],
                    shared_sig=r["shared_sig"], expert_offsets=pm["expert_offsets"],
                    sorted_route=pm["sorted_route"], route_pos=pm["route_pos"], y_routed=fwd["y_sorted"],
                    y_shared=fwd["y_shared"])
        ranks.append({"range": (b, e), "out": out, "args": args, "ws": moe.workspace(d, "backward", dev)})
    for rk in ranks:
        b, e = rk["range"]
        moe.moe_backward_ep(d, b, e, 1, rk["args"], dxr, rk["ws"], stream)
    for rk in ranks:
        b, e = rk["range"]
        moe.moe_backward_ep(d, b, e, 2, rk["args"], dxr, rk["ws"], stream)
    return {"ranks": [rk["out"] for rk in ranks], "dw_gate_up": dw_gate_up, "dw_down": dw_down, "dxr": dxr}


def exchange_rows(y_sorted, offsets_host: Sequence[int], ranges: Sequence[tuple[int, int]], group=None):
    """All-gather of the routed rows: rank i owns sorted rows
    [offsets[b_i], offsets[e_i]) of `y_sorted` (filled locally); afterwards
    every rank holds every row.  Blocks have different lengths, so each is
    padded to the longest for one all_gather, then copied into place (bytes
    only: no arithmetic on the rows)."""
    import torch
    import torch.distributed as dist
    world = dist.get_world_size(group)
    rank = dist.get_rank(group)
    if len(ranges) != world:
        raise ValueError("one expert range per rank")
    E = ranges[-1][1]
    check_partition(ranges, E)
    blocks = [rank_rows(offsets_host, rg) for rg in ranges]
    longest = max(1, max(r1 - r0 for r0, r1 in blocks))
    H = y_sorted.shape[1]
    mine = torch.zeros(longest, H, dtype=y_sorted.dtype, device=y_sorted.device)
    r0, r1 = blocks[rank]
    mine[: r1 - r0] = y_sorted[r0:r1]
    gathered = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(gathered, mine, group=group)
    for i, (b0, b1) in enumerate(blocks):
        if i != rank:
            y_sorted[b0:b1] = gathered[i][: b1 - b0]
    return y_sorted
