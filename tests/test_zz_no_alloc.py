"""moe_permute_noalloc: the permutation for callers that cannot allocate.

Callers such as a custom operator hosted by another runtime (which owns the
device memory pool and passes only input and output buffers) or a loop that
must not call cudaMalloc (it can synchronise the device) cannot give
moe_permute its workspace.  moe_permute_noalloc keeps that scratch in a fixed
array inside the library.  This test calls it through the C ABI twice in a
row, with different sizes, and checks each result against moe_permute (the
permutation is integer work, so the bar is bit-exact), then checks that a
size beyond the fixed scratch is refused before any GPU work.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build

pytestmark = pytest.mark.gpu


def random_ids(T, E, k, seed):
    rng = np.random.default_rng(seed)
    return torch.as_tensor(np.stack([rng.permutation(E)[:k] for _ in range(T)]).astype(np.int32), device="cuda")


def outputs(T, E, k):
    return (torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -7, dtype=torch.int32, device="cuda"))


def test_noalloc_permute_matches_workspace_permute_twice():
    build.build()
    L = moe.lib()
    moe.moe_device_status(reset=True)
    # First call large, second smaller: the second must not see the first's scratch.
    for T, E, k, seed in [(6000, 512, 10, 1), (333, 64, 8, 2)]:
        ids = random_ids(T, E, k, seed)
        d = moe.make_dims(T, 256, E, k, 128, 128, moe.MOE_BF16)
        off, srt, pos = outputs(T, E, k)
        rc = L.moe_permute_noalloc(ctypes.byref(d), ctypes.c_void_p(ids.data_ptr()),
                                   ctypes.c_void_p(off.data_ptr()), ctypes.c_void_p(srt.data_ptr()),
                                   ctypes.c_void_p(pos.data_ptr()), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == 0, moe.status_string(rc)
        ref = moe.permute(ids, E)
        torch.cuda.synchronize()
        assert torch.equal(off, ref["expert_offsets"])
        assert torch.equal(srt, ref["sorted_route"])
        assert torch.equal(pos, ref["route_pos"])
    assert moe.moe_device_status(reset=True) == 0


def test_noalloc_permute_refuses_sizes_beyond_its_scratch():
    build.build()
    T, E, k = 40000, 1024, 16  # needs (1250 * 1024 + 1024) * 4 bytes > 4 MiB
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    off, srt, pos = outputs(T, E, k)
    d = moe.make_dims(T, 256, E, k, 128, 128, moe.MOE_BF16)
    with pytest.raises(moe.MoEError) as e:
        moe.moe_permute_noalloc(d, ids, off, srt, pos)
    assert e.value.status == -2
    torch.cuda.synchronize()
    assert int(off[0]) == -7  # nothing was written
