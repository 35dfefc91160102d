"""moe_permute_noalloc: the permutation for callers that cannot allocate.

Callers such as a custom operator hosted by another runtime (which owns the
device memory pool and passes only input and output buffers) or a loop that
must not call cudaMalloc (it can synchronise the device) cannot give
moe_permute its workspace.  moe_permute_noalloc needs none: up to 2^20
routes it runs the one-launch cluster sort (no scratch), above that the
four-kernel sort with its scratch in a fixed array inside the library, in
128-route chunks where they fit the array and 512-route chunks where only
those do.  This test calls it through the C ABI, two calls in a row on each
form, and checks every result bit for bit against the oracle's counting sort
and against moe_permute (the permutation is integer work, so the bar is
bit-exact); then it checks that a size beyond the fixed array is refused
before any GPU work, with nothing written.

This file is collected last so that a run stopping at the first failure has
already run every other test; it also passes on its own in a fresh process.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import top_routed_grouped_gb300 as moe
from top_routed_grouped_gb300 import build

pytestmark = pytest.mark.gpu

SCRATCH = 4 << 20  # MOE_PERMUTE_NOALLOC_SCRATCH_BYTES


def scratch_bytes(R, E, chunk):
    return (-(-R // chunk) * E + E) * 4


def random_ids(T, E, k, seed):
    """k distinct experts per token, uniformly drawn."""
    rng = np.random.default_rng(seed)
    return np.argsort(rng.random((T, E), dtype=np.float32), axis=1)[:, :k].astype(np.int32)


def outputs(T, E, k):
    return (torch.full((E + 1,), -7, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -7, dtype=torch.int32, device="cuda"),
            torch.full((T * k,), -7, dtype=torch.int32, device="cuda"))


def call_noalloc(L, d, ids, off, srt, pos):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.moe_permute_noalloc(ctypes.byref(d), ctypes.c_void_p(ids.data_ptr()), ctypes.c_void_p(off.data_ptr()),
                                 ctypes.c_void_p(srt.data_ptr()), ctypes.c_void_p(pos.data_ptr()), stream)


# (T, E, k): two consecutive calls per form, the second smaller than the first
# (it must not see the first's scratch).
CASES = {
    "cluster": [(6000, 512, 10), (333, 64, 8)],
    "chunk128": [(150_000, 64, 10), (110_000, 64, 10)],    # > 2^20 routes, 128-route scratch fits
    "chunk512": [(300_000, 64, 8), (270_000, 64, 8)],      # 128-route scratch > 4 MiB, 512-route fits
}


@pytest.mark.parametrize("form", list(CASES))
def test_noalloc_permute_matches_oracle_twice(form):
    build.build()
    L = moe.lib()
    moe.moe_device_status(reset=True)
    for i, (T, E, k) in enumerate(CASES[form]):
        R = T * k
        if form == "cluster":
            assert R <= 1 << 20
        else:
            assert R > 1 << 20
            assert (scratch_bytes(R, E, 128) <= SCRATCH) == (form == "chunk128")
            assert scratch_bytes(R, E, 512) <= SCRATCH
        ids_np = random_ids(T, E, k, seed=100 * i + len(form))
        ids = torch.as_tensor(ids_np, device="cuda")
        d = moe.make_dims(T, 256, E, k, 128, 128, moe.MOE_BF16)
        off, srt, pos = outputs(T, E, k)
        rc = call_noalloc(L, d, ids, off, srt, pos)
        assert rc == 0, moe.status_string(rc)
        torch.cuda.synchronize()
        r_off, r_srt, r_pos = oracle.permute(ids_np, E)
        np.testing.assert_array_equal(off.cpu().numpy(), r_off)
        np.testing.assert_array_equal(srt.cpu().numpy(), r_srt)
        np.testing.assert_array_equal(pos.cpu().numpy(), r_pos)
        ref = moe.permute(ids, E)
        assert torch.equal(off, ref["expert_offsets"])
        assert torch.equal(srt, ref["sorted_route"])
        assert torch.equal(pos, ref["route_pos"])
    assert moe.moe_device_status(reset=True) == 0


def test_noalloc_permute_refuses_sizes_beyond_its_scratch():
    build.build()
    L = moe.lib()
    T, E, k = 70_000, 1024, 16  # 1.12 M routes: (2188 * 1024 + 1024) * 4 bytes > 4 MiB even in 512-route chunks
    assert T * k > 1 << 20 and scratch_bytes(T * k, E, 512) > SCRATCH
    ids = torch.zeros(T, k, dtype=torch.int32, device="cuda")
    off, srt, pos = outputs(T, E, k)
    d = moe.make_dims(T, 256, E, k, 128, 128, moe.MOE_BF16)
    assert call_noalloc(L, d, ids, off, srt, pos) == -2  # MOE_ERR_UNSUPPORTED
    torch.cuda.synchronize()
    for buf in (off, srt, pos):  # nothing was written
        assert bool((buf == -7).all())
    # moe_permute's argument checks apply too: a bf16 layer with H not a multiple of 256
    bad = moe.make_dims(16, 100, 64, 4, 128, 128, moe.MOE_BF16)
    ids16 = torch.zeros(16, 4, dtype=torch.int32, device="cuda")
    o16 = outputs(16, 64, 4)
    assert call_noalloc(L, bad, ids16, *o16) == -2
    torch.cuda.synchronize()
    for buf in o16:
        assert bool((buf == -7).all())
