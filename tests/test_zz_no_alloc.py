"""moe_align_sort_noalloc, the sort for callers that cannot allocate device memory when they
need it (a serving engine whose device memory all belongs to its own pool, or a plugin entry
point given only input and output buffers): its scratch is a static device array inside the
library.  Called through the C ABI with ctypes, it must give exactly what moe_align_sort
gives (integer results: bit-exact), on two calls in a row that share the array.

This file is collected last, so a run that stops at the first failure has run every other
test before it; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "sorted_ids", "tile_expert", "inv_route")


def _noalloc_via_c_abi(ids, E, block_m, dev):
    """Direct ctypes call of moe_align_sort_noalloc with torch-owned output buffers."""
    T, k = ids.shape
    prob = B.make_problem(T, 8, E, 8, k)
    cap = T * k + E * (block_m - 1)
    tile_len = (cap + block_m - 1) // block_m
    out = dict(counts=torch.empty(E, dtype=torch.int32, device=dev),
               offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
               sorted_ids=torch.empty(max(cap, 1), dtype=torch.int32, device=dev),
               tile_expert=torch.empty(max(tile_len, 1), dtype=torch.int32, device=dev),
               inv_route=torch.empty(max(T * k, 1), dtype=torch.int32, device=dev))
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = B.lib().moe_align_sort_noalloc(
        ctypes.byref(prob), block_m, p(ids), p(out["counts"]), p(out["offsets"]),
        p(out["sorted_ids"]), p(out["tile_expert"]), p(out["inv_route"]), p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.MOE_OK, B.status_string(rc)
    out["sorted_ids"] = out["sorted_ids"][:cap]
    out["tile_expert"] = out["tile_expert"][:tile_len]
    out["inv_route"] = out["inv_route"][:T * k]
    return out, status


def test_noalloc_sort_matches_workspace_sort_twice(cuda_device):
    # First call: a large sort with a bad id (sets the status); second call: a different, clean
    # problem that reads fewer chunks and experts than the first left in the shared array.
    cases = [(4096, 8, 256, 1, 999), (300, 4, 40, 16, None)]
    for T, k, E, block_m, bad in cases:
        ids = inputs.random_ids(T, k, E, seed=T + E, pad_frac=0.05)
        if bad is not None:
            ids[5, 3] = bad
        ids = ids.to(cuda_device)
        got, status = _noalloc_via_c_abi(ids, E, block_m, cuda_device)
        ref = B.moe_align_sort(ids, E, block_m)
        torch.cuda.synchronize()
        for key in KEYS:
            assert torch.equal(got[key], ref[key]), (T, E, key)
        want = B.MOE_ERR_BAD_EXPERT_ID if bad is not None else B.MOE_OK
        assert int(status.item()) == want
        assert B.get_device_status(ref["workspace"]) == want


def test_noalloc_sort_rejects_oversized_problem(cuda_device):
    ids = torch.zeros((16384, 8), dtype=torch.int32, device=cuda_device)  # 512 chunks x 1024
    prob = B.make_problem(16384, 8, 1024, 8, 8)
    d = ctypes.c_void_p(ids.data_ptr())
    rc = B.lib().moe_align_sort_noalloc(ctypes.byref(prob), 1, d, d, d, d, None, d, None, None)
    assert rc == B.MOE_ERR_WORKSPACE_TOO_SMALL
