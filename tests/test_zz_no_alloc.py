"""moe_align_sort_noalloc, the sort for callers that cannot allocate device memory when they
need it (a serving engine whose device memory all belongs to its own pool, or a plugin entry
point given only input and output buffers): its scratch is a static device array inside the
library.  Called through the C ABI with ctypes, it must give exactly what the oracle's counting
sort and moe_align_sort give (integer results: bit-exact), on calls in a row that share the
array: a large problem with a bad id, a smaller clean one, an expert-parallel shard (ids of its
local experts) and an empty batch.

This file is collected last, so a run that stops at the first failure has run every other
test before it; it also passes alone in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu

KEYS = ("counts", "offsets", "sorted_ids", "tile_expert", "inv_route")


def _noalloc_via_c_abi(ids, prob, n_experts, block_m, dev):
    """Direct ctypes call of moe_align_sort_noalloc with torch-owned output buffers.
    n_experts: the experts the ids index (the shard's local count when prob is a shard)."""
    T, k = ids.shape
    cap = B.sorted_capacity(prob, block_m)
    tile_len = (cap + block_m - 1) // block_m
    out = dict(counts=torch.full((n_experts,), -7, dtype=torch.int32, device=dev),
               offsets=torch.full((n_experts + 1,), -7, dtype=torch.int32, device=dev),
               sorted_ids=torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev),
               tile_expert=torch.full((max(tile_len, 1),), -7, dtype=torch.int32, device=dev),
               inv_route=torch.full((max(T * k, 1),), -7, dtype=torch.int32, device=dev))
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    p = lambda t: ctypes.c_void_p(t.data_ptr()) if t.numel() else None
    rc = B.lib().moe_align_sort_noalloc(
        ctypes.byref(prob), block_m, p(ids), p(out["counts"]), p(out["offsets"]),
        p(out["sorted_ids"]), p(out["tile_expert"]), p(out["inv_route"]), p(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.MOE_OK, B.status_string(rc)
    out["sorted_ids"] = out["sorted_ids"][:cap]
    out["tile_expert"] = out["tile_expert"][:tile_len]
    out["inv_route"] = out["inv_route"][:T * k]
    return out, status


def _oracle_sort(ids_np, n_experts, block_m, cap):
    """The oracle's counting sort; an id outside [-1, E) is a padding route (the library's
    documented treatment, which also reports it in the status).  Its sorted_ids and
    tile_expert are extended with -1 to the library's capacity (a shard's capacity counts all
    E experts' padding)."""
    clean = np.where((ids_np >= -1) & (ids_np < n_experts), ids_np, -1).astype(np.int32)
    ref = oracle.align_sort(clean, n_experts, block_m)
    tile_len = (cap + block_m - 1) // block_m
    for key, n in (("sorted_ids", cap), ("tile_expert", tile_len)):
        v = ref[key]
        assert n >= v.size
        ref[key] = np.concatenate([v, np.full(n - v.size, -1, np.int32)])
    return ref


# (T, top_k, E, block_m, bad id, shard: (ep_num_local, ep_local_offset) or None)
CASES = [
    (4096, 8, 256, 1, 999, None),     # 128 chunks, a bad id: status set, route dropped
    (300, 4, 40, 16, None, None),     # fewer chunks and experts than the call before left
    (2000, 8, 256, 4, None, (32, 64)),  # a shard: ids are local (0..31) or -1
    (0, 8, 64, 8, None, None),        # empty batch: counts 0, every slot padding
]


def test_noalloc_sort_matches_oracle_and_workspace_sort(cuda_device):
    for T, k, E, block_m, bad, shard in CASES:
        n_loc, off = shard if shard else (0, 0)
        n_exp = n_loc or E
        ids = inputs.random_ids(T, k, n_exp, seed=T + E, pad_frac=0.05)
        if bad is not None:
            ids[5, 3] = bad
        prob = B.make_problem(T, 8, E, 8, k, ep_num_local=n_loc, ep_local_offset=off)
        cap = B.sorted_capacity(prob, block_m)
        ids_d = ids.to(cuda_device).contiguous()
        got, status = _noalloc_via_c_abi(ids_d, prob, n_exp, block_m, cuda_device)
        torch.cuda.synchronize()
        ref = _oracle_sort(ids.numpy(), n_exp, block_m, cap)
        for key in KEYS:
            assert np.array_equal(got[key].cpu().numpy(), ref[key]), (T, E, shard, key)
        want = B.MOE_ERR_BAD_EXPERT_ID if bad is not None else B.MOE_OK
        assert int(status.item()) == want
        if shard is None:  # the workspace sort on the same ids gives the same arrays
            ws = B.moe_align_sort(ids_d, E, block_m)
            torch.cuda.synchronize()
            for key in KEYS:
                assert torch.equal(got[key], ws[key]), (T, E, key)
            assert B.get_device_status(ws["workspace"]) == want


def test_noalloc_sort_rejects_bad_problems(cuda_device):
    ids = torch.zeros((16384, 8), dtype=torch.int32, device=cuda_device)  # 512 chunks x 1024
    d = ctypes.c_void_p(ids.data_ptr())
    prob = B.make_problem(16384, 8, 1024, 8, 8)
    rc = B.lib().moe_align_sort_noalloc(ctypes.byref(prob), 1, d, d, d, d, None, d, None, None)
    assert rc == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # a shard that runs past the last expert, and top_k beyond the kernels' limit
    prob = B.make_problem(64, 8, 256, 8, 8, ep_num_local=64, ep_local_offset=224)
    rc = B.lib().moe_align_sort_noalloc(ctypes.byref(prob), 1, d, d, d, d, None, d, None, None)
    assert rc == B.MOE_ERR_INVALID_ARG
    prob = B.make_problem(64, 8, 256, 8, 40)
    rc = B.lib().moe_align_sort_noalloc(ctypes.byref(prob), 1, d, d, d, d, None, d, None, None)
    assert rc == B.MOE_ERR_UNSUPPORTED
