"""Router and expert sort on the GPU vs the oracle: ids, sort order and inverse map bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from helpers import check_ids_against_plain_selection, oracle_route, run_route
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload
ROUTE_CASES = [
    W("softmax-e8-k2", T=4, H=128, E=8, F=64, top_k=2),
    W("softmax-e128-k8", T=512, H=64, E=128, F=64, top_k=8),
    W("softmax-e128-k8-norenorm", T=300, H=64, E=128, F=64, top_k=8, renormalize=False),
    W("softmax-e40-k3-rsf", T=77, H=64, E=40, F=64, top_k=3, routed_scaling_factor=1.7),
    W("sigmoid-bias-e384-k8", T=512, H=64, E=384, F=64, top_k=8, scoring_func="sigmoid",
      bias_std=0.1, routed_scaling_factor=2.827),
    W("sigmoid-nobias-e64-k6-norenorm", T=100, H=64, E=64, F=64, top_k=6,
      scoring_func="sigmoid", renormalize=False),
    W("grouped-e256-g8-k4", T=4096, H=64, E=256, F=64, top_k=8, scoring_func="sigmoid",
      bias_std=0.1, num_expert_group=8, topk_group=4, routed_scaling_factor=2.5),
    W("grouped-e96-g6-k2", T=33, H=64, E=96, F=64, top_k=5, scoring_func="sigmoid",
      bias_std=0.1, num_expert_group=6, topk_group=2),
    W("wide-e1024-k32", T=40, H=64, E=1024, F=64, top_k=32),
    W("e1-k1", T=5, H=64, E=1, F=64, top_k=1),
]


@pytest.mark.parametrize("w", ROUTE_CASES, ids=lambda w: w.name)
def test_route_matches_oracle(w, cuda_device):
    d = inputs.generate(w, seed=0, device=cuda_device)
    ids, wts = run_route(w, d)
    torch.cuda.synchronize()
    r_ids, r_w, _ = oracle_route(w, d)
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    np.testing.assert_allclose(wts.cpu().numpy(), r_w, rtol=2e-6, atol=1e-7)
    check_ids_against_plain_selection(w, d, ids, what=f"route {w.name}")


def test_route_ties_go_to_lower_id(cuda_device):
    g = torch.zeros((3, 64), dtype=torch.float32, device=cuda_device)
    g[1, 10:20] = 1.0
    ids, w = B.moe_route(g, 4)
    assert ids[0].tolist() == [0, 1, 2, 3]
    assert ids[1].tolist() == [10, 11, 12, 13]
    b = torch.zeros(64, dtype=torch.float32, device=cuda_device)
    ids2, _ = B.moe_route(g, 4, "sigmoid", correction_bias=b, num_expert_group=8, topk_group=2)
    r = oracle.route(g.cpu().numpy(), 4, oracle.SIGMOID, True, 8, 2, 1.0, b.cpu().numpy())
    assert np.array_equal(ids2.cpu().numpy(), r[0])


SORT_CASES = [
    (1, 8, 8, 1, 0.0), (5, 4, 16, 1, 0.3), (300, 4, 10, 16, 0.1), (4096, 8, 256, 1, 0.0),
    (4096, 8, 384, 128, 0.05), (512, 8, 128, 64, 0.0), (33, 8, 1024, 1, 0.0), (0, 8, 16, 1, 0.0),
]


@pytest.mark.parametrize("T,k,E,block_m,pad", SORT_CASES)
def test_align_sort_matches_oracle(T, k, E, block_m, pad, cuda_device):
    ids = inputs.random_ids(T, k, E, seed=T + E, pad_frac=pad)
    g = B.moe_align_sort(ids.to(cuda_device), E, block_m)
    ref = oracle.align_sort(ids.numpy(), E, block_m)
    for key in ("counts", "offsets", "sorted_ids", "tile_expert", "inv_route"):
        assert np.array_equal(g[key].cpu().numpy(), ref[key]), key
    assert B.get_device_status(g["workspace"]) == B.MOE_OK


def test_align_sort_flags_bad_expert_id(cuda_device):
    ids = inputs.random_ids(20, 4, 16, seed=1)
    ids[3, 2] = 999
    ids[7, 0] = -7
    g = B.moe_align_sort(ids.to(cuda_device), 16, 1)
    assert B.get_device_status(g["workspace"]) == B.MOE_ERR_BAD_EXPERT_ID
    assert B.get_device_status(g["workspace"]) == B.MOE_OK  # read clears
    # the bad routes are treated as padding
    clean = ids.clone()
    clean[3, 2] = -1
    clean[7, 0] = -1
    ref = oracle.align_sort(clean.numpy(), 16, 1)
    assert np.array_equal(g["sorted_ids"].cpu().numpy(), ref["sorted_ids"])
