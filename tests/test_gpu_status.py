"""Device-side failure reporting: a bounded wait that runs out, and a bad expert id, are
reported through the workspace status word, and the context stays usable afterwards.

The wait is made to run out with the library's wait-limit knob set to 0 (the first poll that
finds a pipeline stage not yet filled gives up): nothing hangs, traps or faults."""
import numpy as np
import pytest
import torch

from helpers import assert_output_close, oracle_fused, run_fused
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu


def _workspace(w, dev):
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor, w.S)
    return B.new_workspace(B.workspace_size(prob), dev)


@pytest.mark.parametrize("T", [4, 96])  # direct path and sorted path
def test_wait_timeout_is_reported_and_context_survives(T, cuda_device):
    w = inputs.Workload("timeout", T=T, H=4096, E=16, F=512, top_k=4, S=256)
    d = inputs.generate(w, seed=5, device=cuda_device)
    ws = _workspace(w, cuda_device)
    old = B.set_wait_limit_ns(0)
    try:
        run_fused(w, d, workspace=ws)
        status = B.get_device_status(ws)  # synchronises
    finally:
        B.set_wait_limit_ns(old)
    assert status == B.MOE_ERR_TIMEOUT
    assert B.get_device_status(ws) == B.MOE_OK  # reading cleared it
    out = run_fused(w, d, workspace=ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == B.MOE_OK
    ref, _, _, _, noise = oracle_fused(w, d)
    assert_output_close(out, ref, w.dtype, noise, what=f"after timeout T={T}")


# NVFP4: T=4 runs the direct path (32-row gate/up and down projection at two CTAs per SM), T=96
# the 128-row gate/up over token rows (one CTA per SM), T=200 gathered rows in 64-row tiles.
@pytest.mark.parametrize("T", [4, 96, 200])
def test_wait_timeout_in_nvfp4_kernels_is_reported_and_context_survives(T, cuda_device):
    w = inputs.Workload("timeout-w4", T=T, H=1024, E=16, F=256, top_k=4, weights="nvfp4")
    d = inputs.generate(w, seed=6, device=cuda_device)
    ws = _workspace(w, cuda_device)
    old = B.set_wait_limit_ns(0)
    try:
        run_fused(w, d, workspace=ws)
        status = B.get_device_status(ws)  # synchronises
    finally:
        B.set_wait_limit_ns(old)
    assert status == B.MOE_ERR_TIMEOUT
    out = run_fused(w, d, workspace=ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == B.MOE_OK
    ref, _, _, _, noise = oracle_fused(w, d)
    assert_output_close(out, ref, w.dtype, noise, what=f"NVFP4 after timeout T={T}")


def test_bad_expert_id_in_staged_gemm_is_reported(cuda_device):
    # moe_align_sort treats the bad id as padding and reports it.
    ids = inputs.random_ids(12, 2, 8, seed=3)
    ids[2, 1] = 8
    g = B.moe_align_sort(ids.to(cuda_device), 8, 1)
    assert B.get_device_status(g["workspace"]) == B.MOE_ERR_BAD_EXPERT_ID
    assert int(g["inv_route"][5].item()) == -1
    assert np.all(g["counts"].cpu().numpy().sum() == 12 * 2 - 1)
