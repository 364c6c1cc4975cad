"""FP8 (E4M3) block-scaled grouped GEMM on the GPU vs the fp64 oracle (TileOPs MoE page, op
MoEGroupedGemmFP8Fwd): small masked and contiguous cases with every valid row compared, and the
page's full-size workloads on sampled rows of every group."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_rounded_close
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu


# Pipeline stages carry two k blocks for token tiles of up to 64 rows and one for taller tiles:
# (3, 144, ...) and (1, 128, 5120, ...) take one-block stages of 128-row tiles at one CTA per
# SM (the latter one unit of 40 k blocks); (4, 256, 512, ...) 64-row tiles of a 256-row layout
# at two CTAs per SM, with a group of three tiles; (5, 16, 128, ...) a single two-block stage,
# (2, 64, 1024, ...) two-block stages throughout, (8, 48, 384, ...) 48-row stages and an odd
# k-block count (a one-block last stage), all at two CTAs per SM.
@pytest.mark.parametrize("E,max_m,K,N,total", [(3, 144, 384, 256, 200),  # a 2-tile group
                                               (5, 16, 128, 128, 9),       # 1-row groups
                                               (2, 64, 1024, 384, 128),
                                               (1, 128, 5120, 128, 128),
                                               (8, 48, 384, 128, 60),
                                               (4, 256, 512, 256, 600)])
def test_fp8_masked_grouped_gemm_matches_oracle(E, max_m, K, N, total, cuda_device):
    w = inputs.Fp8GemmWorkload("t", E=E, max_m=max_m, K=K, N=N, total=total)
    d = inputs.generate_fp8_gemm(w, seed=E + K, device=cuda_device)
    out = B.moe_grouped_gemm_fp8(d["a"], d["a_scale"], d["b"], d["b_scale"], d["meta"])
    torch.cuda.synchronize()
    meta = d["meta"].cpu().numpy()
    ref = oracle.grouped_gemm_fp8(d["a"].cpu(), d["a_scale"].cpu(), d["b"].cpu(),
                                  d["b_scale"].cpu(), meta, max_m=max_m)
    live = np.concatenate([np.arange(e * max_m, e * max_m + int(meta[e])) for e in range(E)])
    got = out.reshape(E * max_m, N)[torch.from_numpy(live).to(cuda_device)]
    assert_rounded_close(got, ref[live], torch.bfloat16, what=f"fp8 masked E={E} K={K} N={N}")
    dead = np.setdiff1d(np.arange(E * max_m), live)
    assert torch.all(out.reshape(E * max_m, N)[torch.from_numpy(dead).to(cuda_device)] == 0)


def test_fp8_contiguous_grouped_gemm_matches_oracle(cuda_device):
    w = inputs.Fp8GemmWorkload("t", E=4, max_m=96, K=256, N=256, total=150)
    d = inputs.generate_fp8_gemm(w, seed=3, device=cuda_device)
    meta = d["meta"].cpu().numpy()
    psum = np.cumsum(meta).astype(np.int32)
    rows = int(psum[-1])
    a = d["a"].reshape(-1, w.K)[:rows].contiguous()
    sa = d["a_scale"].reshape(-1, w.K // 128)[:rows].contiguous()
    out = B.moe_grouped_gemm_fp8(a, sa, d["b"], d["b_scale"],
                                 torch.from_numpy(psum).to(cuda_device))
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm_fp8(a.cpu(), sa.cpu(), d["b"].cpu(), d["b_scale"].cpu(), psum)
    assert_rounded_close(out, ref, torch.bfloat16, what="fp8 contiguous")


def test_fp8_grouped_gemm_is_deterministic(cuda_device):
    """Every output element is summed in one fixed order: two calls give the same bits."""
    w = inputs.Fp8GemmWorkload("t", E=6, max_m=128, K=2048, N=512, total=500)
    d = inputs.generate_fp8_gemm(w, seed=21, device=cuda_device)
    outs = [B.moe_grouped_gemm_fp8(d["a"], d["a_scale"], d["b"], d["b_scale"], d["meta"])
            for _ in range(2)]
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_fp8_many_groups_take_the_tile_list_kernel(cuda_device):
    """Past 128 groups the tile list comes from the tile-list kernel instead of the GEMM's own
    prologue: 130 groups of up to 3 rows, every valid row compared."""
    w = inputs.Fp8GemmWorkload("t", E=130, max_m=16, K=256, N=128, total=200)
    d = inputs.generate_fp8_gemm(w, seed=4, device=cuda_device)
    out = B.moe_grouped_gemm_fp8(d["a"], d["a_scale"], d["b"], d["b_scale"], d["meta"])
    torch.cuda.synchronize()
    meta = d["meta"].cpu().numpy()
    ref = oracle.grouped_gemm_fp8(d["a"].cpu(), d["a_scale"].cpu(), d["b"].cpu(),
                                  d["b_scale"].cpu(), meta, max_m=w.max_m)
    live = np.concatenate([np.arange(e * w.max_m, e * w.max_m + int(meta[e]))
                           for e in range(w.E)])
    got = out.reshape(w.E * w.max_m, w.N)[torch.from_numpy(live).to(cuda_device)]
    assert_rounded_close(got, ref[live], torch.bfloat16, what="fp8 masked E=130")


def test_fp8_reports_a_bad_prefix_sum(cuda_device):
    """A contiguous layout whose prefix sums decrease: the group is dropped and the status word
    says MOE_ERR_INVALID_ARG."""
    w = inputs.Fp8GemmWorkload("t", E=3, max_m=32, K=128, N=128, total=48)
    d = inputs.generate_fp8_gemm(w, seed=6, device=cuda_device)
    a = d["a"].reshape(-1, w.K)[:32].contiguous()
    sa = d["a_scale"].reshape(-1, w.K // 128)[:32].contiguous()
    meta = torch.tensor([10, 5, 32], dtype=torch.int32, device=cuda_device)  # decreasing
    g = B.GroupedGemm(w.E, w.N, w.K, 0, 32, B.MOE_BF16, 0, 0)
    ws = B.new_workspace(B.lib().moe_grouped_gemm_workspace_size(B.ctypes.byref(g)), cuda_device)
    B.moe_grouped_gemm_fp8(a, sa, d["b"], d["b_scale"], meta, workspace=ws)
    assert B.get_device_status(ws) == B.MOE_ERR_INVALID_ARG


FULL = ["ds-v3-e8-up-masked", "ds-v3-dec-b64-down", "qwen3-235b-dec-b256-up",
        "kimi-k2-dec-b64-up"]


@pytest.mark.parametrize("name", FULL)
def test_fp8_full_size_workloads(name, cuda_device):
    w = inputs.FP8_GEMM_WORKLOADS[name]
    d = inputs.generate_fp8_gemm(w, seed=0, device=cuda_device)
    out = B.moe_grouped_gemm_fp8(d["a"], d["a_scale"], d["b"], d["b_scale"], d["meta"])
    torch.cuda.synchronize()
    meta = d["meta"].cpu().numpy()
    rows = []
    for e in range(w.E):  # every valid row of every group (at most 768 rows)
        rows += list(range(e * w.max_m, e * w.max_m + int(meta[e])))
    rows = np.array(rows)
    grp = rows // w.max_m
    a = d["a"].reshape(-1, w.K)[torch.from_numpy(rows).to(cuda_device)].cpu()
    sa = d["a_scale"].reshape(-1, w.K // 128)[torch.from_numpy(rows).to(cuda_device)].cpu()
    ref = np.empty((rows.size, w.N))
    for e in np.unique(grp):  # each group's sampled rows as a one-group contiguous problem
        sel = np.nonzero(grp == e)[0]
        ref[sel] = oracle.grouped_gemm_fp8(a[sel], sa[sel], d["b"][e:e + 1].cpu(),
                                           d["b_scale"][e:e + 1].cpu(),
                                           np.array([sel.size], np.int32))
    got = out.reshape(-1, w.N)[torch.from_numpy(rows).to(cuda_device)]
    assert_rounded_close(got, ref, torch.bfloat16, what=name)
    assert int(meta.sum()) == min(w.total, int(meta.sum()))
