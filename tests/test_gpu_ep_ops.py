"""Expert-parallel building blocks on the GPU vs the oracle: pre-permute (local expert ids),
the grouped GEMM in its masked and contiguous layouts, and the weighted post-permute.

Shapes follow the TileOPs MoE page's workloads for these ops (MoEPrePermuteFwd,
MoEGroupedGemmFwd "ds-v3-ep8-masked", MoEPostPermuteFwd); the masked GEMM at full size is
checked on sampled rows of every group."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_rms_close, assert_rounded_close, dt_code, log_parity
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu


def _local_ids(T, k, E_global, E_local, seed):
    """Router-like ids over E_global experts mapped to a shard of E_local (others -> -1)."""
    g = inputs.random_ids(T, k, E_global, seed=seed)
    return torch.where(g < E_local, g, torch.full_like(g, -1))


# (name, T, H, k, E_local, E_global, dtype): the page's MoEPrePermuteFwd workloads
PRE = [
    ("decode-t32", 32, 128, 2, 4, 4, torch.float16),
    ("prefill-t512", 512, 128, 2, 4, 4, torch.bfloat16),
    ("ds-v3-ep8-t100", 100, 7168, 8, 32, 256, torch.bfloat16),
    ("qwen3-30b-ep8-b1", 1, 2048, 8, 16, 128, torch.bfloat16),
]


@pytest.mark.parametrize("name,T,H,k,E,Eg,dtype", PRE, ids=[p[0] for p in PRE])
def test_pre_permute_matches_sort_and_gather(name, T, H, k, E, Eg, dtype, cuda_device):
    ids = _local_ids(T, k, Eg, E, seed=T + H)
    hidden = inputs.random_rows(T, H, seed=3, dtype=dtype)
    r = B.moe_pre_permute(hidden.to(cuda_device), ids.to(cuda_device), E)
    torch.cuda.synchronize()
    srt = oracle.align_sort(ids.numpy(), E, 1)
    n = int(srt["offsets"][E])
    assert np.array_equal(r["offsets"].cpu().numpy(), srt["offsets"])
    assert np.array_equal(r["sorted_ids"].cpu().numpy()[:n], srt["sorted_ids"][:n])
    assert np.array_equal(r["inv_route"].cpu().numpy(), srt["inv_route"])
    want = hidden[torch.from_numpy(srt["sorted_ids"][:n] // k).long()]
    assert torch.equal(r["permuted"][:n].cpu(), want)  # a gather: bit-exact


def _masked_case(E, max_m, K, N, activation, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    a = (torch.randn((E, max_m, K), generator=g)).to(dtype)
    nb = 2 * N if activation == "silu" else N
    b = (torch.randn((E, nb, K), generator=g) / K ** 0.5).to(dtype)
    meta = torch.randint(0, max_m + 1, (E,), generator=g, dtype=torch.int32)
    meta[0] = max_m  # a full group
    if E > 2:
        meta[1] = 0  # an empty group
    return a, b, meta


@pytest.mark.parametrize("activation,out_f32,dtype", [("none", False, torch.bfloat16),
                                                      ("silu", False, torch.bfloat16),
                                                      ("none", True, torch.bfloat16),
                                                      ("none", False, torch.float16)])
def test_masked_grouped_gemm_matches_oracle(activation, out_f32, dtype, cuda_device):
    E, max_m, K, N = 6, 144, 320, 136  # ragged K tail, a group of two token tiles
    a, b, meta = _masked_case(E, max_m, K, N, activation, seed=5, dtype=dtype)
    out = B.moe_grouped_gemm(a.to(cuda_device), b.to(cuda_device), meta.to(cuda_device),
                             activation=activation, out_f32=out_f32)
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm(a, b, meta.numpy(), dt_code(dtype),
                              activation=1 if activation == "silu" else 0, max_m=max_m)
    got = out.reshape(E * max_m, N)
    live = np.concatenate([np.arange(e * max_m, e * max_m + int(meta[e])) for e in range(E)])
    idx = torch.from_numpy(live).to(cuda_device)
    if out_f32:
        assert_rms_close(got[idx], ref[live], tol=1e-4, what="masked grouped GEMM f32")
    else:
        assert_rounded_close(got[idx], ref[live], dtype, what=f"masked grouped GEMM {activation}")
    dead = torch.ones(E * max_m, dtype=torch.bool)
    dead[torch.from_numpy(live)] = False
    assert torch.all(got[dead.to(cuda_device)] == 0)  # rows past each group's count untouched


def test_contiguous_grouped_gemm_matches_oracle(cuda_device):
    g = torch.Generator().manual_seed(11)
    counts = torch.tensor([130, 0, 7, 256, 1], dtype=torch.int32)
    psum = torch.cumsum(counts, 0).to(torch.int32)
    P, K, N = int(psum[-1]), 256, 192
    a = torch.randn((P, K), generator=g).to(torch.bfloat16)
    b = (torch.randn((5, 2 * N, K), generator=g) / K ** 0.5).to(torch.bfloat16)
    out = B.moe_grouped_gemm(a.to(cuda_device), b.to(cuda_device), psum.to(cuda_device),
                             activation="silu")
    torch.cuda.synchronize()
    ref = oracle.grouped_gemm(a, b, psum.numpy(), oracle.BF16, activation=1)
    assert_rounded_close(out, ref, torch.bfloat16, what="contiguous grouped GEMM silu")


def test_grouped_gemm_reports_a_bad_prefix_sum(cuda_device):
    a = torch.zeros((32, 64), dtype=torch.bfloat16, device=cuda_device)
    b = torch.zeros((3, 16, 64), dtype=torch.bfloat16, device=cuda_device)
    meta = torch.tensor([10, 5, 32], dtype=torch.int32, device=cuda_device)  # decreasing
    ws = B.new_workspace(B.lib().moe_grouped_gemm_workspace_size(
        B.ctypes.byref(B.grouped_gemm_desc(a, b))), cuda_device)
    B.moe_grouped_gemm(a, b, meta, workspace=ws)
    assert B.get_device_status(ws) == B.MOE_ERR_INVALID_ARG


def test_masked_grouped_gemm_ds_v3_ep8_full_size(cuda_device):
    """The page's ds-v3-ep8-masked workload: a [32, 128, 7168], b [32, 4096, 7168]; valid rows
    per group drawn in [64, 128]; 3 sampled rows per group checked against the oracle."""
    E, max_m, K, N = 32, 128, 7168, 4096
    d = grouped_gemm_inputs(seed=0, device=cuda_device)
    out = B.moe_grouped_gemm(d["a"], d["b"], d["meta"])
    torch.cuda.synchronize()
    meta = d["meta"].cpu().numpy()
    rows = []
    for e in range(E):
        m = int(meta[e])
        rows += [e * max_m, e * max_m + m // 2, e * max_m + m - 1]
    rows = np.array(rows)
    a_s = d["a"].reshape(E * max_m, K)[torch.from_numpy(rows).to(cuda_device)].cpu()
    grp = rows // max_m
    ref = np.empty((rows.size, N))
    for e in range(E):  # one group at a time: a [1, 3, K] against b[e]
        sel = np.nonzero(grp == e)[0]
        ref[sel] = oracle.grouped_gemm(a_s[sel].reshape(1, sel.size, K), d["b"][e:e + 1].cpu(),
                                       np.array([sel.size], np.int32), oracle.BF16,
                                       max_m=sel.size)
    got = out.reshape(E * max_m, N)[torch.from_numpy(rows).to(cuda_device)]
    assert_rounded_close(got, ref, torch.bfloat16, what="ds-v3-ep8-masked")


def grouped_gemm_inputs(seed, device):
    return inputs.generate_grouped_gemm(inputs.GROUPED_GEMM_WORKLOADS["ds-v3-ep8-masked"], seed,
                                        device)


@pytest.mark.parametrize("T,k,H,dtype", [(32, 2, 128, torch.float16), (100, 8, 7168,
                                                                        torch.bfloat16),
                                         (1, 8, 2048, torch.bfloat16)])
def test_post_permute_matches_oracle(T, k, H, dtype, cuda_device):
    rows_n = T * k
    x = inputs.random_rows(rows_n, H, seed=7, dtype=dtype)
    w = inputs.random_weights(T * k, seed=8).reshape(T, k)
    inv = torch.randperm(rows_n, generator=torch.Generator().manual_seed(9)).to(torch.int32)
    inv[::5] = -1  # routes to other GPUs
    out = B.moe_post_permute(x.to(cuda_device), w.to(cuda_device), inv.to(cuda_device))
    torch.cuda.synchronize()
    ref = oracle.post_permute(x, w.numpy().astype(np.float64), inv.numpy(), k, dt_code(dtype))
    assert_rounded_close(out, ref, dtype, what=f"post-permute T={T} k={k}")
