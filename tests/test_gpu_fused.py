"""fused_moe_fwd on the GPU vs the fp64 oracle, end to end.

Small cases cover every routing mode, both dtypes, the direct (T <= 8) and sorted paths, the
shared expert, ragged sizes and several tiles per expert; every output element is compared.
The five workloads the project is measured on run at full size: routing is compared bit-exact
on every token (and with the plain fp64 selection), and every output element with the oracle."""
import numpy as np
import pytest
import torch

from helpers import (assert_output_close, check_ids_against_plain_selection, oracle_fused,
                     oracle_route, run_fused, run_route)
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload
SMALL = [
    W("direct-t1", T=1, H=256, E=16, F=128, top_k=4),
    W("direct-t3-f16", T=3, H=192, E=8, F=72, top_k=2, dtype=torch.float16),
    W("direct-t8-k8", T=8, H=320, E=64, F=192, top_k=8),
    W("direct-t8-sigmoid-shared", T=8, H=256, E=32, F=128, top_k=4, scoring_func="sigmoid",
      bias_std=0.1, routed_scaling_factor=2.5, S=256),
    W("sorted-t9", T=9, H=256, E=16, F=128, top_k=4),
    W("sorted-t37-ragged", T=37, H=328, E=12, F=200, top_k=3),
    W("sorted-t300-multitile", T=300, H=256, E=4, F=128, top_k=2),
    W("sorted-t200-f16", T=200, H=192, E=16, F=256, top_k=4, dtype=torch.float16),
    W("sorted-grouped", T=160, H=256, E=64, F=128, top_k=6, scoring_func="sigmoid",
      bias_std=0.1, num_expert_group=8, topk_group=3, routed_scaling_factor=2.5),
    W("sorted-sigmoid-shared", T=96, H=256, E=24, F=96, top_k=4, scoring_func="sigmoid",
      bias_std=0.1, routed_scaling_factor=2.827, S=384),
    W("sorted-norenorm", T=50, H=128, E=10, F=64, top_k=3, renormalize=False),
    W("sorted-wide-tiles", T=600, H=256, E=4, F=192, top_k=2),  # 256-row tiles, 2 per expert
    W("sorted-wide-grouped-shared", T=400, H=192, E=16, F=128, top_k=4,
      scoring_func="sigmoid", bias_std=0.1, num_expert_group=4, topk_group=2,
      routed_scaling_factor=2.5, S=256),
    # activation variants: GeGLU-tanh (gated) and ReLU2 (single projection, 256-row units
    # whose second half is partial or absent for these F and S)
    W("direct-t5-gelu-tanh", T=5, H=256, E=16, F=128, top_k=4, activation="gelu_tanh"),
    W("sorted-t70-gelu-tanh-shared", T=70, H=192, E=12, F=200, top_k=3, scoring_func="sigmoid",
      bias_std=0.1, routed_scaling_factor=2.5, S=256, activation="gelu_tanh"),
    W("direct-t4-relu2", T=4, H=256, E=8, F=192, top_k=2, activation="relu2"),
    W("sorted-t150-relu2-ragged-shared", T=150, H=328, E=12, F=328, top_k=3, S=136,
      activation="relu2"),
    W("sorted-t600-relu2-wide", T=600, H=256, E=4, F=384, top_k=2, activation="relu2"),
    W("sorted-t40-relu2-f16", T=40, H=192, E=8, F=256, top_k=2, activation="relu2",
      dtype=torch.float16),
    W("sorted-t300-skewed", T=300, H=256, E=32, F=128, top_k=4, skew_alpha=0.3),
    # prefill-sized experts (>= 96 rows on average): the down projection runs on pairs of SMs
    W("pair-t600", T=600, H=512, E=8, F=256, top_k=2),
    W("pair-t1000-grouped-f16", T=1000, H=256, E=16, F=128, top_k=4, dtype=torch.float16,
      scoring_func="sigmoid", bias_std=0.1, num_expert_group=4, topk_group=2,
      routed_scaling_factor=2.5),
    W("pair-t700-gelu-tanh-shared", T=700, H=768, E=8, F=384, top_k=2, activation="gelu_tanh",
      S=256),
    W("pair-t1100-skewed-chunked-sort", T=1100, H=256, E=32, F=256, top_k=8, skew_alpha=0.5),
]
BY_NAME = {w.name: w for w in SMALL}


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fused_small_matches_oracle(w, cuda_device):
    d = inputs.generate(w, seed=1, device=cuda_device)
    out = run_fused(w, d)
    ids, _ = run_route(w, d)
    torch.cuda.synchronize()
    ref, r_ids, _, _, noise = oracle_fused(w, d)
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    check_ids_against_plain_selection(w, d, ids, what=w.name)
    assert_output_close(out, ref, w.dtype, noise, what=w.name)
    assert B.get_device_status(B._workspace(0, cuda_device)) == B.MOE_OK


@pytest.mark.parametrize("w", [BY_NAME[n] for n in ("direct-t8-k8", "sorted-t300-multitile",
                                                    "sorted-sigmoid-shared", "pair-t600")],
                         ids=lambda w: w.name)
def test_fused_is_deterministic_and_graph_replayable(w, cuda_device):
    d = inputs.generate(w, seed=2, device=cuda_device)
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor, w.S)
    ws = B.new_workspace(B.workspace_size(prob), cuda_device)
    a = run_fused(w, d, workspace=ws).clone()
    b = run_fused(w, d, workspace=ws).clone()
    assert torch.equal(a, b)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_fused(w, d, workspace=ws, out=out)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_fused(w, d, workspace=ws, out=out)
    for _ in range(3):
        out.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out, a)


@pytest.mark.parametrize("w", [BY_NAME[n] for n in ("direct-t8-k8", "sorted-t37-ragged",
                                                    "sorted-sigmoid-shared",
                                                    "pair-t1100-skewed-chunked-sort")],
                         ids=lambda w: w.name)
def test_fused_ignores_poisoned_workspace(w, cuda_device):
    """Every workspace byte past the status header starts as 0xFF (NaN for bf16/f16 and -1 for
    ints): nothing may read scratch it did not write."""
    d = inputs.generate(w, seed=3, device=cuda_device)
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor, w.S)
    clean = B.new_workspace(B.workspace_size(prob), cuda_device)
    ref = run_fused(w, d, workspace=clean).clone()
    poison = B.new_workspace(B.workspace_size(prob), cuda_device)
    poison[256:] = 0xFF
    out = torch.full_like(ref, float("nan"))
    run_fused(w, d, workspace=poison, out=out)
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    assert B.get_device_status(poison) == B.MOE_OK


def test_fused_empty_batch(cuda_device):
    w = W("empty", T=0, H=128, E=8, F=64, top_k=2)
    d = inputs.generate(w, seed=0, device=cuda_device)
    out = run_fused(w, d)
    assert out.shape == (0, 128)


# ---------------------------------------------------------------- full-size measured workloads
# Every output element of every workload is compared with the oracle (the DeepSeek-V3 prefill
# oracle is 2.9e12 fp64 multiply-adds, about a minute on 16 host cores, and holds a 23 GB host
# copy of the experts).
FULL = ["tiny-softmax", "qwen3-30b-a3b-decode-t32", "qwen3-235b-a22b-decode-t512",
        "deepseek-v3-grouped-prefill-t4096", "kimi-k2-shared-t512"]


@pytest.mark.parametrize("name", FULL)
def test_fused_full_size_workloads(name, cuda_device):
    _full_size_check(inputs.WORKLOADS[name], cuda_device)


@pytest.mark.parametrize("name", sorted(n for n, v in inputs.VARIANTS.items()
                                         if v.weights == "bf16" and v.ep_local == 0))
def test_fused_full_size_variants(name, cuda_device):
    """Skewed routing and the activation variants on the Qwen3-235B-A22B decode shape (the
    NVFP4 and expert-parallel variants are in test_gpu_w4a16.py)."""
    _full_size_check(inputs.VARIANTS[name], cuda_device)


def test_fused_full_size_qwen3_235b_f16(cuda_device):
    w = inputs.WORKLOADS["qwen3-235b-a22b-decode-t512"].with_(dtype=torch.float16)
    _full_size_check(w, cuda_device)


def _full_size_check(w, dev):
    d = inputs.generate(w, seed=0, device=dev)
    out = run_fused(w, d)
    ids, wts = run_route(w, d)
    torch.cuda.synchronize()
    routed = oracle_route(w, d)
    assert np.array_equal(ids.cpu().numpy(), routed[0]), "routing ids differ"
    check_ids_against_plain_selection(w, d, ids, what=f"{w.name} routing")
    np.testing.assert_allclose(wts.cpu().numpy(), routed[1], rtol=2e-6, atol=1e-7)
    ref, _, _, _, noise = oracle_fused(w, d, routed=routed)
    assert_output_close(out, ref, w.dtype, noise, what=f"{w.name} {str(w.dtype)[6:]}")
    del ref, noise
    out2 = run_fused(w, d)
    assert torch.equal(out, out2), "repeat call not bit-identical"
    assert B.get_device_status(B._workspace(0, dev)) == B.MOE_OK
    del d
    torch.cuda.empty_cache()


HOST_CASES = [BY_NAME["direct-t8-k8"], BY_NAME["sorted-sigmoid-shared"], W("sorted-t200-w4a16", T=200, H=256, E=16, F=128, top_k=4,
                                     weights="nvfp4")]


@pytest.mark.parametrize("w", HOST_CASES, ids=lambda w: w.name)
def test_fused_from_host_buffers(w, cuda_device):
    """fused_moe_fwd_host / fused_moe_fwd_w4a16_host: the batch comes from and goes back to
    page-locked host buffers inside one library call; the result equals the device-buffer call
    bit for bit and the oracle within the usual bound, on two calls in a row."""
    from helpers import packed_w4
    d = inputs.generate(w, seed=4, device=cuda_device)
    ref_dev = run_fused(w, d).clone()
    h_hidden = d["hidden_states"].cpu().pin_memory()
    h_gating = d["gating_output"].cpu().pin_memory()
    if w.weights == "nvfp4":
        w1, w2 = packed_w4(d)
        kw = dict(correction_bias=d["correction_bias"], **w.kwargs())
    else:
        w1, w2 = d["w_gate_up"], d["w_down"]
        kw = dict(correction_bias=d["correction_bias"], shared_w_gate_up=d["shared_w_gate_up"],
                  shared_w_down=d["shared_w_down"], **w.kwargs())
    for _ in range(2):
        h_out = torch.full((w.T, w.H), float("nan"), dtype=w.dtype).pin_memory()
        B.fused_moe_fwd_host(h_hidden, h_gating, w1, w2, out_host=h_out, **kw)
        torch.cuda.synchronize()
        assert torch.equal(h_out, ref_dev.cpu())
    ref, _, _, _, noise = oracle_fused(w, d)
    assert_output_close(h_out, ref, w.dtype, noise, what=f"{w.name} host buffers")
