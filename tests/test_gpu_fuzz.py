"""fused_moe_fwd and fused_moe_fwd_w4a16 on seeded random problems vs the fp64 oracle.

The shapes, routing modes, activations, shared experts and expert-parallel shards are drawn by
a fixed numpy generator (the list is the same on every run), inside the limits the header
states for each entry point: 16-bit problems with H, F and S multiples of 8, NVFP4 problems
with H and F multiples of 128 and no shared expert.  Each case checks the router's ids
bit-exact against the oracle's and against the plain fp64 selection, and every output element
under the parity bound of the other tests."""
import numpy as np
import pytest
import torch

from helpers import (assert_output_close, check_ids_against_plain_selection, oracle_fused,
                     run_fused, run_route)
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu


def _draw_cases(n, seed=2026):
    rng = np.random.default_rng(seed)
    cases = []
    for i in range(n):
        w4 = i % 3 == 2
        T = int(rng.choice([1, 2, 5, 8, 13, 31, 64, 97, 128, 129, 250, 400]))
        E = int(rng.choice([4, 8, 12, 16, 32, 64]))
        top_k = int(rng.integers(1, min(E, 8) + 1))
        if w4:
            H, F, S = 128 * int(rng.integers(1, 5)), 128 * int(rng.integers(1, 4)), 0
            dtype = torch.bfloat16
        else:
            H, F = 8 * int(rng.integers(8, 65)), 8 * int(rng.integers(8, 49))
            S = int(rng.choice([0, 0, 64, 200]))
            dtype = torch.float16 if rng.random() < 0.25 else torch.bfloat16
        kw = dict(T=T, H=H, E=E, F=F, top_k=top_k, S=S, dtype=dtype,
                  weights="nvfp4" if w4 else "bf16",
                  activation=str(rng.choice(["silu", "silu", "gelu_tanh", "relu2"])))
        if rng.random() < 0.5:  # sigmoid scores with a correction bias, maybe grouped
            kw.update(scoring_func="sigmoid", bias_std=0.1,
                      routed_scaling_factor=float(rng.choice([1.0, 2.5])))
            groups = [g for g in (2, 4, 8) if E % g == 0 and g < E]
            if groups and rng.random() < 0.5:
                G = int(rng.choice(groups))
                keep = int(rng.integers(1, G))
                if top_k <= keep * (E // G):
                    kw.update(num_expert_group=G, topk_group=keep)
        elif rng.random() < 0.3:
            kw.update(renormalize=False)
        if rng.random() < 0.25 and E >= 8:  # an expert-parallel shard
            loc = E // 4
            kw.update(ep_local=loc, ep_offset=loc * int(rng.integers(0, 4)))
        if rng.random() < 0.2:
            kw.update(skew_alpha=0.3)
        name = (f"fuzz{i}-{'w4' if w4 else ('f16' if dtype == torch.float16 else 'bf16')}"
                f"-t{T}-e{E}-k{top_k}-h{H}-f{F}")
        cases.append(inputs.Workload(name, **kw))
    return cases


CASES = _draw_cases(18)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_random_problem_matches_oracle(w, cuda_device):
    d = inputs.generate(w, seed=11, device=cuda_device)
    out = run_fused(w, d)
    ids, _ = run_route(w, d)
    torch.cuda.synchronize()
    ref, r_ids, _, _, noise = oracle_fused(w, d)
    assert np.array_equal(ids.cpu().numpy(), r_ids), w.name
    check_ids_against_plain_selection(w, d, ids, what=w.name)
    assert_output_close(out, ref, w.dtype, noise, what=w.name)
    assert B.get_device_status(B._workspace(0, cuda_device)) == B.MOE_OK
