"""Grouped GEMMs, combine and shared expert on the GPU (staged C-ABI calls) vs the oracle.

Shapes are small enough for the oracle to finish in seconds but span several K blocks, a
ragged K tail, a ragged weight slab (F, H not multiples of 128), experts with more than one
128-row tile, empty experts and padding rows."""
import numpy as np
import pytest
import torch

import oracle
from helpers import assert_rms_close, assert_rounded_close, dt_code, log_parity
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu

# (T, k, E, H, F, block_m, pad_frac, dtype)
GEMM_CASES = [
    (150, 4, 6, 320, 192, 1, 0.0, torch.bfloat16),     # ~100 rows/expert, ragged K and slab
    (300, 2, 3, 256, 128, 1, 0.0, torch.bfloat16),     # 200 rows/expert: two tiles each
    (64, 8, 32, 192, 256, 16, 0.1, torch.bfloat16),    # padded segments, padding routes
    (40, 4, 12, 136, 72, 1, 0.0, torch.float16),       # K tail of 8, F < 128
    (9, 8, 64, 512, 96, 1, 0.0, torch.bfloat16),       # decode-like: 1-2 rows per expert
    (800, 2, 3, 256, 136, 1, 0.0, torch.bfloat16),     # 256-row tiles, ~530 rows per expert
    (260, 4, 8, 192, 128, 8, 0.05, torch.float16),     # 256-row tiles with padded segments
    (6, 4, 16, 256, 128, 1, 0.0, torch.bfloat16),      # T <= 8: staged calls still gather
]


# (T, k, E, H, F, activation, dtype): the gate/up GEMM with the other activations
ACT_CASES = [
    (150, 4, 6, 320, 200, "gelu_tanh", torch.bfloat16),
    (9, 8, 64, 256, 96, "gelu_tanh", torch.float16),
    (150, 4, 6, 320, 200, "relu2", torch.bfloat16),   # units of 256 rows: halves 128 + 72
    (300, 2, 3, 256, 384, "relu2", torch.bfloat16),   # second unit is a single 128-row half
    (40, 4, 12, 136, 72, "relu2", torch.float16),     # F < 128: no second half at all
]


def _expert_of_rows(sorted_ids, offsets, E):
    eo = np.full(sorted_ids.size, -1, np.int32)
    for e in range(E):
        seg = slice(offsets[e], offsets[e + 1])
        eo[seg] = np.where(sorted_ids[seg] >= 0, e, -1)
    return eo


@pytest.mark.parametrize("T,k,E,H,F,block_m,pad,dtype", GEMM_CASES)
def test_gemm1_and_gemm2_match_oracle(T, k, E, H, F, block_m, pad, dtype, cuda_device):
    w = inputs.Workload("g", T=T, H=H, E=E, F=F, top_k=k, dtype=dtype)
    d = inputs.generate(w, seed=T + E, device=cuda_device)
    ids = inputs.random_ids(T, k, E, seed=T * 7 + E, pad_frac=pad)
    srt = oracle.align_sort(ids.numpy(), E, block_m)
    sorted_ids = torch.from_numpy(srt["sorted_ids"]).to(cuda_device)
    offsets = torch.from_numpy(srt["offsets"]).to(cuda_device)
    act = B.moe_gemm1_swiglu(d["hidden_states"], sorted_ids, offsets, d["w_gate_up"], k, block_m)
    torch.cuda.synchronize()
    # oracle act, row by row in sorted order
    eo = _expert_of_rows(srt["sorted_ids"], srt["offsets"], E)
    rows = srt["offsets"][E]
    x_rows = torch.zeros((rows, H), dtype=dtype)
    hid = d["hidden_states"].cpu()
    sid = srt["sorted_ids"][:rows]
    live = sid >= 0
    x_rows[torch.from_numpy(np.nonzero(live)[0])] = hid[torch.from_numpy(sid[live] // k)]
    ref_act = oracle.expert_act(x_rows, eo[:rows], d["w_gate_up"].cpu(), dt_code(dtype))
    assert_rounded_close(act[:rows], ref_act, dtype, what=f"act T={T} E={E} H={H} F={F}")
    assert torch.all(act[:rows][torch.from_numpy(~live).to(cuda_device)] == 0)

    # gemm2 on a seeded act (not the GPU's), with route weights
    a_in = inputs.random_rows(act.shape[0], F, seed=3, dtype=dtype, std=0.5).to(cuda_device)
    tw = inputs.random_weights(T * k, seed=4).to(cuda_device)
    y = B.moe_gemm2(a_in, sorted_ids, offsets, tw, d["w_down"], T, k, block_m)
    torch.cuda.synchronize()
    scale = np.where(live, tw.cpu().numpy()[np.maximum(sid, 0)], 0.0)
    ref_y = oracle.expert_down(a_in[:rows].cpu(), eo[:rows], scale, d["w_down"].cpu(),
                               dt_code(dtype))
    assert_rms_close(y[:rows], ref_y, tol=1e-4, what=f"y_route T={T} E={E} H={H} F={F}")
    assert torch.all(y[:rows][torch.from_numpy(~live).to(cuda_device)] == 0)
    ws = B._workspace(0, cuda_device)
    assert B.get_device_status(ws) == B.MOE_OK


@pytest.mark.parametrize("T,k,E,H,F,activation,dtype", ACT_CASES)
def test_gemm1_activation_variants_match_oracle(T, k, E, H, F, activation, dtype, cuda_device):
    w = inputs.Workload("g", T=T, H=H, E=E, F=F, top_k=k, dtype=dtype, activation=activation)
    d = inputs.generate(w, seed=T + E + 1, device=cuda_device)
    ids = inputs.random_ids(T, k, E, seed=T * 5 + E)
    srt = oracle.align_sort(ids.numpy(), E, 1)
    sorted_ids = torch.from_numpy(srt["sorted_ids"]).to(cuda_device)
    offsets = torch.from_numpy(srt["offsets"]).to(cuda_device)
    act = B.moe_gemm1_swiglu(d["hidden_states"], sorted_ids, offsets, d["w_gate_up"], k, 1,
                             activation=activation)
    torch.cuda.synchronize()
    eo = _expert_of_rows(srt["sorted_ids"], srt["offsets"], E)
    rows = srt["offsets"][E]
    sid = srt["sorted_ids"][:rows]
    x_rows = d["hidden_states"].cpu()[torch.from_numpy(sid // k).long()]
    code = {"gelu_tanh": oracle.ACT_GELU_TANH, "relu2": oracle.ACT_RELU2}[activation]
    ref_act = oracle.expert_act(x_rows, eo[:rows], d["w_gate_up"].cpu(), dt_code(dtype),
                                activation=code)
    assert_rounded_close(act[:rows], ref_act, dtype, what=f"act {activation} T={T} F={F}")
    assert B.get_device_status(B._workspace(0, cuda_device)) == B.MOE_OK


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_combine_matches_oracle(dtype, cuda_device):
    T, k, E, H = 70, 4, 9, 264
    ids = inputs.random_ids(T, k, E, seed=2, pad_frac=0.1)
    srt = oracle.align_sort(ids.numpy(), E, 4)
    cap = srt["sorted_ids"].size
    # f32 rows that are exactly representable in bf16 so the oracle can read them as bits
    y16 = inputs.random_rows(cap, H, seed=5, dtype=torch.bfloat16)
    sh16 = inputs.random_rows(T, H, seed=6, dtype=torch.bfloat16)
    y = y16.float().to(cuda_device)
    sh = sh16.float().to(cuda_device)
    inv = torch.from_numpy(srt["inv_route"]).to(cuda_device)
    out = B.moe_combine(y, inv, T, k, topk_ids=ids.to(cuda_device), shared_out=sh, dtype=dtype)
    ref = oracle.combine(y16, srt["inv_route"], k, oracle.BF16, shared=sh16)
    assert_rounded_close(out, ref, dtype, rel_rms=1e-6, what="combine")
    out2 = B.moe_combine(y, None, T, k, topk_ids=ids.to(cuda_device), dtype=dtype)  # identity
    ref2 = oracle.combine(y16, np.where(ids.numpy().reshape(-1) >= 0,
                                        np.arange(T * k), -1).astype(np.int32), k, oracle.BF16)
    assert_rounded_close(out2, ref2, dtype, rel_rms=1e-6, what="combine identity")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_combine_on_an_expert_parallel_shard(dtype, cuda_device):
    """A shard holding 32 of 256 experts: a token averages one route with a row here, and at
    2048 tokens of H = 7168 a CTA covers at least 8 column chunks, so the combine takes its
    shard form (each token's local routes listed first).  Tokens 0-3 have all 8 routes local,
    token 4 five, and about a third have none (their output is the shared row alone)."""
    T, k, E, n_loc, H = 2048, 8, 256, 32, 7168
    ids = inputs.random_ids(T, k, E, seed=21).numpy()
    ids[0:4] = np.arange(8, dtype=np.int32)             # all eight routes local
    ids[4] = np.array([0, 40, 1, 2, 90, 3, 4, 200], np.int32)  # five of eight
    local = np.where(ids < n_loc, ids, -1).astype(np.int32)
    is_local = local.reshape(-1) >= 0
    n_rows = int(is_local.sum())
    rng = np.random.default_rng(21)
    inv = np.full(T * k, -1, np.int32)
    inv[is_local] = rng.permutation(n_rows).astype(np.int32)  # rows in a shuffled order
    y16 = inputs.random_rows(n_rows, H, seed=22, dtype=torch.bfloat16)
    sh16 = inputs.random_rows(T, H, seed=23, dtype=torch.bfloat16)
    out = B.moe_combine(y16.float().to(cuda_device), torch.from_numpy(inv).to(cuda_device), T, k,
                        topk_ids=torch.from_numpy(local).to(cuda_device),
                        shared_out=sh16.float().to(cuda_device), dtype=dtype, E=E,
                        ep_num_local=n_loc, ep_local_offset=0)
    ref = oracle.combine(y16, inv, k, oracle.BF16, shared=sh16)
    assert_rounded_close(out, ref, dtype, rel_rms=1e-6, what="combine on a shard")


@pytest.mark.parametrize("T,H,S", [(1, 256, 128), (37, 192, 320), (300, 128, 136)])
def test_shared_expert_matches_oracle(T, H, S, cuda_device):
    w = inputs.Workload("s", T=T, H=H, E=2, F=16, top_k=1, S=S)
    d = inputs.generate(w, seed=S, device=cuda_device)
    out = B.moe_shared_expert_fwd(d["hidden_states"], d["shared_w_gate_up"], d["shared_w_down"])
    torch.cuda.synchronize()
    none = np.full((T, 1), -1, np.int32)
    ref = oracle.moe_tokens(d["hidden_states"].cpu(), none, np.zeros((T, 1)), d["w_gate_up"].cpu(),
                            d["w_down"].cpu(), 0, shared_w_gate_up=d["shared_w_gate_up"].cpu(),
                            shared_w_down=d["shared_w_down"].cpu())
    # The only rounding on the path is SiLU(g)*u to bf16 (at most 2^-8 relative) before the f32
    # down projection, so |gpu - oracle|_h <= 2^-8 * sum_f |Wd[h,f]| |act_f| (+ f32 slack).
    act = oracle.expert_act(d["hidden_states"].cpu(), np.zeros(T, np.int32),
                            d["shared_w_gate_up"].cpu()[None], oracle.BF16)
    wd_abs = np.abs(d["shared_w_down"].double().cpu().numpy())
    bound = 2.0 ** -8 * (np.abs(act) @ wd_abs.T) + 1e-5 * np.sqrt(np.mean(ref * ref))
    err = np.abs(out.double().cpu().numpy() - ref)
    log_parity(f"shared T={T} H={H} S={S}", max_err_over_rms=float(err.max()) /
               float(np.sqrt(np.mean(ref * ref))), max_err_over_bound=float((err / bound).max()))
    assert np.all(err <= bound)
