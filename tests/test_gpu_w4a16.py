"""NVFP4 (W4A16) experts and expert-parallel shards on the GPU vs the fp64 oracle.

The staged GEMMs run at shapes that span several 128-k stages, several token tiles per expert,
both gate/up layouts (gated and the single-projection ReLU2 with a half-empty second unit) and
empty experts.  The fused path covers the direct (T <= 8), token-rows (T <= 128) and gathered
(T > 128) forms, shards of the experts, and the measured W4A16 workloads at full size."""
import numpy as np
import pytest
import torch

import oracle
from helpers import (ACT_CODES, RMS_TOL, assert_output_close, assert_rms_close,
                     assert_rounded_close, half_ulp, local_ids, log_parity, oracle_fused,
                     oracle_route, packed_w4, run_fused, run_route, to_np)
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

pytestmark = pytest.mark.gpu

W = inputs.Workload

# (T, k, E, H, F, activation)
STAGED = [
    (150, 4, 6, 256, 256, "silu"),      # ~100 rows per expert, 2 k stages
    (9, 8, 64, 512, 128, "silu"),       # decode-like: 1-2 rows per expert, empty experts
    (300, 2, 3, 384, 256, "gelu_tanh"),  # 200 rows per expert: two token tiles each
    (40, 4, 12, 256, 384, "relu2"),     # ReLU2 units of 256 rows: second unit is one half
]


def _expert_of_rows(sorted_ids, offsets, E):
    eo = np.full(sorted_ids.size, -1, np.int32)
    for e in range(E):
        seg = slice(offsets[e], offsets[e + 1])
        eo[seg] = np.where(sorted_ids[seg] >= 0, e, -1)
    return eo


@pytest.mark.parametrize("T,k,E,H,F,activation", STAGED)
def test_w4a16_gemms_match_oracle(T, k, E, H, F, activation, cuda_device):
    w = W("g", T=T, H=H, E=E, F=F, top_k=k, weights="nvfp4", activation=activation)
    d = inputs.generate(w, seed=T + E, device=cuda_device)
    ids = inputs.random_ids(T, k, E, seed=T * 3 + E)
    srt = oracle.align_sort(ids.numpy(), E, 1)
    sorted_ids = torch.from_numpy(srt["sorted_ids"]).to(cuda_device)
    offsets = torch.from_numpy(srt["offsets"]).to(cuda_device)
    w1_packed, w2_packed = packed_w4(d)
    act = B.moe_gemm1_w4a16(d["hidden_states"], sorted_ids, offsets, w1_packed, k,
                            activation=activation)
    torch.cuda.synchronize()
    rows = srt["offsets"][E]
    eo = _expert_of_rows(srt["sorted_ids"], srt["offsets"], E)[:rows]
    sid = srt["sorted_ids"][:rows]
    x_rows = d["hidden_states"].cpu()[torch.from_numpy(sid // k).long()]
    w1 = tuple(t.cpu() for t in d["w_gate_up"])
    ref_act = oracle.expert_act_w4(x_rows, eo, w1, oracle.BF16, activation=ACT_CODES[activation])
    assert act.dtype == torch.float16  # the NVFP4 GEMMs compute in f16
    assert_rounded_close(act[:rows], ref_act, torch.float16, what=f"w4 act {activation} T={T}")

    a_in = inputs.random_rows(act.shape[0], F, seed=5, dtype=torch.float16, std=0.5)
    a_in = a_in.to(cuda_device)
    tw = inputs.random_weights(T * k, seed=6).to(cuda_device)
    y = B.moe_gemm2_w4a16(a_in, sorted_ids, offsets, tw, w2_packed, T, k)
    torch.cuda.synchronize()
    scale = tw.cpu().numpy().astype(np.float64)[sid]
    w2 = tuple(t.cpu() for t in d["w_down"])
    ref_y = oracle.expert_down_w4(a_in[:rows].cpu(), eo, scale, w2, oracle.F16)
    assert_rms_close(y[:rows], ref_y, tol=1e-4, what=f"w4 y_route T={T} H={H} F={F}")
    assert B.get_device_status(B._workspace(0, cuda_device)) == B.MOE_OK


SMALL = [
    W("w4-direct-t4", T=4, H=256, E=16, F=128, top_k=4, weights="nvfp4"),
    W("w4-direct-t8-k8", T=8, H=384, E=64, F=256, top_k=8, weights="nvfp4"),
    # 128 routes on the direct path: past the 64-row two-CTA kernel (its epilogue keeps one
    # entry per route), so the 128-row kernel runs it
    W("w4-direct-t8-k16", T=8, H=256, E=64, F=128, top_k=16, weights="nvfp4"),
    W("w4-sorted-t37-sigmoid", T=37, H=256, E=12, F=256, top_k=3, scoring_func="sigmoid",
      bias_std=0.1, routed_scaling_factor=2.5, weights="nvfp4"),
    W("w4-sorted-t300-gathered", T=300, H=256, E=8, F=128, top_k=2, weights="nvfp4"),
    W("w4-sorted-t200-grouped-gelu", T=200, H=384, E=32, F=128, top_k=4, scoring_func="sigmoid",
      bias_std=0.1, num_expert_group=4, topk_group=2, routed_scaling_factor=2.5,
      activation="gelu_tanh", weights="nvfp4"),
    W("w4-sorted-t64-relu2", T=64, H=256, E=8, F=384, top_k=2, activation="relu2",
      weights="nvfp4"),
    # gathered rows, 10 routes per expert on average: 32-row gate/up tiles; the skew gives some
    # experts several tiles
    W("w4-sorted-t160-32row-tiles-skewed", T=160, H=256, E=64, F=128, top_k=4, skew_alpha=0.5,
      weights="nvfp4"),
]


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fused_w4a16_matches_oracle(w, cuda_device):
    d = inputs.generate(w, seed=2, device=cuda_device)
    out = run_fused(w, d)
    ids, _ = run_route(w, d)
    torch.cuda.synchronize()
    ref, r_ids, _, _, noise = oracle_fused(w, d)
    assert np.array_equal(ids.cpu().numpy(), r_ids)
    assert_output_close(out, ref, w.dtype, noise, what=w.name)
    assert B.get_device_status(B._workspace(0, cuda_device)) == B.MOE_OK


def _shard_weights(t, sl):
    return tuple(x[sl] for x in t) if isinstance(t, tuple) else t[sl]


def check_shards_sum_to_full(w, dev, seed, n_sample=None):
    """Expert parallelism checked by its defining property: the E / ep_local shards of one full
    expert set, each run on the GPU with only its slice of the weights and routing over all E
    experts, add up to the full MoE output.  Each shard's rows with no local route are exactly
    zero.  The sum is compared with the full oracle under the usual bound, plus half an ulp per
    shard (each shard's output is rounded to bf16/f16 once).  The shared expert, when present,
    runs on shard 0 only, as one would deploy it."""
    wf = w.with_(ep_local=0, ep_offset=0)
    d = inputs.generate(wf, seed=seed, device=dev)
    routed = oracle_route(wf, d)
    El = w.ep_local
    total, hu = None, None
    for r in range(w.E // El):
        sl = slice(r * El, (r + 1) * El)
        ws = w.with_(ep_offset=r * El, S=w.S if r == 0 else 0)
        dr = {k: v for k, v in d.items() if k != "w4_packed"}
        dr["w_gate_up"] = _shard_weights(d["w_gate_up"], sl)
        dr["w_down"] = _shard_weights(d["w_down"], sl)
        if r:
            dr["shared_w_gate_up"] = dr["shared_w_down"] = None
        out = run_fused(ws, dr)
        torch.cuda.synchronize()
        o = to_np(out)
        dead = ~np.any(local_ids(ws, routed[0]) >= 0, axis=1)
        if ws.S == 0:
            assert np.all(o[dead] == 0.0), f"shard {r}: rows with no local route are not zero"
        total = o.astype(np.float64) if total is None else total + o
        hu = half_ulp(o, w.dtype) if hu is None else hu + half_ulp(o, w.dtype)
    tokens = (np.arange(w.T) if n_sample is None
              else np.unique(np.linspace(0, w.T - 1, n_sample).astype(np.int32)))
    ref, _, _, _, noise = oracle_fused(wf, d, tokens=tokens, routed=routed)
    got, hu = total[tokens], hu[tokens]
    # each shard's output was rounded once: the half ulps of the shards replace the one of a
    # single output (with the binade-crossing margin of the shards' own values)
    assert_output_close(got, ref, w.dtype, noise, what=w.name + " shard sum",
                        extra_ulps=hu * (1 + 2.0 ** -7))
    del d
    torch.cuda.empty_cache()


SHARDED = [
    W("w4-ep-shards-t6", T=6, H=256, E=32, F=128, top_k=4, scoring_func="sigmoid",
      bias_std=0.01, num_expert_group=4, topk_group=2, routed_scaling_factor=2.5,
      weights="nvfp4", ep_local=8),
    W("w4-ep-shards-t160", T=160, H=256, E=32, F=256, top_k=4, scoring_func="sigmoid",
      bias_std=0.01, num_expert_group=4, topk_group=2, routed_scaling_factor=2.5,
      weights="nvfp4", ep_local=8),
    W("bf16-ep-shards-t160", T=160, H=256, E=32, F=192, top_k=4, ep_local=8),
    W("bf16-ep-shards-t5-shared", T=5, H=192, E=16, F=64, top_k=2, ep_local=4, S=128),
]


@pytest.mark.parametrize("w", SHARDED, ids=lambda w: w.name)
def test_expert_parallel_shards_sum_to_full_output(w, cuda_device):
    check_shards_sum_to_full(w, cuda_device, seed=2)


def test_shard_route_ids_are_local(cuda_device):
    w = SHARDED[1].with_(ep_offset=8)
    d = inputs.generate(w, seed=3, device=cuda_device)
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor,
                          ep_num_local=w.ep_local, ep_local_offset=w.ep_offset)
    ids = torch.empty((w.T, w.top_k), dtype=torch.int32, device=cuda_device)
    wts = torch.empty((w.T, w.top_k), dtype=torch.float32, device=cuda_device)
    B._check(B.lib().moe_route(B.ctypes.byref(prob), B._p(d["gating_output"]),
                               B._p(d["correction_bias"]), B._p(ids), B._p(wts), None),
             "moe_route")
    torch.cuda.synchronize()
    g_ids, _, _ = oracle_route(w, d)
    assert np.array_equal(ids.cpu().numpy(), local_ids(w, g_ids))


def test_w4a16_is_deterministic_and_graph_replayable(cuda_device):
    w = SMALL[3]
    d = inputs.generate(w, seed=4, device=cuda_device)
    a = run_fused(w, d).clone()
    b = run_fused(w, d).clone()
    assert torch.equal(a, b)
    out = torch.empty_like(a)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        run_fused(w, d, out=out)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        run_fused(w, d, out=out)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, a)


SPLIT = [
    # units = active experts x F/128, few against the SMs, and 8 K steps each: every unit's K
    # range is split in two
    W("w4-split-t16", T=16, H=1024, E=8, F=640, top_k=2, weights="nvfp4"),
    # odd number of 128-k steps (9: halves of 4 and 5), GeGLU-tanh, sigmoid routing
    W("w4-split-t24-odd-k-gelu", T=24, H=1152, E=6, F=256, top_k=3, scoring_func="sigmoid",
      bias_std=0.1, routed_scaling_factor=2.5, activation="gelu_tanh", weights="nvfp4"),
    # ReLU2: 256-row units whose second half can be empty
    W("w4-split-t40-relu2", T=40, H=1024, E=8, F=384, top_k=2, activation="relu2",
      weights="nvfp4"),
]


@pytest.mark.parametrize("w", SPLIT, ids=lambda w: w.name)
def test_w4a16_split_k_matches_oracle_and_unsplit_run(w, cuda_device):
    """The gate/up GEMM's split-K path (workspace of moe_workspace_size_w4a16 bytes) and the
    unsplit one (moe_workspace_size bytes) each match the oracle and are deterministic, and they
    agree with each other to a few f32 roundings.  The split path's per-unit counters, which
    sit right after the common workspace, end each call at 2 (both halves counted in)."""
    d = inputs.generate(w, seed=7, device=cuda_device)
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor, 0,
                          w.activation)
    n_small, n_big = B.workspace_size(prob), B.workspace_size_w4a16(prob)
    assert n_big > n_small
    ws_small = B.new_workspace(n_small, cuda_device)
    ws_big = B.new_workspace(n_big, cuda_device)
    ref, _, _, _, noise = oracle_fused(w, d)
    outs = {}
    for name, ws in (("unsplit", ws_small), ("split", ws_big)):
        a = run_fused(w, d, workspace=ws).clone()
        b = run_fused(w, d, workspace=ws).clone()
        torch.cuda.synchronize()
        assert B.get_device_status(ws) == B.MOE_OK
        assert torch.equal(a, b), f"{w.name} {name}: repeat call not bit-identical"
        assert_output_close(a, ref, w.dtype, noise, what=f"{w.name} {name}")
        outs[name] = a
    cnt = ws_big[n_small:n_small + 4 * 64].view(torch.int32).cpu().numpy()
    assert set(np.unique(cnt)) <= {0, 2} and cnt.max() == 2, f"split counters {cnt[:16]}"
    # A workspace whose every byte past the status header starts as 0xFF (counters at -1,
    # partials NaN): the sort zeroes the counters and each half writes its partials before the
    # other reads them, so the result is the clean run's, bit for bit.
    poison = B.new_workspace(n_big, cuda_device)
    poison[256:] = 0xFF
    c = run_fused(w, d, workspace=poison).clone()
    torch.cuda.synchronize()
    assert B.get_device_status(poison) == B.MOE_OK
    assert torch.equal(c, outs["split"]), f"{w.name}: poisoned split workspace changed the output"
    # Each output is rounded once to bf16 from f32 sums that differ only in their grouping
    # (and through gemm1's bf16-rounded activations): within one ulp plus a sliver of the RMS.
    sp, un = to_np(outs["split"]), to_np(outs["unsplit"])
    rms = float(np.sqrt(np.mean(un * un)))
    err = np.abs(sp - un)
    bound = 2 * half_ulp(np.abs(un) * (1 + 2.0 ** -7), w.dtype) + 2e-3 * rms
    log_parity(f"{w.name} split vs unsplit", max_err_over_rms=float(err.max()) / rms)
    assert np.all(err <= bound), f"{w.name}: split and unsplit differ by {err.max():.3e}"


RANGE_CASES = [
    ("token rows, a hidden value past f16", W("r1", T=16, H=256, E=8, F=128, top_k=2,
                                              weights="nvfp4"), "hidden"),
    ("gathered rows, a hidden value past f16", W("r2", T=200, H=256, E=8, F=128, top_k=2,
                                                 weights="nvfp4"), "hidden"),
    ("act past f16 from in-range tokens", W("r3", T=16, H=256, E=8, F=128, top_k=2,
                                            weights="nvfp4"), "act"),
]


@pytest.mark.parametrize("what,w,kind", RANGE_CASES, ids=[c[0] for c in RANGE_CASES])
def test_w4a16_flags_values_past_the_f16_range(what, w, kind, cuda_device):
    """The NVFP4 path computes in f16: a bf16 hidden value of 65536 (the first past f16's
    range), or an act that grows past it, sets MOE_ERR_F16_RANGE in the status word; the same
    inputs brought into range leave it clear."""
    d = inputs.generate(w, seed=4, device=cuda_device)
    x = d["hidden_states"]
    if kind == "hidden":
        # hidden column 5 meets only zero gate/up weights (E2M1 code 0: element 5 is the high
        # nibble of byte 2), so only the token-row conversion can see the value there
        d["w_gate_up"][0][:, :, 2] &= 0x0F
        x[3, 5] = 65536.0
    else:  # every token 2000: gate and up values near 2000, act near 2000 * 2000
        x.fill_(2000.0)
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor, 0,
                          w.activation)
    ws = B.new_workspace(B.workspace_size(prob), cuda_device)
    run_fused(w, d, workspace=ws)
    torch.cuda.synchronize()
    assert B.get_device_status(ws) == B.MOE_ERR_F16_RANGE, what
    if kind == "hidden":
        x[3, 5] = 60000.0  # in range: exact in f16
    else:
        x.fill_(2.0)
    ws2 = B.new_workspace(B.workspace_size(prob), cuda_device)
    run_fused(w, d, workspace=ws2)
    torch.cuda.synchronize()
    assert B.get_device_status(ws2) == B.MOE_OK, what


def test_w4a16_rejects_unsupported_shapes(cuda_device):
    w = W("bad", T=4, H=192, E=4, F=128, top_k=2, weights="nvfp4")  # H not a multiple of 128
    d = inputs.generate(w, seed=0, device=cuda_device)
    with pytest.raises(B.MoeError) as ei:
        run_fused(w, d)
    assert ei.value.code == B.MOE_ERR_UNSUPPORTED


FULL = [
    ("qwen3-30b-a3b-decode-t32-w4a16", None),
    ("deepseek-v3-ep8-shard-t512-w4a16", None),
]


@pytest.mark.parametrize("name,n_sample", FULL, ids=[f[0] for f in FULL])
def test_w4a16_full_size_workloads(name, n_sample, cuda_device):
    """W4A16 at full size on one device's experts; for the EP8 shard every expert is local
    here (ep_local = 0), the shard semantics being checked by the shard-sum tests."""
    w = inputs.VARIANTS[name].with_(ep_local=0)
    d = inputs.generate(w, seed=0, device=cuda_device)
    out = run_fused(w, d)
    ids, wts = run_route(w, d)
    torch.cuda.synchronize()
    routed = oracle_route(w, d)
    assert np.array_equal(ids.cpu().numpy(), routed[0]), "routing ids differ"
    tokens = (np.arange(w.T) if n_sample is None
              else np.unique(np.linspace(0, w.T - 1, n_sample).astype(np.int32)))
    ref, _, _, _, noise = oracle_fused(w, d, tokens=tokens, routed=routed)
    assert_output_close(out[torch.from_numpy(tokens).to(cuda_device).long()], ref, w.dtype, noise,
                        what=name)
    out2 = run_fused(w, d)
    assert torch.equal(out, out2), "repeat call not bit-identical"
    assert B.get_device_status(B._workspace(0, cuda_device)) == B.MOE_OK
    del d
    torch.cuda.empty_cache()


@pytest.mark.parametrize("name,n_sample", [("deepseek-v3-ep8-shard-t32-w4a16", None),
                                           ("deepseek-v3-ep8-shard-t32", None),
                                           ("deepseek-v3-ep8-shard-t4096", 512)],
                         ids=["t32-w4a16", "t32-bf16", "t4096-bf16"])
def test_ep8_shards_of_deepseek_v3_sum_to_full_output(name, n_sample, cuda_device):
    """The eight EP8 shards of DeepSeek-V3 (32 experts each), run one after another."""
    check_shards_sum_to_full(inputs.VARIANTS[name], cuda_device, seed=0, n_sample=n_sample)


def _pack_reference(codes, scales):
    """The packed tile layout, written out in numpy from its definition in include/moe.h."""
    n, rows, half_k = codes.shape
    K = half_k * 2
    out = []
    for m in range(n):
        for s in range(rows // 128):
            for b in range(K // 128):
                tile = np.zeros(9216, np.uint8)
                for r in range(128):
                    row = codes[m, s * 128 + r, b * 64:(b + 1) * 64]
                    for j in range(4):
                        pos = j ^ ((r >> 1) & 3)
                        tile[r * 64 + pos * 16:r * 64 + pos * 16 + 16] = row[j * 16:j * 16 + 16]
                    tile[8192 + r * 8:8192 + r * 8 + 8] = scales[m, s * 128 + r, b * 8:b * 8 + 8]
                out.append(tile)
    return np.concatenate(out)


@pytest.mark.parametrize("n,rows,K", [(1, 128, 128), (3, 256, 384)])
def test_nvfp4_pack_matches_its_layout_definition(n, rows, K, cuda_device):
    g = torch.Generator().manual_seed(rows + K)
    codes = torch.randint(0, 256, (n, rows, K // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    scales = torch.randint(0, 256, (n, rows, K // 16), generator=g,
                           dtype=torch.int32).to(torch.uint8)
    alpha = torch.ones(n, dtype=torch.float32)
    w = B.pack_nvfp4_weights(codes.to(cuda_device), scales.to(cuda_device),
                             alpha.to(cuda_device))
    torch.cuda.synchronize()
    assert np.array_equal(w.tiles.cpu().numpy(), _pack_reference(codes.numpy(), scales.numpy()))


def test_nvfp4_pack_rejects_unaligned_sizes(cuda_device):
    codes = torch.zeros((1, 64, 64), dtype=torch.uint8, device=cuda_device)
    scales = torch.zeros((1, 64, 8), dtype=torch.uint8, device=cuda_device)
    with pytest.raises(B.MoeError):
        B.pack_nvfp4_weights(codes, scales, torch.ones(1, device=cuda_device))
