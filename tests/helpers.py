"""Shared helpers of the GPU parity tests: run the oracle on the same seeded inputs the CUDA path
gets (copied to the host), and compare with the tolerance max|gpu - oracle| <= 1e-2 * RMS."""
import math

import numpy as np
import torch

import oracle
from mixture_experts_forward_moe_gb300 import binding as B
from mixture_experts_forward_moe_gb300 import inputs

RMS_TOL = 1e-2  # max |gpu - oracle| <= RMS_TOL * RMS(oracle), bf16/f16 with f32 accumulation


def dt_code(dtype):
    return oracle.BF16 if dtype == torch.bfloat16 else oracle.F16


def to_np(x):
    if isinstance(x, torch.Tensor):
        return x.detach().double().cpu().numpy()
    return np.asarray(x, dtype=np.float64)


def assert_rms_close(gpu, ref, tol=RMS_TOL, what=""):
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    rms = math.sqrt(float(np.mean(r * r))) if r.size else 0.0
    err = float(np.max(np.abs(g - r))) if r.size else 0.0
    assert err <= tol * rms + 1e-30, f"{what}: max|gpu-ref|={err:.3e} > {tol}*RMS={tol * rms:.3e}"
    return err / rms if rms > 0 else 0.0


def scoring_code(w):
    return oracle.SOFTMAX if w.scoring_func == "softmax" else oracle.SIGMOID


def oracle_route(w, d):
    bias = None if d["correction_bias"] is None else d["correction_bias"].cpu().numpy()
    return oracle.route(d["gating_output"].cpu().numpy(), w.top_k, scoring_code(w),
                        w.renormalize, w.num_expert_group, w.topk_group,
                        w.routed_scaling_factor, bias)


def oracle_fused(w, d, tokens=None, routed=None):
    """fp64 oracle output for `tokens` (all when None), its ids and weights.  Only the experts
    the listed tokens use are copied to the host."""
    ids, wts, near = routed if routed is not None else oracle_route(w, d)
    tl = np.arange(w.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    used = sorted(set(int(e) for e in ids[tl].reshape(-1) if e >= 0))
    slot = np.full(w.E, -1, np.int32)
    slot[used] = np.arange(len(used), dtype=np.int32)
    idx = torch.tensor(used, dtype=torch.long, device=d["w_gate_up"].device)
    wgu = d["w_gate_up"].index_select(0, idx).cpu() if used else d["w_gate_up"][:1].cpu()
    wd = d["w_down"].index_select(0, idx).cpu() if used else d["w_down"][:1].cpu()
    sgu = None if d["shared_w_gate_up"] is None else d["shared_w_gate_up"].cpu()
    sd = None if d["shared_w_down"] is None else d["shared_w_down"].cpu()
    out = oracle.moe_tokens(d["hidden_states"].cpu(), ids, wts, wgu, wd, dt_code(w.dtype),
                            tokens=tl, expert_slot=slot, num_experts=w.E,
                            shared_w_gate_up=sgu, shared_w_down=sd)
    return out, ids, wts, near


def run_fused(w, d, **kw):
    return B.fused_moe_fwd(d["hidden_states"], d["gating_output"], d["w_gate_up"], d["w_down"],
                           correction_bias=d["correction_bias"],
                           shared_w_gate_up=d["shared_w_gate_up"],
                           shared_w_down=d["shared_w_down"], **w.kwargs(), **kw)


def run_route(w, d):
    return B.moe_route(d["gating_output"], w.top_k, w.scoring_func, w.renormalize,
                       d["correction_bias"], w.num_expert_group, w.topk_group,
                       w.routed_scaling_factor)
