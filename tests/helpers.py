"""Shared helpers of the GPU parity tests: run the oracle on the same seeded inputs the CUDA path
gets (copied to the host), and compare with the tolerance max|gpu - oracle| <= 1e-2 * RMS."""
import json
import math
import os

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


def half_ulp(x, dtype):
    """Half the spacing of `dtype` (bf16: 8 significant bits, f16: 11) at |x|: the largest
    error of one round-to-nearest of a value of that magnitude."""
    bits = 8 if dtype == torch.bfloat16 else 11
    tiny = 2.0 ** -133 if dtype == torch.bfloat16 else 2.0 ** -25  # half the subnormal step
    a = np.abs(np.asarray(x, dtype=np.float64))
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.maximum(np.where(a > 0, np.exp2(e - bits), 0.0), tiny)


PARITY_RECORDS = []  # every log_parity record of this session (conftest prints the summaries)


def log_parity(what, **kw):
    PARITY_RECORDS.append(dict(what=what, **kw))
    path = os.environ.get("MOE_PARITY_LOG")
    if path:
        with open(path, "a") as f:
            f.write(json.dumps(dict(what=what, **kw)) + "\n")


def assert_rms_close(gpu, ref, tol=RMS_TOL, what=""):
    """max |gpu - ref| <= tol * RMS(ref) (intermediates kept in f32)."""
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    rms = math.sqrt(float(np.mean(r * r))) if r.size else 0.0
    err = float(np.max(np.abs(g - r))) if r.size else 0.0
    log_parity(what, max_err_over_rms=err / rms if rms else 0.0, tol=tol)
    assert err <= tol * rms + 1e-30, f"{what}: max|gpu-ref|={err:.3e} > {tol}*RMS={tol * rms:.3e}"
    return err / rms if rms > 0 else 0.0


def assert_rounded_close(gpu, ref, dtype, rel_rms=1e-3, what=""):
    """A 16-bit output rounded once from an f32 value: |gpu - ref| <= half an ulp of the
    dtype at |ref| (allowing for a crossing into the next binade) + rel_rms * RMS(ref)."""
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    if not r.size:
        return 0.0
    rms = math.sqrt(float(np.mean(r * r)))
    err = np.abs(g - r)
    bound = half_ulp(np.abs(r) * (1 + 2.0 ** -7), dtype) + rel_rms * rms
    worst = int(np.argmax(err - bound))
    log_parity(what, max_err_over_rms=float(err.max()) / rms, rounded_rel_rms=rel_rms)
    assert np.all(err <= bound), (f"{what}: |gpu-ref|={err.flat[worst]:.3e} at ref="
                                  f"{r.flat[worst]:.4e} > bound {bound.flat[worst]:.3e}")
    return float(err.max()) / rms


ACT_Z = 7.0          # standard deviations of the act-rounding error allowed per element
SLACK_RMS = 1e-3     # f32 accumulation, f32 route rows and weights, fast SiLU: all far below


def assert_output_close(gpu, ref, dtype, noise=None, tol=RMS_TOL, what="", extra_ulps=None):
    """The fused output against the fp64 oracle.

    Every element must satisfy
        |gpu - oracle| <= half_ulp(|oracle|) + ACT_Z * sigma + SLACK_RMS * RMS(oracle)
    where half_ulp is the final rounding to the output dtype (extra_ulps replaces it when several
    rounded outputs were summed) and sigma = noise / sqrt(3) is the standard deviation of the
    error that rounding each act value to the 16-bit dtype before the down projection adds
    (noise from oracle.moe_tokens(..., act_noise=True); each rounding error is uniform within
    +-half an ulp of its act value).  Where noise is None, or for f16 outputs in addition, the
    stated bound |gpu - oracle| <= tol * RMS + half_ulp is checked.  Logs the plain
    max|gpu - oracle| / RMS, the same after half an ulp, and the worst element's error in sigmas."""
    g, r = to_np(gpu), to_np(ref)
    assert g.shape == r.shape, (what, g.shape, r.shape)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU values"
    if not r.size:
        return 0.0
    rms = math.sqrt(float(np.mean(r * r)))
    err = np.abs(g - r)
    hu = half_ulp(r, dtype) if extra_ulps is None else extra_ulps
    hu_x = half_ulp(np.abs(r) * (1 + 2.0 ** -7), dtype) if extra_ulps is None else extra_ulps
    excess = float(np.max(err - hu)) / rms
    rec = dict(max_err_over_rms=float(err.max()) / rms, max_err_minus_half_ulp_over_rms=excess,
               tol=tol, rows=int(r.shape[0]) if r.ndim > 1 else 1, summary=True)
    checks = []
    if noise is not None:
        sigma = np.asarray(noise, np.float64) / math.sqrt(3.0)
        assert sigma.shape == r.shape, (what, sigma.shape, r.shape)
        over = err - hu_x - SLACK_RMS * rms
        z = np.where(sigma > 0, over / np.where(sigma > 0, sigma, 1.0),
                     np.where(over > 0, np.inf, 0.0))
        rec["max_z"] = float(np.max(z))
        rec["over_stated"] = int(np.sum(err > tol * rms + hu))
        checks.append(("derived", z <= ACT_Z, z))
    if noise is None or dtype == torch.float16:
        checks.append(("stated", err <= tol * rms + hu, err - hu))
    log_parity(what, **rec)
    for name, ok, score in checks:
        worst = int(np.argmax(score))
        assert np.all(ok), (f"{what}: |gpu-ref|={err.flat[worst]:.3e} at ref={r.flat[worst]:.4e} "
                            f"exceeds the {name} bound (RMS {rms:.3e}, half ulp "
                            f"{hu.flat[worst]:.3e}" + (f", {ACT_Z} sigma "
                            f"{ACT_Z * float(np.asarray(noise).flat[worst]) / math.sqrt(3):.3e}"
                            if name == "derived" else "") + ")")
    return float(err.max()) / rms


NEAR_TIE = 1e-6  # fp64 gap at a selection boundary below which the f32 keys may choose otherwise


def check_ids_against_plain_selection(w, d, ids, what=""):
    """Sigmoid routing: the GPU's ids (chosen on f32 keys) against the selection of the plain
    fp64 definition (oracle.route_select_f64: fp64 sigmoid + bias, groups by the sum of the two
    largest keys, ties to the lower index).  On every token whose fp64 boundary gap is at
    least NEAR_TIE the experts must be the same, and in the same order where consecutive
    selected keys are also that far apart.  Returns (tokens, near-tie tokens at a boundary,
    tokens with near-equal selected keys), also written to the parity log."""
    if w.scoring_func != "sigmoid":
        return None
    got = ids.cpu().numpy() if isinstance(ids, torch.Tensor) else np.asarray(ids)
    bias = None if d["correction_bias"] is None else d["correction_bias"].cpu().numpy()
    ref, bgap, ogap = oracle.route_select_f64(d["gating_output"].cpu().numpy(), w.top_k,
                                              w.num_expert_group, w.topk_group, bias)
    clear = bgap >= NEAR_TIE
    same_set = np.all(np.sort(got, axis=1) == np.sort(ref, axis=1), axis=1)
    bad = np.nonzero(clear & ~same_set)[0]
    assert bad.size == 0, f"{what}: ids differ from the fp64 selection on tokens {bad[:10]}"
    ordered = clear & (ogap >= NEAR_TIE)
    assert np.array_equal(got[ordered], ref[ordered]), f"{what}: id order differs from fp64"
    counts = (int(got.shape[0]), int((~clear).sum()), int((clear & ~ordered).sum()))
    log_parity(what, tokens=counts[0], near_tie_tokens=counts[1], order_near_tie_tokens=counts[2])
    print(f"{what}: ids equal the fp64 selection on {counts[0] - counts[1]} of {counts[0]} "
          f"tokens ({counts[1]} near-tie at a boundary, {counts[2]} with near-equal keys)")
    return counts


def scoring_code(w):
    return oracle.SOFTMAX if w.scoring_func == "softmax" else oracle.SIGMOID


ACT_CODES = {"silu": oracle.ACT_SILU, "gelu_tanh": oracle.ACT_GELU_TANH,
             "relu2": oracle.ACT_RELU2}


def oracle_route(w, d):
    bias = None if d["correction_bias"] is None else d["correction_bias"].cpu().numpy()
    return oracle.route(d["gating_output"].cpu().numpy(), w.top_k, scoring_code(w),
                        w.renormalize, w.num_expert_group, w.topk_group,
                        w.routed_scaling_factor, bias)


def local_ids(w, ids):
    """The router's global ids as indices of the shard's experts (-1 outside the shard)."""
    if w.ep_local <= 0:
        return ids
    off = w.ep_offset
    return np.where((ids >= off) & (ids < off + w.ep_local), ids - off, -1).astype(np.int32)


def oracle_fused(w, d, tokens=None, routed=None):
    """fp64 oracle output for `tokens` (all when None), its (global) ids, weights, near-tie
    flags and the per-element act-rounding noise scale.  Only the experts the listed tokens use
    are copied to the host (16-bit weights)."""
    ids, wts, near = routed if routed is not None else oracle_route(w, d)
    tl = np.arange(w.T, dtype=np.int32) if tokens is None else np.asarray(tokens, np.int32)
    lids = local_ids(w, ids)
    if w.weights == "nvfp4":
        w1 = tuple(t.cpu() for t in d["w_gate_up"])
        w2 = tuple(t.cpu() for t in d["w_down"])
        # the NVFP4 path keeps its act in f16
        out, noise = oracle.moe_tokens_w4(d["hidden_states"].cpu(), lids, wts, w1, w2,
                                          dt_code(w.dtype), tokens=tl,
                                          activation=ACT_CODES[w.activation], act_noise=True,
                                          act_dtype=oracle.F16)
        return out, ids, wts, near, noise
    ids_g, ids = ids, lids
    used = sorted(set(int(e) for e in ids[tl].reshape(-1) if e >= 0))
    slot = np.full(w.E_local, -1, np.int32)
    slot[used] = np.arange(len(used), dtype=np.int32)
    if len(used) == w.E_local:  # every expert: copy the weights as they are
        wgu, wd = d["w_gate_up"].cpu(), d["w_down"].cpu()
    else:
        idx = torch.tensor(used, dtype=torch.long, device=d["w_gate_up"].device)
        wgu = d["w_gate_up"].index_select(0, idx).cpu() if used else d["w_gate_up"][:1].cpu()
        wd = d["w_down"].index_select(0, idx).cpu() if used else d["w_down"][:1].cpu()
    sgu = None if d["shared_w_gate_up"] is None else d["shared_w_gate_up"].cpu()
    sd = None if d["shared_w_down"] is None else d["shared_w_down"].cpu()
    out, noise = oracle.moe_tokens(d["hidden_states"].cpu(), ids, wts, wgu, wd,
                                   dt_code(w.dtype), tokens=tl, expert_slot=slot,
                                   num_experts=w.E_local, shared_w_gate_up=sgu, shared_w_down=sd,
                                   activation=ACT_CODES[w.activation], act_noise=True)
    return out, ids_g, wts, near, noise


def packed_w4(d):
    """The NVFP4 weights of input dict d in the library's packed layout (packed once, kept in d)."""
    if "w4_packed" not in d:
        d["w4_packed"] = (B.pack_nvfp4_weights(*d["w_gate_up"]), B.pack_nvfp4_weights(*d["w_down"]))
    return d["w4_packed"]


def run_fused(w, d, **kw):
    if w.weights == "nvfp4":
        w1, w2 = packed_w4(d)
        return B.fused_moe_fwd_w4a16(d["hidden_states"], d["gating_output"], w1, w2,
                                     correction_bias=d["correction_bias"], **w.kwargs(), **kw)
    return B.fused_moe_fwd(d["hidden_states"], d["gating_output"], d["w_gate_up"], d["w_down"],
                           correction_bias=d["correction_bias"],
                           shared_w_gate_up=d["shared_w_gate_up"],
                           shared_w_down=d["shared_w_down"], **w.kwargs(), **kw)


def run_route(w, d):
    return B.moe_route(d["gating_output"], w.top_k, w.scoring_func, w.renormalize,
                       d["correction_bias"], w.num_expert_group, w.topk_group,
                       w.routed_scaling_factor)
