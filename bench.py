#!/usr/bin/env python
"""Benchmark of the GB300 fused MoE forward (one JSON line on rank 0).

A step is one fused_moe_fwd call (router, sort, gather, gemm1 + SwiGLU, gemm2 x route weight,
combine, shared expert when present) over one batch of seeded synthetic inputs that are already
resident in HBM.  When a step streams more than twice the L2 in expert weights (every measured
workload but the tiny one) nothing is flushed between steps; otherwise the L2 is flushed outside
the timed events by a 256 MiB write followed by a 256 MiB read (clean lines, no write-back).
A step is one replay of a CUDA graph that holds one captured fused_moe_fwd call (its kernels
and their programmatic dependencies), so the host issues one launch per step; `--eager` times
the eager calls instead, and the eager time is reported beside it in any case.  Each step is
timed with a CUDA event pair on the launching stream; the K step times are summed.  `value` is whole-job TFLOP/s with the TileOPs MoE page's FLOP count
2*T*k*3*F*H (+ 2*T*3*S*H).

Also reported: HBM GB/s over the algorithmic bytes, the roofline of the dominant kernel (its
event-timed average launch against the measured HBM copy peak), an end-to-end figure through
the public API from pinned host buffers (host->device inputs and device->host output inside the
timed region), SM clocks sampled during the timed region, and the CPU oracle timed on the
host's cores on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun every rank runs its own replica of the workload on its own GPU (no collective on
the data path: weak scaling); the timed region is bracketed by a barrier and a synchronize on
both sides and the slowest rank's time is used.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT_WORKLOAD = "deepseek-v3-grouped-prefill-t4096"
METRIC = "fused_moe_fwd device ms, TFLOP/s & HBM GB/s; % of GB300 roofline per config"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 126 << 20  # GB300 L2 (about 129 MB)


class L2Flush:
    """Evicts the L2 between timed steps, outside their events: a 256 MiB write (the flush), then
    a 256 MiB read of another buffer, so the lines left behind are clean and unrelated to the
    step and the next step pays no write-back of the flush's dirty lines."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        self.r.sum()

    note = "flushed between steps outside the timed events (256 MiB write, then 256 MiB read)"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0

# Throughput printed on the TileOPs benchmark page ("MoE" section, FusedMoEFwd and
# FusedMoESharedExpertFwd tables) for the same shapes; hardware not stated there.
# Context only (other hardware, other routing seed): the W4A16 PR's B300 medians, ms per call of
# one DeepSeek-V3 EP8 rank (flashinfer PR #4048, CuTe W4A16 inference / TRTLLM BF16 columns).
PUBLISHED_MS = {
    "deepseek-v3-ep8-shard-t32-w4a16": 0.118, "deepseek-v3-ep8-shard-t512-w4a16": 0.169,
    "deepseek-v3-ep8-shard-t4096-w4a16": 0.363, "deepseek-v3-ep8-shard-t32": 0.285,
    "deepseek-v3-ep8-shard-t512": 0.435, "deepseek-v3-ep8-shard-t4096": 0.529,
}

PUBLISHED_TFLOPS = {
    ("qwen3-30b-a3b-decode-t32", "bf16"): 9.11,
    ("qwen3-235b-a22b-decode-t512", "bf16"): 128.0,
    ("qwen3-235b-a22b-decode-t512", "f16"): 129.0,
    ("deepseek-v3-grouped-prefill-t4096", "bf16"): 406.0,
    ("kimi-k2-shared-t512", "bf16"): 151.0,
}


# ----------------------------------------------------------------------- rank helpers (CPU ok)
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", str(rank)))
    return ws, rank, local


def max_over_ranks(x: float) -> float:
    """The largest x over all ranks (x itself without a process group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([float(x)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def job_throughput(units_per_rank: float, n_ranks: int, steps: int, max_ms: float) -> float:
    """Whole-job rate: units every rank processed in `steps` steps over the slowest rank's time."""
    return units_per_rank * n_ranks * steps / (max_ms * 1e-3)


# --------------------------------------------------------------------------------- accounting
def elt_bytes(w) -> int:
    return 2


def weight_bytes_per_elem(w) -> float:
    """Bytes per routed-expert weight: 2 (bf16/f16), or 0.5 + 1/16 for NVFP4 (an E2M1 code and
    a sixteenth of an E4M3 block scale)."""
    return 0.5 + 1.0 / 16.0 if w.weights == "nvfp4" else float(elt_bytes(w))


def algorithmic_bytes(w, n_unique: int, P=None) -> dict:
    """Bytes the path must move at least once (weights of the experts touched, activations).
    P: routes computed here (T * top_k, or the routes to local experts on a shard)."""
    eb = elt_bytes(w)
    wb = weight_bytes_per_elem(w)
    P = w.T * w.top_k if P is None else P
    g = 2 if w.gated else 1  # gate/up matrices per expert (ReLU2 has a single projection)
    weights = n_unique * (g + 1) * w.F * w.H * wb + (g + 1) * w.S * w.H * eb
    acts = w.T * w.H * eb * 2 + w.T * w.E * 4 + (w.E * 4 if w.bias_std > 0 else 0)
    direct = w.T <= 8 and P <= 128
    b1 = w.T * w.H * eb if direct else P * w.H * eb  # gemm1 token rows read
    return dict(
        total=weights + acts,
        gemm1=n_unique * g * w.F * w.H * wb + b1 + P * w.F * eb,
        gemm2=n_unique * w.H * w.F * wb + P * w.F * eb + P * w.H * 4,  # f32 route rows
        shared_gemm1=g * w.S * w.H * eb + w.T * w.H * eb + w.T * w.S * eb,
        shared_gemm2=w.S * w.H * eb + w.T * w.S * eb + w.T * w.H * 4,  # f32 shared output
    )


def stage_flops(w, P=None) -> dict:
    P = w.T * w.top_k if P is None else P
    g = 2 if w.gated else 1
    return dict(gemm1=2.0 * P * g * w.F * w.H, gemm2=2.0 * P * w.F * w.H,
                shared_gemm1=2.0 * w.T * g * w.S * w.H, shared_gemm2=2.0 * w.T * w.S * w.H)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return (float(d["hbm_gbs"]), float(d["bf16_tflops"]), float(d["bf16_tflops_sustained"]),
                "measured")
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS, 1700.0, "fallback"


GEMM_SOURCES = ("gemm.cu", "gemm_pair.cu", "ptx.cuh", "common.cuh", "nvfp4.cuh")


def _code_only(text: str) -> str:
    """C++ source without its comments, trailing blanks and empty lines: edits to comments
    leave a kernel as it was."""
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    lines = (re.sub(r"//.*", "", ln).rstrip() for ln in text.splitlines())
    return "\n".join(ln for ln in lines if ln)


def kernel_source_hash() -> str:
    """Hash of the code (comments left out) of the sources that define the grouped GEMM kernel
    (the dominant kernel)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "mixture_experts_forward_moe_gb300", "csrc")
    for fn in GEMM_SOURCES:
        with open(os.path.join(csrc, fn), encoding="utf-8") as f:
            h.update(fn.encode() + _code_only(f.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, stage: str):
    """DRAM bytes per launch of `stage` from the committed ncu summary, if the kernels have not
    changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("kernel_source_hash") != kernel_source_hash():
        return None
    return d.get("per_launch_bytes", {}).get(workload, {}).get(stage)


# ------------------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        vis = [v for v in os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",") if v.strip()]
        target = vis[gpu_index].strip() if gpu_index < len(vis) else str(gpu_index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-i", target],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "samples": len(sm), "reasons": sorted(reasons)}


def local_ids(w, ids):
    """Global router ids as indices of this shard's experts (-1 elsewhere); identity when every
    expert is local."""
    import numpy as np
    if w.ep_local <= 0:
        return ids
    off = w.ep_offset
    return np.where((ids >= off) & (ids < off + w.ep_local), ids - off, -1).astype(np.int32)


# ------------------------------------------------------------------------------- CPU oracle arm
class OracleSample:
    """The CPU oracle (routing + per-token expert MLP) on the first n tokens of a workload, n
    sized so that one pass takes about a quarter of `budget_s`.  The setup (the full routing,
    the used experts' weights copied to the host) runs once; `run` then times passes."""

    def __init__(self, w, d, budget_s: float, max_tokens=None):
        import numpy as np
        import torch

        import oracle
        self.w, self.oracle = w, oracle
        gating = d["gating_output"].cpu().numpy()
        self.bias = None if d["correction_bias"] is None else d["correction_bias"].cpu().numpy()
        self.sc = oracle.SOFTMAX if w.scoring_func == "softmax" else oracle.SIGMOID
        ids, wts, _ = oracle.route(gating, w.top_k, self.sc, w.renormalize, w.num_expert_group,
                                   w.topk_group, w.routed_scaling_factor, self.bias)
        self.ids, self.wts = local_ids(w, ids), wts
        self.flops_tok = w.flops(int((self.ids >= 0).sum())) / w.T
        self.cores = oracle.num_threads()
        n = max(1, min(w.T, int(0.25 * budget_s * 2e9 * self.cores / self.flops_tok)))
        if max_tokens:
            n = min(n, max_tokens)
        self.n = n
        self.toks = np.arange(n, dtype=np.int32)
        self.act = {"silu": oracle.ACT_SILU, "gelu_tanh": oracle.ACT_GELU_TANH,
                    "relu2": oracle.ACT_RELU2}[w.activation]
        self.g_n = np.ascontiguousarray(gating[:n])
        self.hid = d["hidden_states"].cpu()
        self.w4 = w.weights == "nvfp4"
        if self.w4:
            self.w1 = tuple(t.cpu() for t in d.get("w_gate_up_canonical", d["w_gate_up"]))
            self.w2 = tuple(t.cpu() for t in d.get("w_down_canonical", d["w_down"]))
            return
        used = sorted(set(int(e) for e in self.ids[:n].reshape(-1) if e >= 0))
        self.slot = np.full(w.E_local, -1, np.int32)
        self.slot[used] = np.arange(len(used), dtype=np.int32)
        idx = torch.tensor(used, dtype=torch.long, device=d["w_gate_up"].device)
        self.wgu = d["w_gate_up"].index_select(0, idx).cpu()
        self.wdn = d["w_down"].index_select(0, idx).cpu()
        self.sgu = None if d["shared_w_gate_up"] is None else d["shared_w_gate_up"].cpu()
        self.sdn = None if d["shared_w_down"] is None else d["shared_w_down"].cpu()
        self.dt = oracle.BF16 if w.dtype == torch.bfloat16 else oracle.F16

    def one_pass(self):
        w, o = self.w, self.oracle
        o.route(self.g_n, w.top_k, self.sc, w.renormalize, w.num_expert_group, w.topk_group,
                w.routed_scaling_factor, self.bias)
        if self.w4:
            o.moe_tokens_w4(self.hid, self.ids, self.wts, self.w1, self.w2, o.BF16,
                            tokens=self.toks, activation=self.act)
        else:
            o.moe_tokens(self.hid, self.ids, self.wts, self.wgu, self.wdn, self.dt,
                         tokens=self.toks, expert_slot=self.slot, num_experts=w.E_local,
                         shared_w_gate_up=self.sgu, shared_w_down=self.sdn, activation=self.act)

    def run(self, budget_s: float):
        """Passes (at least one) until budget_s has elapsed: (seconds, passes)."""
        passes, t0 = 0, time.perf_counter()
        while True:
            self.one_pass()
            passes += 1
            el = time.perf_counter() - t0
            if el >= budget_s or el * (passes + 1) / passes > 3 * budget_s:
                return el, passes

    def flops(self, passes: int) -> float:
        return self.flops_tok * self.n * passes

    def parity(self, out_gpu) -> dict:
        """The GPU output on the sampled tokens against the oracle: max|gpu - oracle| / RMS, the
        same after half an ulp of the final rounding, and the worst element in standard
        deviations of the act-rounding error (the bound of the parity tests is 7)."""
        import numpy as np
        import torch
        w, o = self.w, self.oracle
        if self.w4:
            ref, noise = o.moe_tokens_w4(self.hid, self.ids, self.wts, self.w1, self.w2, o.BF16,
                                         tokens=self.toks, activation=self.act, act_noise=True,
                                         act_dtype=o.F16)  # the NVFP4 path's act is f16
        else:
            ref, noise = o.moe_tokens(self.hid, self.ids, self.wts, self.wgu, self.wdn, self.dt,
                                      tokens=self.toks, expert_slot=self.slot,
                                      num_experts=w.E_local, shared_w_gate_up=self.sgu,
                                      shared_w_down=self.sdn, activation=self.act,
                                      act_noise=True)
        got = out_gpu[: self.n].double().cpu().numpy()
        rms = math.sqrt(float(np.mean(ref * ref)))
        err = np.abs(got - ref)
        bits = 8 if w.dtype == torch.bfloat16 else 11
        a = np.abs(ref)
        hu = np.where(a > 0, np.exp2(np.floor(np.log2(np.where(a > 0, a, 1.0))) - bits), 0.0)
        au = a * (1 + 2.0 ** -7)
        hux = np.where(au > 0, np.exp2(np.floor(np.log2(np.where(au > 0, au, 1.0))) - bits), 0.0)
        sigma = noise / math.sqrt(3.0)
        z = (err - hux - 1e-3 * rms) / np.where(sigma > 0, sigma, np.inf)
        res = float(np.max(err - hu)) / rms
        if self.w4:
            note = (f"act in f16 (the NVFP4 path); the stated 1e-2 RMS + half an ulp is "
                    f"{'met' if res <= 1e-2 else 'not met'}")
        else:
            note = (f"act in {'bf16' if bits == 8 else 'f16'}; the stated 1e-2 RMS + half an ulp "
                    f"is {'met' if res <= 1e-2 else 'not met'} on this sample (a bf16 act "
                    f"intermediate cannot meet it on whole outputs)")
        return {"tokens": int(self.n), "max_err_over_rms": float(err.max()) / rms,
                "max_err_minus_half_ulp_over_rms": res,
                "max_err_in_act_rounding_sigmas": float(z.max()),
                "bound": "|gpu - oracle| <= half ulp of the output + 7 sigma of the act rounding "
                         "+ 1e-3 RMS; " + note}


# ------------------------------------------------------------------------------------ main arm
def run_ours(args, w, ws_n, rank, local):
    import numpy as np
    import torch

    from mixture_experts_forward_moe_gb300 import binding as B
    from mixture_experts_forward_moe_gb300 import inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    d = inputs.generate(w, seed=args.seed, device=dev)
    w4 = w.weights == "nvfp4"
    kw = dict(correction_bias=d["correction_bias"], **w.kwargs())
    if w4:  # the library's packed NVFP4 layout, made once when the weights are loaded
        d["w_gate_up_canonical"], d["w_down_canonical"] = d["w_gate_up"], d["w_down"]
        d["w_gate_up"] = B.pack_nvfp4_weights(*d["w_gate_up"])
        d["w_down"] = B.pack_nvfp4_weights(*d["w_down"])
    else:
        kw.update(shared_w_gate_up=d["shared_w_gate_up"], shared_w_down=d["shared_w_down"])
    fwd = B.fused_moe_fwd_w4a16 if w4 else B.fused_moe_fwd
    prob = B.make_problem(w.T, w.H, w.E, w.F, w.top_k, w.dtype, w.scoring_func, w.renormalize,
                          w.num_expert_group, w.topk_group, w.routed_scaling_factor, w.S,
                          w.activation, w.ep_local, w.ep_offset)
    # the W4A16 path also takes the gate/up GEMM's split-K scratch
    wsp = B.new_workspace(B.workspace_size_w4a16(prob) if w4 else B.workspace_size(prob), dev)
    out = torch.empty((w.T, w.H), dtype=w.dtype, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        fwd(d["hidden_states"], d["gating_output"], d["w_gate_up"], d["w_down"], out=out,
            workspace=wsp, **kw)

    ids, _ = B.moe_route(d["gating_output"], w.top_k, w.scoring_func, w.renormalize,
                         d["correction_bias"], w.num_expert_group, w.topk_group,
                         w.routed_scaling_factor)
    lids = torch.from_numpy(local_ids(w, ids.cpu().numpy()))
    n_unique = int(torch.unique(lids[lids >= 0]).numel())
    P_local = int((lids >= 0).sum())  # routes this GPU computes
    # Between steps: when the expert weights one step streams exceed twice the L2, nothing of a
    # step's weights survives into the next and no flush is needed; otherwise the L2 is flushed.
    weight_bytes = algorithmic_bytes(w, n_unique, P_local)["total"]
    if weight_bytes > 2 * L2_BYTES:
        flush = None
        l2_note = (f"no flush: each step streams {weight_bytes / 1e9:.2f} GB of expert weights, "
                   f"more than twice the {L2_BYTES >> 20} MiB L2")
    else:
        flush = L2Flush(dev)
        l2_note = L2Flush.note

    def do_flush():
        if flush is not None:
            flush()

    for _ in range(args.warmup):
        do_flush()
        step()
    torch.cuda.synchronize()
    st = B.get_device_status(wsp)
    if st != B.MOE_OK:
        raise RuntimeError(f"device status after warm-up: {B.status_string(st)}")

    dominant_candidates = ["gemm1", "gemm2"] + (["shared_gemm1", "shared_gemm2"] if w.S else [])

    def timed_loop(fn, profile_stages):
        """K steps of fn, each bracketed by an event pair on the launching stream; with
        profile_stages the library also records event pairs around those stages."""
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
        barrier()
        torch.cuda.synchronize()
        B.profile_enable(profile_stages)
        for i in range(args.steps):
            do_flush()
            starts[i].record(stream)
            fn()
            ends[i].record(stream)
        torch.cuda.synchronize()
        barrier()
        prof = B.profile_collect()
        B.profile_enable([])
        return [a.elapsed_time(b) for a, b in zip(starts, ends)], prof

    # One fused call captured into a CUDA graph (its kernels and their programmatic
    # dependencies): a replay costs the host one launch instead of one per kernel.
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()

    def replay():
        graph.replay()

    headline = replay if graph is not None else step
    # The headline loop records no events inside a step: an event between two kernels would
    # stop the next one from starting early (programmatic dependent launch).
    clocks = ClockSampler(local) if rank == 0 else None
    step_ms, _ = timed_loop(headline, [])
    clk = clocks.stop() if clocks else None
    total_ms = float(sum(step_ms))
    max_ms = max_over_ranks(total_ms)
    # The same K steps launched eagerly (one host launch per kernel), for comparison and for the
    # launch count.
    eager_ms, prof_clean = timed_loop(step, [])
    # The roofline loop: the same K steps with event pairs around the GEMM stages (eager).
    prof_step_ms, prof = timed_loop(step, dominant_candidates)
    st = B.get_device_status(wsp)
    if st != B.MOE_OK:
        raise RuntimeError(f"device status after timed steps: {B.status_string(st)}")

    flops = w.flops(P_local)
    value = job_throughput(flops, ws_n, args.steps, max_ms) / 1e12
    ms_per_step = max_ms / args.steps
    ab = algorithmic_bytes(w, n_unique, P_local)
    hbm_gbs, bf16_peak, bf16_sust, peak_src = measured_peaks()
    launches = sum(v[2] for v in prof_clean.values())

    # Dominant kernel: the instrumented stage with the largest summed device time.
    dom = max(dominant_candidates, key=lambda s: prof[s][0])
    dom_ms, dom_calls, _ = prof[dom]
    dom_avg = dom_ms / max(dom_calls, 1)
    achieved = ab[dom] / (dom_avg * 1e-3) / 1e9
    traffic = recorded_traffic(w.name, dom)
    hbm = {"bound": "hbm", "kernel": f"moe_gemm_kernel ({dom})", "achieved": achieved,
           "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
           "traffic": traffic, "algorithmic_bytes": ab[dom], "avg_launch_ms": dom_avg,
           "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
           if peak_src == "measured" else "fallback 6.8 TB/s",
           "timing": "event pair around each launch of the kernel over a second loop of "
                     "the same K steps"}
    dom_flops = stage_flops(w, P_local)[dom]
    tensor = {"achieved_tflops": dom_flops / (dom_avg * 1e-3) / 1e12,
              "peak_tflops": bf16_sust, "peak_source": f"{peak_src} bf16_tflops_sustained"}
    tensor["frac"] = tensor["achieved_tflops"] / bf16_sust
    # The bound is whichever resource the kernel's algorithmic work needs longer on.
    if dom_flops / (bf16_sust * 1e12) > ab[dom] / (hbm_gbs * 1e9):
        roofline = {"bound": "tensor", "kernel": hbm["kernel"],
                    "achieved": tensor["achieved_tflops"], "peak": bf16_sust,
                    "unit": "TFLOP/s", "frac": tensor["frac"], "traffic": traffic,
                    "algorithmic_flops": dom_flops, "avg_launch_ms": dom_avg,
                    "peak_source": tensor["peak_source"], "timing": hbm["timing"], "hbm": hbm}
    else:
        roofline = hbm
        roofline["tensor"] = tensor
    stages = {k: {"avg_ms": v[0] / v[1], "calls": v[1]} for k, v in prof.items() if v[1]}

    res = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": ws_n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak",
        # the NVFP4 path's GEMMs take f16 tokens and decoded f16 weights (bf16 in and out)
        "vs_baseline": None,
        "dtype": "f16" if w.weights == "nvfp4" or w.dtype != torch.bfloat16 else "bf16",
        "data": "synthetic: seeded N(0,1) hidden states and router logits, N(0,1/fan_in) "
                "weights" + (", N(0, 0.1^2) correction bias" if w.bias_std else ""),
        "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "F": w.F,
                   "top_k": w.top_k, "S": w.S, "scoring": w.scoring_func,
                   "num_expert_group": w.num_expert_group, "topk_group": w.topk_group,
                   "routed_scaling_factor": w.routed_scaling_factor,
                   "activation": w.activation, "skew_alpha": w.skew_alpha,
                   "weights": w.weights, "ep_local_experts": w.ep_local,
                   "routes_computed": P_local,
                   "global_batch": w.T * ws_n, "parallelism": f"replicas x{ws_n}",
                   "l2": l2_note,
                   "timing": ("one CUDA-graph replay of the fused call per step"
                              if graph is not None else "eager launches")
                             + "; CUDA event pair per step on the launching stream; sum of K"},
        "eager_ms_per_step": statistics.mean(eager_ms),
        "roofline_loop_ms_per_step": statistics.mean(prof_step_ms),
        "ms_median": statistics.median(step_ms), "hbm_gbs": ab["total"] / (ms_per_step * 1e-3) / 1e9,
        "hbm_frac": ab["total"] / (ms_per_step * 1e-3) / 1e9 / hbm_gbs,
        "unique_experts": n_unique, "roofline": roofline, "gpu_launches": launches,
        "launches_per_step": launches / args.steps, "stages": stages, "clocks": clk,
    }
    if w.name in PUBLISHED_MS:
        res["context_published_ms"] = {"ms": PUBLISHED_MS[w.name],
                                       "where": "flashinfer PR #4048, B300, another routing seed"}
    pub = PUBLISHED_TFLOPS.get((w.name, res["dtype"]))
    if pub:
        res["vs_baseline"] = value / pub

    # End to end through the public API from pinned host buffers: each step is one library call
    # (fused_moe_fwd_host) that enqueues the host->device copies of the step's inputs, the fused
    # path and the device->host copy of the output.
    if not args.no_e2e:
        h_hidden = d["hidden_states"].cpu().pin_memory()
        h_gating = d["gating_output"].cpu().pin_memory()
        h_out = torch.empty((w.T, w.H), dtype=w.dtype, pin_memory=True)
        wsh = B.new_workspace(B.host_workspace_size(prob, w4), dev)
        n_e2e = max(1, min(args.steps, 200))

        def host_step():
            B.fused_moe_fwd_host(h_hidden, h_gating, d["w_gate_up"], d["w_down"], out_host=h_out,
                                 workspace=wsh, **kw)

        for _ in range(3):
            host_step()
        torch.cuda.synchronize()
        es = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_e2e)]
        barrier()
        torch.cuda.synchronize()
        for i in range(n_e2e):
            do_flush()
            es[2 * i].record(stream)
            host_step()
            es[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        barrier()
        e2e_ms = max_over_ranks(sum(es[2 * i].elapsed_time(es[2 * i + 1]) for i in range(n_e2e)))
        if not torch.equal(h_out, out.cpu()):
            raise RuntimeError("the host-buffer call's output differs from the device call's")
        del wsh
        res["e2e"] = {"value": job_throughput(flops, ws_n, n_e2e, e2e_ms) / 1e12,
                      "unit": "TFLOP/s", "steps": n_e2e,
                      "h2d_bytes_per_step": h_hidden.numel() * h_hidden.element_size()
                      + h_gating.numel() * 4,
                      "d2h_bytes_per_step": h_out.numel() * h_out.element_size(),
                      "ms_per_step": e2e_ms / n_e2e,
                      "call": "fused_moe_fwd_host" + ("" if not w4 else " (w4a16)")
                              + ": one C-ABI call per step from page-locked host buffers, "
                                "eager launches"}

    if rank == 0 and ws_n == 1 and not args.no_cpu_baseline:
        sample = OracleSample(w, d, args.cpu_budget)
        el, passes = sample.run(args.cpu_budget)
        rate, n, cores = sample.flops(passes) / el / 1e12, sample.n, sample.cores
        res["cpu_baseline"] = {"value": rate, "unit": "TFLOP/s", "cores": cores,
                               "kind": "oracle",
                               "sample": f"{n} of {w.T} tokens (routing + expert MLP, fp64), "
                                         f"{passes} passes in {el:.1f} s"}
        # the timed output of the last step against the oracle on the same tokens
        res["parity_sample"] = sample.parity(out)
    return res


def run_reference(args, w):
    """The CPU oracle as a bench arm: each step is one oracle pass over a bounded token sample."""
    import torch

    from mixture_experts_forward_moe_gb300 import inputs
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    d = inputs.generate(w, seed=args.seed, device=dev)
    # About two minutes of oracle work over all warm-up and timed steps, whatever K and W are.
    per_step = max(0.01, min(10.0, 120.0 / max(1, args.steps + args.warmup)))
    sample = OracleSample(w, d, per_step)
    for _ in range(args.warmup):
        sample.run(per_step)
    times, flops = [], 0.0
    for _ in range(args.steps):
        el, passes = sample.run(per_step)
        times.append(el)
        flops += sample.flops(passes)
    n_last, cores = sample.n, sample.cores
    total = sum(times)
    value = flops / total / 1e12
    res = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": 1,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": total / args.steps * 1e3,
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f64", "data": "synthetic (same seeded inputs as the GPU arm)",
           "config": {"workload": w.name, "T": w.T, "H": w.H, "E": w.E, "F": w.F,
                      "top_k": w.top_k, "S": w.S},
           "impl": "reference",
           "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                            "sample": f"{n_last} of {w.T} tokens per pass, ~{per_step:.1f} s "
                                      f"per step"},
           "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    return res


# ----------------------------------------------------------- grouped GEMM (masked layout) arm
PUBLISHED_GROUPED_MS = {  # TileOPs MoE page, MoEGroupedGemmFwd / MoEGroupedGemmFP8Fwd (hardware
    "ds-v3-ep8-masked": 0.4851,  # not stated)
    "ds-v3-e8-up-masked": 0.0743, "ds-v3-e8-down-masked": 0.0424, "ds-v3-dec-b64-up": 0.2266,
    "ds-v3-dec-b64-down": 0.1157, "ds-v3-dec-b256-up": 0.2420, "ds-v3-dec-b256-down": 0.1309,
    "qwen3-235b-dec-b64-up": 0.0598, "qwen3-235b-dec-b64-down": 0.0351,
    "qwen3-235b-dec-b256-up": 0.0605, "qwen3-235b-dec-b256-down": 0.0358,
    "kimi-k2-dec-b64-up": 0.2638, "kimi-k2-dec-b64-down": 0.1430, "kimi-k2-dec-b256-up": 0.3545,
    "kimi-k2-dec-b256-down": 0.1892,
}


def run_grouped_gemm(args, w, ws_n, rank, local):
    """moe_grouped_gemm on a masked-layout workload: K timed calls (a CUDA-graph replay each),
    inputs resident in HBM; the same contract as the fused line."""
    import numpy as np
    import torch

    import oracle
    from mixture_experts_forward_moe_gb300 import binding as B
    from mixture_experts_forward_moe_gb300 import inputs

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    fp8 = isinstance(w, inputs.Fp8GemmWorkload)
    d = (inputs.generate_fp8_gemm if fp8 else inputs.generate_grouped_gemm)(w, seed=args.seed,
                                                                           device=dev)
    a, b, meta = d["a"], d["b"], d["meta"]
    out = torch.zeros((w.E, w.max_m, w.N), dtype=torch.bfloat16, device=dev)
    g = B.GroupedGemm(w.E, w.N, w.K, w.max_m, 0, B.MOE_BF16, 0, 0)
    wsp = B.new_workspace(B.lib().moe_grouped_gemm_workspace_size(B.ctypes.byref(g)), dev)
    stream = torch.cuda.current_stream()
    valid = int(meta.sum())
    # groups with at least one valid row: the only weights the op has to read
    active = int((meta > 0).sum())

    def step():
        if fp8:
            B.moe_grouped_gemm_fp8(a, d["a_scale"], b, d["b_scale"], meta, out=out,
                                   workspace=wsp)
        else:
            B.moe_grouped_gemm(a, b, meta, out=out, workspace=wsp)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    graph = None
    if not args.eager:
        cap = torch.cuda.Stream()
        cap.wait_stream(stream)
        with torch.cuda.stream(cap):
            step()
        stream.wait_stream(cap)
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
    run = graph.replay if graph is not None else step
    # Between steps: a call that streams more than twice the L2 in weights leaves nothing of
    # them for the next one; a smaller one gets the L2 flushed by a write outside its events.
    eb = 1 if fp8 else 2  # bytes per element of a and b
    weight_bytes = active * w.N * w.K * eb
    flush = L2Flush(dev) if weight_bytes <= 2 * L2_BYTES else None
    l2_note = (f"no flush: each call streams {weight_bytes / 1e9:.2f} GB of weights, more than "
               f"twice the {L2_BYTES >> 20} MiB L2" if flush is None else
               f"each call streams {weight_bytes / 1e9:.2f} GB of weights; " + L2Flush.note)
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    clocks = ClockSampler(local) if rank == 0 else None
    barrier()
    torch.cuda.synchronize()
    for i in range(args.steps):
        if flush is not None:
            flush()
        starts[i].record(stream)
        run()
        ends[i].record(stream)
    torch.cuda.synchronize()
    barrier()
    clk = clocks.stop() if clocks else None
    step_ms = [x.elapsed_time(y) for x, y in zip(starts, ends)]
    max_ms = max_over_ranks(float(sum(step_ms)))
    ms = max_ms / args.steps
    st = B.get_device_status(wsp)
    if st != B.MOE_OK:
        raise RuntimeError(f"device status: {B.status_string(st)}")
    flops = w.flops(valid)
    value = job_throughput(flops, ws_n, args.steps, max_ms) / 1e12
    hbm_gbs, bf16_peak, bf16_sust, peak_src = measured_peaks()
    # the weights (+ their block scales) of the groups that have rows, + the valid rows in (+ their
    # scales) and out (bf16); an empty group's weights are never read
    ab = (active * w.N * w.K * eb + valid * w.K * eb + valid * w.N * 2 +
          ((active * (w.N // 128) * (w.K // 128) + valid * (w.K // 128)) * 4 if fp8 else 0))
    achieved = ab / (ms * 1e-3) / 1e9
    # FP8 tensor peak: the measured bf16 peak times the nominal fp8/bf16 ratio (4.5 / 2.25)
    tpeak = bf16_sust * (2.0 if fp8 else 1.0)
    roofline = {"bound": "hbm", "kernel": ("moe_gemm_fp8_kernel" if fp8 else "moe_gemm_kernel")
                + " (grouped, masked layout)",
                "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s", "frac": achieved / hbm_gbs,
                "traffic": None, "algorithmic_bytes": ab, "avg_launch_ms": ms,
                "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)",
                "timing": "event pair around each call (one graph replay: tile list + GEMM)",
                "tensor": {"achieved_tflops": flops / (ms * 1e-3) / 1e12,
                           "peak_tflops": tpeak,
                           "peak_source": "bf16_tflops_sustained" + (" x 2 (fp8 nominal ratio)"
                                                                    if fp8 else ""),
                           "frac": flops / (ms * 1e-3) / 1e12 / tpeak}}
    if flops / (tpeak * 1e12) > ab / (hbm_gbs * 1e9):  # tensor-bound by the algorithmic work
        hbm_part = dict(roofline)
        roofline = {"bound": "tensor", "kernel": hbm_part["kernel"],
                    "achieved": flops / (ms * 1e-3) / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                    "frac": flops / (ms * 1e-3) / 1e12 / tpeak, "traffic": None,
                    "algorithmic_flops": flops, "avg_launch_ms": ms, "hbm": hbm_part}
    res = {
        "metric": ("moe_grouped_gemm_fp8" if fp8 else "moe_grouped_gemm")
                  + " device ms, TFLOP/s & HBM GB/s (masked layout)",
        "value": value, "unit": "TFLOP/s", "n_gpus": ws_n, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "e4m3" if fp8 else "bf16",
        "data": ("synthetic: N(0,1) a and N(0,1/K) b quantised to E4M3 with block scales, "
                 f"{w.total} valid rows spread uniformly over the groups" if fp8 else
                 "synthetic: N(0,1) a, N(0,1/K) b, valid rows per group uniform in "
                 f"[{w.m_lo}, {w.m_hi}]"),
        "config": {"workload": w.name, "E": w.E, "max_m": w.max_m, "K": w.K, "N": w.N,
                   "weights": "e4m3 with 128x128 f32 block scales" if fp8 else "bf16",
                   "valid_rows": valid, "active_groups": active, "global_batch": valid * ws_n,
                   "parallelism": f"replicas x{ws_n}",
                   "l2": l2_note,
                   "timing": "one CUDA-graph replay per step; CUDA event pair per step"},
        "roofline": roofline, "gpu_launches": 2 * args.steps, "clocks": clk,
        "context_published_ms": {"ms": PUBLISHED_GROUPED_MS.get(w.name),
                                 "where": "TileOPs MoE page, MoEGroupedGemmFwd (hardware not "
                                          "stated)"},
    }
    if not args.no_e2e and not fp8:
        h_a = a.cpu().pin_memory()
        h_meta = meta.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        a_dev, meta_dev = torch.empty_like(a), torch.empty_like(meta)
        n_e2e = max(1, min(args.steps, 50))
        es = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_e2e)]
        torch.cuda.synchronize()
        for i in range(n_e2e):
            es[2 * i].record(stream)
            a_dev.copy_(h_a, non_blocking=True)
            meta_dev.copy_(h_meta, non_blocking=True)
            B.moe_grouped_gemm(a_dev, b, meta_dev, out=out, workspace=wsp)
            h_out.copy_(out, non_blocking=True)
            es[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = statistics.mean(es[2 * i].elapsed_time(es[2 * i + 1]) for i in range(n_e2e))
        res["e2e"] = {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "h2d_bytes_per_step": h_a.numel() * 2 + h_meta.numel() * 4,
                      "d2h_bytes_per_step": h_out.numel() * 2, "ms_per_step": e2e_ms}
    if not args.no_e2e and fp8:
        h_a = a.cpu().pin_memory()
        h_sa = d["a_scale"].cpu().pin_memory()
        h_meta = meta.cpu().pin_memory()
        h_out = torch.empty(out.shape, dtype=out.dtype, pin_memory=True)
        a_dev, sa_dev, meta_dev = torch.empty_like(a), torch.empty_like(d["a_scale"]), \
            torch.empty_like(meta)
        n_e2e = max(1, min(args.steps, 50))
        es = [torch.cuda.Event(enable_timing=True) for _ in range(2 * n_e2e)]
        torch.cuda.synchronize()
        for i in range(n_e2e):
            es[2 * i].record(stream)
            a_dev.copy_(h_a, non_blocking=True)
            sa_dev.copy_(h_sa, non_blocking=True)
            meta_dev.copy_(h_meta, non_blocking=True)
            B.moe_grouped_gemm_fp8(a_dev, sa_dev, b, d["b_scale"], meta_dev, out=out,
                                   workspace=wsp)
            h_out.copy_(out, non_blocking=True)
            es[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        e2e_ms = statistics.mean(es[2 * i].elapsed_time(es[2 * i + 1]) for i in range(n_e2e))
        res["e2e"] = {"value": flops / (e2e_ms * 1e-3) / 1e12, "unit": "TFLOP/s",
                      "h2d_bytes_per_step": h_a.numel() + h_sa.numel() * 4 + h_meta.numel() * 4,
                      "d2h_bytes_per_step": h_out.numel() * 2, "ms_per_step": e2e_ms}
    if not args.no_cpu_baseline and rank == 0 and fp8:
        rows = np.arange(w.E) * w.max_m
        idx = torch.from_numpy(rows).to(dev)
        a_s = a.reshape(w.E * w.max_m, w.K)[idx].cpu()
        sa_s = d["a_scale"].reshape(w.E * w.max_m, w.K // 128)[idx].cpu()
        b_c, bs_c = b.cpu(), d["b_scale"].cpu()
        t0, passes = time.perf_counter(), 0
        while time.perf_counter() - t0 < args.cpu_budget and passes < 1000:
            for e in range(w.E):
                oracle.grouped_gemm_fp8(a_s[e:e + 1], sa_s[e:e + 1], b_c[e:e + 1],
                                        bs_c[e:e + 1], np.array([1], np.int32))
            passes += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": w.flops(w.E) * passes / el / 1e12, "unit": "TFLOP/s",
                               "cores": oracle.num_threads(), "kind": "oracle",
                               "sample": f"1 row per group ({w.E} rows) per pass, {passes} "
                                         f"passes in {el:.1f} s"}
    if not args.no_cpu_baseline and rank == 0 and not fp8:
        # the oracle on one sampled row per group, timed for about cpu_budget seconds
        rows = np.arange(w.E) * w.max_m
        a_s = a.reshape(w.E * w.max_m, w.K)[torch.from_numpy(rows).to(dev)].cpu()
        b_c = b.cpu()
        t0, passes = time.perf_counter(), 0
        while time.perf_counter() - t0 < args.cpu_budget and passes < 1000:
            for e in range(w.E):
                oracle.grouped_gemm(a_s[e:e + 1].reshape(1, 1, w.K), b_c[e:e + 1],
                                    np.array([1], np.int32), oracle.BF16, max_m=1)
            passes += 1
        el = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": w.flops(w.E) * passes / el / 1e12, "unit": "TFLOP/s",
                               "cores": oracle.num_threads(), "kind": "oracle",
                               "sample": f"1 valid row per group ({w.E} rows) per pass, "
                                         f"{passes} passes in {el:.1f} s"}
    return res


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--dtype", default="bf16", choices=["bf16", "f16"])
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of a CUDA-graph replay of the fused call")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    import torch

    from mixture_experts_forward_moe_gb300 import inputs
    if args.workload in inputs.GROUPED_GEMM_WORKLOADS or \
            args.workload in inputs.FP8_GEMM_WORKLOADS:
        gw = inputs.GROUPED_GEMM_WORKLOADS.get(args.workload) or \
            inputs.FP8_GEMM_WORKLOADS[args.workload]
        ws_n, rank, local = dist_env()
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable": "the oracle arm covers the "
                                  "fused workloads; the grouped GEMM line carries its own "
                                  "cpu_baseline"}), flush=True)
            return 0
        if ws_n > 1:
            import torch.distributed as dist
            torch.cuda.set_device(local)
            dist.init_process_group("nccl")
        try:
            res = run_grouped_gemm(args, gw, ws_n, rank, local)
        finally:
            if ws_n > 1:
                import torch.distributed as dist
                dist.destroy_process_group()
        if rank == 0:
            print(json.dumps(res), flush=True)
        return 0
    w = inputs.workload(args.workload)
    if args.dtype == "f16":
        w = w.with_(dtype=torch.float16)
    ws_n, rank, local = dist_env()

    if args.impl == "reference":
        if rank != 0:
            return 0
        res = run_reference(args, w)
        print(json.dumps(res), flush=True)
        return 0

    if ws_n > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    try:
        res = run_ours(args, w, ws_n, rank, local)
    finally:
        if ws_n > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
    if rank == 0:
        print(json.dumps(res), flush=True)
    return 0


if __name__ == "__main__":
    sys.exit(main())
