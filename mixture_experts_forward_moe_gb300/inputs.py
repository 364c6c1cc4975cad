"""Seeded synthetic inputs for the fused MoE forward pass.

This module holds the workload recipes and the random generators only: it computes nothing
of the method.  Both the CUDA path and the CPU oracle are fed copies of the same tensors.

Recipe (the pages' workloads; TileOPs benchmark page "MoE" section, FusedMoEFwd and
FusedMoESharedExpertFwd shape lists; flashinfer PR #4048 DeepSeek-V3 benchmark workload):
  hidden_states  ~ N(0, 1)                      rounded to bf16/f16 (round to nearest even)
  gating_output  ~ N(0, 1) in f32
  correction_bias ~ N(0, 0.1^2) in f32          (sigmoid workloads)
  w_gate_up      ~ N(0, 1/H)  (std 1/sqrt(fan_in), fan_in = H)
  w_down         ~ N(0, 1/F)  (fan_in = F)
  shared_w_gate_up ~ N(0, 1/H), shared_w_down ~ N(0, 1/S)
One torch.Generator seeded with `seed` draws, in this order: hidden, gating, bias, w_gate_up,
w_down, shared_w_gate_up, shared_w_down.  Large weights are drawn expert by expert (chunks of
rows) so the f32 staging stays small; the chunking is part of the recipe.  w_gate_up has 2F
rows per expert for the gated activations (SiLU, GeGLU-tanh) and F rows for ReLU2.

NVFP4 experts (flashinfer PR #4048, W4A16): the same N(0, 1/fan_in) draws, quantised per expert
matrix W [rows, K]: alpha = max|W| / (6 * 448); per block of 16 consecutive k, the E4M3 scale is
min(448, max|block| / 6 / alpha) rounded to nearest even by torch's float8_e4m3fn conversion;
each code is the E2M1 value nearest to w / (scale * alpha) (ties toward zero, |v| > 6 clamps to
6), two codes per byte with element 2i in the low nibble.  A block whose scale rounds to zero
gets zero codes.

Expert-parallel shard (the same PR's DeepSeek-V3 EP8 benchmark, 32 local of 256 experts): the
router scores all E experts; only the weights of the ep_local local experts are drawn.

Skewed routing (flashinfer PR #4048 benchmark, "Skewed routing"): when skew_alpha > 0 the
gating logits of expert e get the fixed bias -skew_alpha * log(1 + rank[e]), rank a random
permutation of the experts drawn by a second generator seeded with seed + 7919 (so the other
inputs are the same as without skew).  skew_alpha is chosen per workload so that the most
popular expert receives about twice the mean load.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int
    H: int
    E: int
    F: int
    top_k: int
    scoring_func: str = "softmax"
    renormalize: bool = True
    bias_std: float = 0.0          # 0: no correction_bias
    num_expert_group: int = 0
    topk_group: int = 0
    routed_scaling_factor: float = 1.0
    S: int = 0
    dtype: torch.dtype = torch.bfloat16
    activation: str = "silu"       # "silu", "gelu_tanh" (gated) or "relu2" (single projection)
    skew_alpha: float = 0.0         # > 0: skewed routing bias on the gating logits
    weights: str = "bf16"           # "bf16" (the dtype) or "nvfp4" (W4A16 experts)
    ep_local: int = 0               # > 0: experts held by this GPU (shard [ep_offset, +ep_local))
    ep_offset: int = 0

    @property
    def E_local(self) -> int:
        return self.ep_local if self.ep_local > 0 else self.E

    @property
    def gated(self) -> bool:
        return self.activation != "relu2"

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)

    def flops(self, routes=None) -> float:
        """2*T*k*3*F*H (+ 2*T*3*S*H): the FLOP count the TileOPs MoE page's TFLOP/s uses (three
        F x H matrices per expert; two for the single-projection ReLU2 MLP).  `routes` replaces
        T*k when only some routes are computed (the local experts of a shard)."""
        m = 3 if self.gated else 2
        P = self.T * self.top_k if routes is None else routes
        return 2.0 * P * m * self.F * self.H + 2.0 * self.T * m * self.S * self.H

    def kwargs(self) -> dict:
        return dict(top_k=self.top_k, scoring_func=self.scoring_func,
                    renormalize=self.renormalize, num_expert_group=self.num_expert_group,
                    topk_group=self.topk_group,
                    routed_scaling_factor=self.routed_scaling_factor,
                    activation=self.activation, ep_local_offset=self.ep_offset)


# The five workloads this project is measured on (sizes from the pages' shape lists).
WORKLOADS = {
    "tiny-softmax": Workload("tiny-softmax", T=4, H=128, E=8, F=64, top_k=2),
    "qwen3-30b-a3b-decode-t32": Workload("qwen3-30b-a3b-decode-t32", T=32, H=2048, E=128,
                                         F=768, top_k=8),
    "qwen3-235b-a22b-decode-t512": Workload("qwen3-235b-a22b-decode-t512", T=512, H=4096,
                                            E=128, F=1536, top_k=8),
    "deepseek-v3-grouped-prefill-t4096": Workload(
        "deepseek-v3-grouped-prefill-t4096", T=4096, H=7168, E=256, F=2048, top_k=8,
        scoring_func="sigmoid", bias_std=0.1, num_expert_group=8, topk_group=4,
        routed_scaling_factor=2.5),
    "kimi-k2-shared-t512": Workload(
        "kimi-k2-shared-t512", T=512, H=7168, E=384, F=2048, top_k=8, scoring_func="sigmoid",
        bias_std=0.1, routed_scaling_factor=2.827, S=18432),
}

# Variants of the measured shapes (flashinfer PR #4048: skewed routing; activation variants of
# the W4A16 follow-up and the W4A8 validation list).  With N(0,1) softmax logits over 128
# experts and top-8, skew_alpha = 0.10 gives the most popular expert 2.0x the mean load.
_Q235 = WORKLOADS["qwen3-235b-a22b-decode-t512"]
# flashinfer PR #4048's W4A16 benchmark: one DeepSeek-V3 EP8 rank (32 of the 256 experts,
# top-8, 8 groups keep 4, rsf 2.5, correction-bias scale 0.01) at 32, 512 and 4096 tokens.
_DSV3_EP8 = Workload("deepseek-v3-ep8-shard", T=32, H=7168, E=256, F=2048, top_k=8,
                     scoring_func="sigmoid", bias_std=0.01, num_expert_group=8, topk_group=4,
                     routed_scaling_factor=2.5, ep_local=32)
VARIANTS = {
    "qwen3-235b-a22b-decode-t512-skewed": _Q235.with_(
        name="qwen3-235b-a22b-decode-t512-skewed", skew_alpha=0.10),
    "qwen3-235b-a22b-decode-t512-gelu-tanh": _Q235.with_(
        name="qwen3-235b-a22b-decode-t512-gelu-tanh", activation="gelu_tanh"),
    "qwen3-235b-a22b-decode-t512-relu2": _Q235.with_(
        name="qwen3-235b-a22b-decode-t512-relu2", activation="relu2"),
    "qwen3-30b-a3b-decode-t32-w4a16": WORKLOADS["qwen3-30b-a3b-decode-t32"].with_(
        name="qwen3-30b-a3b-decode-t32-w4a16", weights="nvfp4"),
}
for _t in (32, 512, 4096):
    for _wf in ("bf16", "nvfp4"):
        _n = f"deepseek-v3-ep8-shard-t{_t}" + ("-w4a16" if _wf == "nvfp4" else "")
        VARIANTS[_n] = _DSV3_EP8.with_(name=_n, T=_t, weights=_wf)

# Small cases of the same kernels for hardware-counter captures, which must stay at a few GB on
# the device: the DeepSeek-V3 expert shapes and routing with 32 experts (about 128 routed rows
# per expert, skewed by the correction bias), 2.8 GB of weights.
PROBES = {
    "prefill-probe-e32-t512": Workload(
        "prefill-probe-e32-t512", T=512, H=7168, E=32, F=2048, top_k=8, scoring_func="sigmoid",
        bias_std=0.1, num_expert_group=8, topk_group=4, routed_scaling_factor=2.5),
    # about 256 rows per expert: several token tiles per expert, as in the T=4096 prefill
    "prefill-probe-e32-t1024": Workload(
        "prefill-probe-e32-t1024", T=1024, H=7168, E=32, F=2048, top_k=8,
        scoring_func="sigmoid", bias_std=0.1, num_expert_group=8, topk_group=4,
        routed_scaling_factor=2.5),
}


def workload(name: str) -> Workload:
    for table in (WORKLOADS, VARIANTS, PROBES):
        if name in table:
            return table[name]
    raise KeyError(name)

_CHUNK_ELEMS = 1 << 28  # f32 staging per draw: 1 GiB


def _randn(shape, gen, device, std, dtype):
    """N(0, std^2) drawn in f32 chunks along dim 0, rounded to `dtype`."""
    out = torch.empty(shape, dtype=dtype, device=device)
    if out.numel() == 0:
        return out
    per_row = out[0].numel() if out.dim() > 1 else 1
    rows = max(1, _CHUNK_ELEMS // max(per_row, 1))
    flat = out.view(shape[0], -1) if out.dim() > 1 else out.view(-1, 1)
    for r0 in range(0, shape[0], rows):
        r1 = min(shape[0], r0 + rows)
        x = torch.randn((r1 - r0, flat.shape[1]), generator=gen, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        flat[r0:r1].copy_(x.to(dtype))
        del x
    return out


_E2M1_MIDPOINTS = (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0)  # between 0,.5,1,1.5,2,3,4,6


def quantize_nvfp4(w: torch.Tensor):
    """One f32 matrix [rows, K] -> (codes u8 [rows, K/2], scales u8 [rows, K/16], alpha f32)."""
    rows, K = w.shape
    amax = float(w.abs().max()) if w.numel() else 0.0
    alpha = amax / (6.0 * 448.0) if amax > 0 else 1.0
    alpha = float(torch.tensor(alpha, dtype=torch.float32))
    blocks = w.view(rows, K // 16, 16)
    bmax = blocks.abs().amax(-1)
    sf = (bmax / 6.0 / alpha).clamp_(max=448.0).to(torch.float8_e4m3fn)
    scale = sf.to(torch.float32) * alpha
    v = torch.where(scale[..., None] > 0, blocks / scale[..., None].clamp(min=1e-38),
                    torch.zeros((), device=w.device))
    mids = torch.tensor(_E2M1_MIDPOINTS, dtype=torch.float32, device=w.device)
    code = torch.bucketize(v.abs(), mids, right=False).to(torch.uint8)
    code |= (v < 0).to(torch.uint8) << 3
    code = code.view(rows, K)
    q = code[:, 0::2] | (code[:, 1::2] << 4)
    return q.contiguous(), sf.view(torch.uint8).contiguous(), alpha


def _randn_nvfp4(shape, gen, device, std):
    """N(0, std^2) expert matrices [E, rows, K] drawn as in _randn (f32, chunks of rows per
    expert), each quantised to NVFP4: returns (codes, scales, alpha [E])."""
    E, rows, K = shape
    q = torch.empty((E, rows, K // 2), dtype=torch.uint8, device=device)
    sf = torch.empty((E, rows, K // 16), dtype=torch.uint8, device=device)
    alpha = torch.empty((E,), dtype=torch.float32, device=device)
    for e in range(E):
        x = _randn((rows, K), gen, device, std, torch.float32)
        q[e], sf[e], alpha[e] = quantize_nvfp4(x)
        del x
    return q, sf, alpha


def generate(w: Workload, seed: int = 0, device="cuda") -> dict:
    """All inputs of workload `w` as tensors on `device` (the recipe in the module doc)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    dt = w.dtype
    d = {}
    d["hidden_states"] = _randn((w.T, w.H), gen, device, 1.0, dt)
    d["gating_output"] = _randn((w.T, w.E), gen, device, 1.0, torch.float32)
    if w.skew_alpha > 0:
        d["gating_output"] += skew_bias(w.E, w.skew_alpha, seed).to(device)
    d["correction_bias"] = (_randn((w.E,), gen, device, w.bias_std, torch.float32)
                            if w.bias_std > 0 else None)
    rows = 2 if w.gated else 1
    El = w.E_local
    if w.weights == "nvfp4":
        d["w_gate_up"] = _randn_nvfp4((El, rows * w.F, w.H), gen, device, 1.0 / math.sqrt(w.H))
        d["w_down"] = _randn_nvfp4((El, w.H, w.F), gen, device, 1.0 / math.sqrt(w.F))
    else:
        d["w_gate_up"] = _randn((El, rows * w.F, w.H), gen, device, 1.0 / math.sqrt(w.H), dt)
        d["w_down"] = _randn((El, w.H, w.F), gen, device, 1.0 / math.sqrt(w.F), dt)
    if w.S > 0:
        d["shared_w_gate_up"] = _randn((rows * w.S, w.H), gen, device, 1.0 / math.sqrt(w.H),
                                       dt)
        d["shared_w_down"] = _randn((w.H, w.S), gen, device, 1.0 / math.sqrt(w.S), dt)
    else:
        d["shared_w_gate_up"] = None
        d["shared_w_down"] = None
    return d


def skew_bias(E: int, alpha: float, seed: int) -> torch.Tensor:
    """[E] f32: -alpha * log(1 + rank[e]) for a seeded random ranking of the experts."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 7919)
    rank = torch.randperm(E, generator=g).to(torch.float64)
    return (-alpha * torch.log1p(rank)).to(torch.float32)


def random_ids(T: int, top_k: int, E: int, seed: int = 0, device="cpu", pad_frac: float = 0.0,
               distinct: bool = True) -> torch.Tensor:
    """Seeded topk_ids [T, top_k] int32 for the staged sort/GEMM tests: distinct experts per
    token (unless distinct=False), a fraction pad_frac of routes set to -1 (padding)."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    if distinct:
        ids = torch.stack([torch.randperm(E, generator=gen)[:top_k] for _ in range(T)]) \
            if T > 0 else torch.empty((0, top_k), dtype=torch.int64)
    else:
        ids = torch.randint(0, E, (T, top_k), generator=gen)
    if pad_frac > 0 and T > 0:
        mask = torch.rand((T, top_k), generator=gen) < pad_frac
        ids = ids.masked_fill(mask, -1)
    return ids.to(torch.int32).to(device)


def random_rows(n: int, cols: int, seed: int, dtype=torch.bfloat16, device="cpu",
                std: float = 1.0) -> torch.Tensor:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return (torch.randn((n, cols), generator=gen) * std).to(dtype).to(device)


def random_weights(n: int, seed: int, device="cpu") -> torch.Tensor:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    return torch.rand((n,), generator=gen, dtype=torch.float32).to(device)


# --------------------------------------------------------------------------- grouped GEMM
@dataclasses.dataclass(frozen=True)
class GroupedGemmWorkload:
    """A masked-layout grouped GEMM (TileOPs MoE page, op MoEGroupedGemmFwd): a [E, max_m, K],
    b [E, N, K], and the valid rows of each group drawn uniformly in [m_lo, m_hi]."""
    name: str
    E: int
    max_m: int
    K: int
    N: int
    m_lo: int
    m_hi: int
    dtype: torch.dtype = torch.bfloat16

    def flops(self, valid_rows: int) -> float:
        return 2.0 * valid_rows * self.N * self.K


# The page's "ds-v3-ep8-masked" workload: 32 local experts, up to 128 rows each, the DeepSeek-V3
# gate/up weights [4096, 7168].  Its printed 372 TFLOP/s at 0.4851 ms implies 96 valid rows per
# group on average, the mean of the uniform draw in [64, 128] used here.
GROUPED_GEMM_WORKLOADS = {
    "ds-v3-ep8-masked": GroupedGemmWorkload("ds-v3-ep8-masked", E=32, max_m=128, K=7168,
                                            N=4096, m_lo=64, m_hi=128),
}


def generate_grouped_gemm(w: GroupedGemmWorkload, seed: int = 0, device="cuda") -> dict:
    """a ~ N(0, 1), b ~ N(0, 1/K) (one generator seeded with `seed`, in that order) and the
    valid-row counts (a CPU generator seeded with seed + 1)."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    a = _randn((w.E, w.max_m, w.K), gen, device, 1.0, w.dtype)
    b = _randn((w.E, w.N, w.K), gen, device, 1.0 / math.sqrt(w.K), w.dtype)
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    meta = torch.randint(w.m_lo, w.m_hi + 1, (w.E,), generator=g, dtype=torch.int32)
    return {"a": a, "b": b, "meta": meta.to(device)}


# -------------------------------------------------------------- FP8 block-scaled grouped GEMM
@dataclasses.dataclass(frozen=True)
class Fp8GemmWorkload:
    """A masked-layout FP8 grouped GEMM (TileOPs MoE page, op MoEGroupedGemmFP8Fwd): a
    [E, max_m, K] and b [E, N, K] in E4M3 with f32 scales per 128-k block of a row of a and per
    128 x 128 block of b; `total` valid rows spread over the groups (the page's "T")."""
    name: str
    E: int
    max_m: int
    K: int
    N: int
    total: int

    def flops(self, valid_rows: int) -> float:
        return 2.0 * valid_rows * self.N * self.K


def _fp8_table():
    out = {}
    shapes = {"ds-v3": (7168, 4096, 2048), "qwen3-235b": (4096, 3072, 1536),
              "kimi-k2": (7168, 4096, 2048)}
    experts = {"ds-v3": 32, "qwen3-235b": 16, "kimi-k2": 48}
    rows = [("ds-v3-e8", 8, 128, 768)]
    for model in ("ds-v3", "qwen3-235b", "kimi-k2"):
        for b_, t in ((64, 64), (256, 256)):
            rows.append((f"{model}-dec-b{b_}", experts[model], b_, t))
    for prefix, E, max_m, T in rows:
        model = prefix.split("-dec")[0].replace("-e8", "")
        H, up_n, F = shapes[model]
        suffix = "-masked" if prefix == "ds-v3-e8" else ""
        out[f"{prefix}-up{suffix}"] = Fp8GemmWorkload(f"{prefix}-up{suffix}", E, max_m, H,
                                                      up_n, T)
        out[f"{prefix}-down{suffix}"] = Fp8GemmWorkload(f"{prefix}-down{suffix}", E, max_m, F,
                                                        H, T)
    return out


# The page's 14 MoEGroupedGemmFP8Fwd workloads (a [E, max_m, K], b [E, N, K], T valid rows).
FP8_GEMM_WORKLOADS = _fp8_table()


def quantize_fp8_blocks(x: torch.Tensor, block_rows: int):
    """x [rows, K] f32 -> (E4M3 bytes [rows, K], f32 scales [ceil(rows/block_rows), K/128]):
    one scale per block of block_rows x 128, amax / 448 (1 for an all-zero block), values
    rounded to nearest even by torch's float8_e4m3fn conversion."""
    rows, K = x.shape
    nb = (rows + block_rows - 1) // block_rows
    pad = nb * block_rows - rows
    xp = torch.nn.functional.pad(x, (0, 0, 0, pad)) if pad else x
    blocks = xp.view(nb, block_rows, K // 128, 128)
    amax = blocks.abs().amax(dim=(1, 3))  # [nb, K/128]
    scale = torch.where(amax > 0, amax / 448.0, torch.ones_like(amax))
    q = (blocks / scale[:, None, :, None]).clamp_(-448.0, 448.0).to(torch.float8_e4m3fn)
    q = q.view(nb * block_rows, K)[:rows]
    return q.view(torch.uint8).contiguous(), scale.contiguous()


def generate_fp8_gemm(w: Fp8GemmWorkload, seed: int = 0, device="cuda") -> dict:
    """a ~ N(0, 1) and b ~ N(0, 1/K) (one generator seeded with `seed`, a first), quantised
    to E4M3 with per-(row, 128-k) scales for a and per-(128 x 128) scales for b; the valid rows
    of each group are `total` draws of a uniformly random group (a CPU generator seeded with
    seed + 1), each count capped at max_m."""
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    a32 = _randn((w.E * w.max_m, w.K), gen, device, 1.0, torch.float32)
    a, a_scale = quantize_fp8_blocks(a32, 1)
    del a32
    b = torch.empty((w.E, w.N, w.K), dtype=torch.uint8, device=device)
    b_scale = torch.empty((w.E, w.N // 128, w.K // 128), dtype=torch.float32, device=device)
    for e in range(w.E):
        x = _randn((w.N, w.K), gen, device, 1.0 / math.sqrt(w.K), torch.float32)
        b[e], b_scale[e] = quantize_fp8_blocks(x, 128)
        del x
    g = torch.Generator(device="cpu")
    g.manual_seed(seed + 1)
    pick = torch.randint(0, w.E, (w.total,), generator=g)
    meta = torch.bincount(pick, minlength=w.E).clamp_(max=w.max_m).to(torch.int32)
    return {"a": a.view(w.E, w.max_m, w.K), "a_scale": a_scale.view(w.E, w.max_m, w.K // 128),
            "b": b, "b_scale": b_scale, "meta": meta.to(device)}
