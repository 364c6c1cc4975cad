"""Thin ctypes binding over libgb300moe.so, with the C ABI's names.

Argument marshalling only: every step of the path runs in the library's CUDA kernels.  torch is
used for device memory (outputs, workspaces) and for the current CUDA stream.  There is no
fallback: if the library cannot be loaded the call raises.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from . import build as _build

MOE_OK, MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED = 0, 1, 2
MOE_ERR_WORKSPACE_TOO_SMALL, MOE_ERR_CUDA, MOE_ERR_TIMEOUT, MOE_ERR_BAD_EXPERT_ID = 3, 4, 5, 6
MOE_ERR_F16_RANGE = 7
MOE_BF16, MOE_F16 = 0, 1
MOE_SOFTMAX, MOE_SIGMOID = 0, 1

_DTYPES = {torch.bfloat16: MOE_BF16, torch.float16: MOE_F16}
_SCORING = {"softmax": MOE_SOFTMAX, "sigmoid": MOE_SIGMOID}
# moe_activation_t: the two gated forms keep 2F rows per expert in w_gate_up, ReLU2 keeps F.
_ACTIVATIONS = {"silu": 0, "gelu_tanh": 1, "relu2": 2}


def gate_up_rows(activation: str, F: int) -> int:
    """Rows per expert of w_gate_up for `activation`."""
    if activation not in _ACTIVATIONS:
        raise ValueError(f"unsupported activation {activation}")
    return F if activation == "relu2" else 2 * F

# Every symbol include/moe.h declares.
EXPORTED = (
    "moe_workspace_size", "moe_workspace_size_w4a16", "moe_sorted_capacity",
    "moe_stage_workspace_size",
    "moe_workspace_init", "fused_moe_fwd", "moe_route", "moe_align_sort", "moe_gemm1_swiglu",
    "moe_gemm2", "moe_combine", "moe_shared_expert_fwd", "moe_get_device_status",
    "moe_status_string", "moe_set_wait_limit_ns", "moe_stage_name", "moe_profile_enable",
    "moe_profile_collect", "moe_align_sort_noalloc", "fused_moe_fwd_w4a16", "moe_gemm1_w4a16",
    "moe_gemm2_w4a16", "moe_nvfp4_pack", "moe_nvfp4_packed_bytes", "moe_pre_permute",
    "moe_grouped_gemm_workspace_size", "moe_grouped_gemm", "moe_post_permute",
    "moe_grouped_gemm_fp8", "moe_host_staging_bytes", "fused_moe_fwd_host",
    "fused_moe_fwd_w4a16_host",
)


class MoeProblem(ctypes.Structure):
    _fields_ = [
        ("T", ctypes.c_int32), ("H", ctypes.c_int32), ("E", ctypes.c_int32),
        ("F", ctypes.c_int32), ("top_k", ctypes.c_int32), ("dtype", ctypes.c_int32),
        ("scoring", ctypes.c_int32), ("renormalize", ctypes.c_int32),
        ("num_expert_group", ctypes.c_int32), ("topk_group", ctypes.c_int32),
        ("routed_scaling_factor", ctypes.c_float), ("S", ctypes.c_int32),
        ("activation", ctypes.c_int32), ("ep_num_local", ctypes.c_int32),
        ("ep_local_offset", ctypes.c_int32),
    ]


class GroupedGemm(ctypes.Structure):
    _fields_ = [
        ("E", ctypes.c_int32), ("N", ctypes.c_int32), ("K", ctypes.c_int32),
        ("max_m", ctypes.c_int32), ("rows", ctypes.c_int64), ("dtype", ctypes.c_int32),
        ("activation", ctypes.c_int32), ("out_f32", ctypes.c_int32),
    ]


class MoeError(RuntimeError):
    def __init__(self, code: int, what: str):
        self.code = code
        super().__init__(f"{what}: {status_string(code)} (code {code})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libgb300moe.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = ctypes.CDLL(path)
            P, sz, i32, i64, u64 = (ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32,
                                    ctypes.c_int64, ctypes.c_uint64)
            PP = ctypes.POINTER(MoeProblem)
            L.moe_workspace_size.restype = sz
            L.moe_workspace_size.argtypes = [PP]
            L.moe_workspace_size_w4a16.restype = sz
            L.moe_workspace_size_w4a16.argtypes = [PP]
            L.moe_sorted_capacity.restype = i64
            L.moe_sorted_capacity.argtypes = [PP, i32]
            L.moe_stage_workspace_size.restype = sz
            L.moe_stage_workspace_size.argtypes = [PP, i32]
            L.moe_workspace_init.argtypes = [P, sz, P]
            L.fused_moe_fwd.argtypes = [PP, P, P, P, P, P, P, P, P, P, sz, P]
            L.moe_route.argtypes = [PP, P, P, P, P, P]
            L.moe_align_sort.argtypes = [PP, i32, P, P, P, P, P, P, P, sz, P]
            L.moe_gemm1_swiglu.argtypes = [PP, i32, P, P, P, P, P, P, sz, P]
            L.moe_gemm2.argtypes = [PP, i32, P, P, P, P, P, P, P, sz, P]
            L.moe_combine.argtypes = [PP, P, P, P, P, P, P]
            L.moe_shared_expert_fwd.argtypes = [PP, P, P, P, P, P, sz, P]
            L.moe_get_device_status.argtypes = [P, P]
            L.moe_status_string.restype = ctypes.c_char_p
            L.moe_status_string.argtypes = [ctypes.c_int]
            L.moe_set_wait_limit_ns.restype = u64
            L.moe_set_wait_limit_ns.argtypes = [u64]
            L.moe_stage_name.restype = ctypes.c_char_p
            L.moe_stage_name.argtypes = [i32]
            L.moe_profile_enable.restype = ctypes.c_int
            L.moe_profile_enable.argtypes = [i32]
            L.moe_profile_collect.restype = i32
            L.moe_profile_collect.argtypes = [P, P, P, i32]
            L.moe_align_sort_noalloc.restype = ctypes.c_int
            L.moe_align_sort_noalloc.argtypes = [PP, i32, P, P, P, P, P, P, P, P]
            L.fused_moe_fwd_w4a16.argtypes = [PP, P, P, P, P, P, P, P, P, P, sz, P]
            L.moe_host_staging_bytes.restype = sz
            L.moe_host_staging_bytes.argtypes = [PP]
            L.fused_moe_fwd_host.argtypes = [PP, P, P, P, P, P, P, P, P, P, sz, P]
            L.fused_moe_fwd_w4a16_host.argtypes = [PP, P, P, P, P, P, P, P, P, P, sz, P]
            L.moe_gemm1_w4a16.argtypes = [PP, i32, P, P, P, P, P, P, P, sz, P]
            L.moe_gemm2_w4a16.argtypes = [PP, i32, P, P, P, P, P, P, P, P, sz, P]
            L.moe_nvfp4_pack.restype = ctypes.c_int
            L.moe_nvfp4_pack.argtypes = [i64, i32, i32, P, P, P, P]
            L.moe_pre_permute.argtypes = [PP, P, P, P, P, P, P, P, sz, P]
            GG = ctypes.POINTER(GroupedGemm)
            L.moe_grouped_gemm_workspace_size.restype = sz
            L.moe_grouped_gemm_workspace_size.argtypes = [GG]
            L.moe_grouped_gemm.argtypes = [GG, P, P, P, P, P, sz, P]
            L.moe_post_permute.argtypes = [PP, P, P, P, P, P]
            L.moe_grouped_gemm_fp8.argtypes = [GG, P, P, P, P, P, P, P, sz, P]
            L.moe_grouped_gemm_fp8.restype = ctypes.c_int
            for fn in ("moe_pre_permute", "moe_grouped_gemm", "moe_post_permute"):
                getattr(L, fn).restype = ctypes.c_int
            L.moe_nvfp4_packed_bytes.restype = i64
            L.moe_nvfp4_packed_bytes.argtypes = [i64, i32, i32]
            for fn in ("fused_moe_fwd", "moe_route", "moe_align_sort", "moe_gemm1_swiglu",
                       "moe_gemm2", "moe_combine", "moe_shared_expert_fwd",
                       "moe_get_device_status", "moe_workspace_init", "fused_moe_fwd_w4a16",
                       "moe_gemm1_w4a16", "moe_gemm2_w4a16"):
                getattr(L, fn).restype = ctypes.c_int
            _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().moe_status_string(int(code)).decode()


def _check(rc: int, what: str):
    if rc != MOE_OK:
        raise MoeError(rc, what)


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype=None, shape=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must have dtype {dtype}, got {t.dtype}")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)}, got {tuple(t.shape)}")
    return t


def make_problem(T, H, E, F, top_k, dtype=torch.bfloat16, scoring_func="softmax",
                 renormalize=True, num_expert_group=0, topk_group=0, routed_scaling_factor=1.0,
                 S=0, activation="silu", ep_num_local=0, ep_local_offset=0) -> MoeProblem:
    if dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {dtype}")
    if scoring_func not in _SCORING:
        raise ValueError(f"unsupported scoring_func {scoring_func}")
    if activation not in _ACTIVATIONS:
        raise ValueError(f"unsupported activation {activation}")
    return MoeProblem(int(T), int(H), int(E), int(F), int(top_k), _DTYPES[dtype],
                      _SCORING[scoring_func], int(bool(renormalize)), int(num_expert_group),
                      int(topk_group), float(routed_scaling_factor), int(S),
                      _ACTIVATIONS[activation], int(ep_num_local), int(ep_local_offset))


def workspace_size(prob: MoeProblem) -> int:
    n = lib().moe_workspace_size(ctypes.byref(prob))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_size")
    return int(n)


def workspace_size_w4a16(prob: MoeProblem) -> int:
    n = lib().moe_workspace_size_w4a16(ctypes.byref(prob))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_workspace_size_w4a16")
    return n


def stage_workspace_size(prob: MoeProblem, block_m: int) -> int:
    n = lib().moe_stage_workspace_size(ctypes.byref(prob), int(block_m))
    if n == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_stage_workspace_size")
    return int(n)


def sorted_capacity(prob: MoeProblem, block_m: int) -> int:
    n = lib().moe_sorted_capacity(ctypes.byref(prob), int(block_m))
    if n < 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_sorted_capacity")
    return int(n)


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """A zeroed uint8 device buffer (the status header must start at zero)."""
    return torch.zeros(int(nbytes), dtype=torch.uint8, device=device or "cuda")


_ws_cache: dict = {}


def _workspace(nbytes: int, device) -> torch.Tensor:
    key = (str(device), threading.get_ident())
    ws = _ws_cache.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = new_workspace(nbytes, device)
        _ws_cache[key] = ws
    return ws


def get_device_status(workspace: torch.Tensor, stream=None) -> int:
    return int(lib().moe_get_device_status(_p(workspace), _stream(stream)))


def set_wait_limit_ns(limit_ns: int) -> int:
    return int(lib().moe_set_wait_limit_ns(int(limit_ns)))


NUM_STAGES = 9


def stage_names():
    return [lib().moe_stage_name(i).decode() for i in range(NUM_STAGES)]


def profile_enable(stages=None):
    """Record event pairs around the named stages (all when None; none when [])."""
    names = stage_names()
    if stages is None:
        mask = (1 << NUM_STAGES) - 1
    else:
        mask = 0
        for s in stages:
            mask |= 1 << names.index(s)
    _check(lib().moe_profile_enable(mask), "moe_profile_enable")


def profile_collect() -> dict:
    """{stage: (total_ms, calls, launches)} since profile_enable; resets the totals."""
    ms = (ctypes.c_double * NUM_STAGES)()
    calls = (ctypes.c_int64 * NUM_STAGES)()
    launches = (ctypes.c_int64 * NUM_STAGES)()
    n = lib().moe_profile_collect(ms, calls, launches, NUM_STAGES)
    names = stage_names()
    return {names[i]: (float(ms[i]), int(calls[i]), int(launches[i])) for i in range(n)}


def fused_moe_fwd(hidden_states, gating_output, w_gate_up, w_down, top_k, renormalize=True,
                  scoring_func="softmax", correction_bias=None, num_expert_group=0, topk_group=0,
                  routed_scaling_factor=1.0, shared_w_gate_up=None, shared_w_down=None, out=None,
                  workspace=None, stream=None, activation="silu", ep_local_offset=0):
    """The whole fused MoE forward (include/moe.h: fused_moe_fwd); returns out [T, H].
    ``activation``: "silu" (default), "gelu_tanh" or "relu2" (w_gate_up then has F rows).
    When the weights hold fewer experts than gating_output scores, they are the shard
    [ep_local_offset, ep_local_offset + E_local) of an expert-parallel layout."""
    T, H = hidden_states.shape
    E = gating_output.shape[1]
    E_l = w_gate_up.shape[0]
    F = w_down.shape[2]
    S = 0 if shared_w_down is None else shared_w_down.shape[1]
    dt = hidden_states.dtype
    _need(hidden_states, "hidden_states", dt)
    _need(gating_output, "gating_output", torch.float32, (T, E))
    _need(w_gate_up, "w_gate_up", dt, (E_l, gate_up_rows(activation, F), H))
    _need(w_down, "w_down", dt, (E_l, H, F))
    if correction_bias is not None:
        _need(correction_bias, "correction_bias", torch.float32, (E,))
    if S:
        _need(shared_w_gate_up, "shared_w_gate_up", dt, (gate_up_rows(activation, S), H))
        _need(shared_w_down, "shared_w_down", dt, (H, S))
    prob = make_problem(T, H, E, F, top_k, dt, scoring_func, renormalize, num_expert_group,
                        topk_group, routed_scaling_factor, S, activation,
                        E_l if E_l != E else 0, ep_local_offset)
    nbytes = workspace_size(prob)
    if workspace is None:
        workspace = _workspace(nbytes, hidden_states.device)
    if out is None:
        out = torch.empty((T, H), dtype=dt, device=hidden_states.device)
    _need(out, "out", dt, (T, H))
    rc = lib().fused_moe_fwd(ctypes.byref(prob), _p(hidden_states), _p(gating_output),
                             _p(w_gate_up), _p(w_down), _p(correction_bias),
                             _p(shared_w_gate_up), _p(shared_w_down), _p(out), _p(workspace),
                             workspace.numel(), _stream(stream))
    _check(rc, "fused_moe_fwd")
    return out


def moe_route(gating_output, top_k, scoring_func="softmax", renormalize=True,
              correction_bias=None, num_expert_group=0, topk_group=0,
              routed_scaling_factor=1.0, stream=None):
    """Router top-k (include/moe.h: moe_route); returns (topk_ids int32, topk_weights f32)."""
    _need(gating_output, "gating_output", torch.float32)
    T, E = gating_output.shape
    if correction_bias is not None:
        _need(correction_bias, "correction_bias", torch.float32, (E,))
    prob = make_problem(T, 8, E, 8, top_k, torch.bfloat16, scoring_func, renormalize,
                        num_expert_group, topk_group, routed_scaling_factor)
    ids = torch.empty((T, top_k), dtype=torch.int32, device=gating_output.device)
    w = torch.empty((T, top_k), dtype=torch.float32, device=gating_output.device)
    _check(lib().moe_route(ctypes.byref(prob), _p(gating_output), _p(correction_bias), _p(ids),
                           _p(w), _stream(stream)), "moe_route")
    return ids, w


def moe_align_sort(topk_ids, num_experts, block_m=1, workspace=None, stream=None,
                   want_tile_expert=True):
    """Expert sort (include/moe.h: moe_align_sort); returns a dict of device tensors."""
    _need(topk_ids, "topk_ids", torch.int32)
    T, k = topk_ids.shape
    E = int(num_experts)
    prob = make_problem(T, 8, E, 8, k)
    cap = sorted_capacity(prob, block_m)
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    tile_len = (cap + block_m - 1) // block_m
    tile_expert = (torch.empty(max(tile_len, 1), dtype=torch.int32, device=dev)
                   if want_tile_expert else None)
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    nbytes = workspace_size(prob)
    if workspace is None:
        workspace = _workspace(nbytes, dev)
    _check(lib().moe_align_sort(ctypes.byref(prob), int(block_m), _p(topk_ids), _p(counts),
                                _p(offsets), _p(sorted_ids), _p(tile_expert), _p(inv),
                                _p(workspace), workspace.numel(), _stream(stream)),
           "moe_align_sort")
    return dict(counts=counts, offsets=offsets, sorted_ids=sorted_ids[:cap],
                tile_expert=None if tile_expert is None else tile_expert[:tile_len],
                inv_route=inv[:T * k], workspace=workspace)


def moe_align_sort_noalloc(topk_ids, num_experts, block_m=1, stream=None):
    """The expert sort with the library's static scratch instead of a workspace (include/moe.h:
    moe_align_sort_noalloc), for callers that cannot allocate device memory when they sort;
    the output tensors here are torch's, the sort itself allocates nothing.  Returns the same
    dict as moe_align_sort plus a device int32 `status`."""
    _need(topk_ids, "topk_ids", torch.int32)
    T, k = topk_ids.shape
    E = int(num_experts)
    prob = make_problem(T, 8, E, 8, k)
    cap = sorted_capacity(prob, block_m)
    dev = topk_ids.device
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_ids = torch.empty(max(cap, 1), dtype=torch.int32, device=dev)
    tile_len = (cap + block_m - 1) // block_m
    tile_expert = torch.empty(max(tile_len, 1), dtype=torch.int32, device=dev)
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    _check(lib().moe_align_sort_noalloc(ctypes.byref(prob), int(block_m), _p(topk_ids),
                                        _p(counts), _p(offsets), _p(sorted_ids),
                                        _p(tile_expert), _p(inv), _p(status), _stream(stream)),
           "moe_align_sort_noalloc")
    return dict(counts=counts, offsets=offsets, sorted_ids=sorted_ids[:cap],
                tile_expert=tile_expert[:tile_len], inv_route=inv[:T * k], status=status)


def moe_gemm1_swiglu(hidden_states, sorted_ids, offsets, w_gate_up, top_k, block_m=1,
                     workspace=None, stream=None, activation="silu"):
    """Grouped gate/up GEMM + activation (include/moe.h: moe_gemm1_swiglu); returns act
    [cap, F].  ``activation``: "silu" (SiLU(gate)*up), "gelu_tanh" or "relu2"."""
    T, H = hidden_states.shape
    E, rows, _ = w_gate_up.shape
    F = rows if activation == "relu2" else rows // 2
    dt = hidden_states.dtype
    _need(hidden_states, "hidden_states", dt)
    _need(w_gate_up, "w_gate_up", dt, (E, gate_up_rows(activation, F), H))
    _need(sorted_ids, "sorted_ids", torch.int32)
    _need(offsets, "offsets", torch.int32, (E + 1,))
    prob = make_problem(T, H, E, F, top_k, dt, activation=activation)
    cap = sorted_capacity(prob, block_m)
    act = torch.empty((max(cap, 1), F), dtype=dt, device=hidden_states.device)
    nbytes = stage_workspace_size(prob, block_m)
    if workspace is None:
        workspace = _workspace(nbytes, hidden_states.device)
    _check(lib().moe_gemm1_swiglu(ctypes.byref(prob), int(block_m), _p(hidden_states),
                                  _p(sorted_ids), _p(offsets), _p(w_gate_up), _p(act),
                                  _p(workspace), workspace.numel(), _stream(stream)),
           "moe_gemm1_swiglu")
    return act[:cap]


def moe_gemm2(act, sorted_ids, offsets, topk_weights, w_down, T, top_k, block_m=1,
              workspace=None, stream=None):
    """Grouped down GEMM x route weight (include/moe.h: moe_gemm2); returns f32 y_route
    [cap, H]."""
    E, H, F = w_down.shape
    dt = w_down.dtype
    _need(w_down, "w_down", dt)
    _need(act, "act", dt)
    _need(sorted_ids, "sorted_ids", torch.int32)
    _need(offsets, "offsets", torch.int32, (E + 1,))
    _need(topk_weights, "topk_weights", torch.float32)
    prob = make_problem(T, H, E, F, top_k, dt)
    cap = sorted_capacity(prob, block_m)
    if act.shape[0] < cap or act.shape[1] != F:
        raise ValueError(f"act must have at least {cap} rows of {F} columns")
    y = torch.empty((max(cap, 1), H), dtype=torch.float32, device=w_down.device)
    nbytes = stage_workspace_size(prob, block_m)
    if workspace is None:
        workspace = _workspace(nbytes, w_down.device)
    _check(lib().moe_gemm2(ctypes.byref(prob), int(block_m), _p(act), _p(sorted_ids),
                           _p(offsets), _p(topk_weights), _p(w_down), _p(y), _p(workspace),
                           workspace.numel(), _stream(stream)), "moe_gemm2")
    return y[:cap]


def moe_combine(y_route, inv_route, T, top_k, topk_ids=None, shared_out=None, out=None,
                dtype=torch.bfloat16, stream=None, E=None, ep_num_local=0, ep_local_offset=0):
    """Deterministic top-k combine (include/moe.h: moe_combine) of f32 rows; returns out
    [T, H] in `dtype`.  E, ep_num_local and ep_local_offset describe an expert-parallel shard
    (topk_ids then hold local ids, -1 for routes to other shards)."""
    _need(y_route, "y_route", torch.float32)
    H = y_route.shape[1]
    if inv_route is not None:
        _need(inv_route, "inv_route", torch.int32)
    if topk_ids is not None:
        _need(topk_ids, "topk_ids", torch.int32)
    if shared_out is not None:
        _need(shared_out, "shared_out", torch.float32, (T, H))
    prob = make_problem(T, H, E if E is not None else max(top_k, 1), 8, top_k, dtype,
                        ep_num_local=ep_num_local, ep_local_offset=ep_local_offset)
    if out is None:
        out = torch.empty((T, H), dtype=dtype, device=y_route.device)
    _check(lib().moe_combine(ctypes.byref(prob), _p(y_route), _p(inv_route), _p(topk_ids),
                             _p(shared_out), _p(out), _stream(stream)), "moe_combine")
    return out


def moe_shared_expert_fwd(hidden_states, shared_w_gate_up, shared_w_down, workspace=None,
                          stream=None, activation="silu"):
    """Dense shared expert (include/moe.h: moe_shared_expert_fwd); returns f32 [T, H]."""
    T, H = hidden_states.shape
    S = shared_w_down.shape[1]
    dt = hidden_states.dtype
    _need(hidden_states, "hidden_states", dt)
    _need(shared_w_gate_up, "shared_w_gate_up", dt, (gate_up_rows(activation, S), H))
    _need(shared_w_down, "shared_w_down", dt, (H, S))
    prob = make_problem(T, H, 1, 8, 1, dt, S=S, activation=activation)
    out = torch.empty((T, H), dtype=torch.float32, device=hidden_states.device)
    nbytes = workspace_size(prob)
    if workspace is None:
        workspace = _workspace(nbytes, hidden_states.device)
    _check(lib().moe_shared_expert_fwd(ctypes.byref(prob), _p(hidden_states),
                                       _p(shared_w_gate_up), _p(shared_w_down), _p(out),
                                       _p(workspace), workspace.numel(), _stream(stream)),
           "moe_shared_expert_fwd")
    return out


def _need_host(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor) or t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous host tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must be {dtype} {tuple(shape)}, got {t.dtype} {tuple(t.shape)}")


def host_workspace_size(prob: MoeProblem, w4a16=False) -> int:
    """Workspace bytes of the host entry points: the fused call's plus the device staging of
    the inputs and the output (include/moe.h: moe_host_staging_bytes)."""
    base = workspace_size_w4a16(prob) if w4a16 else workspace_size(prob)
    return base + int(lib().moe_host_staging_bytes(ctypes.byref(prob)))


def fused_moe_fwd_host(hidden_host, gating_host, w_gate_up, w_down, top_k, renormalize=True,
                       scoring_func="softmax", correction_bias=None, num_expert_group=0,
                       topk_group=0, routed_scaling_factor=1.0, shared_w_gate_up=None,
                       shared_w_down=None, out_host=None, workspace=None, stream=None,
                       activation="silu", ep_local_offset=0):
    """The fused forward from HOST buffers in one library call (include/moe.h:
    fused_moe_fwd_host, or fused_moe_fwd_w4a16_host for Nvfp4Weights): the host->device copies
    of hidden_host and gating_host, the fused path and the device->host copy into out_host
    (page-locked when it is created here) are all enqueued on the stream by the library.
    Returns out_host, valid once the stream has reached the end of the call."""
    w4 = isinstance(w_gate_up, Nvfp4Weights)
    T, H = hidden_host.shape
    E = gating_host.shape[1]
    dt = hidden_host.dtype
    dev = w_gate_up.device
    if w4:
        E_l, F = w_gate_up.n_mats, w_down.K
        _need_w4(w_gate_up, "w_gate_up", E_l, gate_up_rows(activation, F), H)
        _need_w4(w_down, "w_down", E_l, H, F)
        S = 0
    else:
        E_l, F = w_gate_up.shape[0], w_down.shape[2]
        _need(w_gate_up, "w_gate_up", dt, (E_l, gate_up_rows(activation, F), H))
        _need(w_down, "w_down", dt, (E_l, H, F))
        S = 0 if shared_w_down is None else shared_w_down.shape[1]
    _need_host(hidden_host, "hidden_host", dt, (T, H))
    _need_host(gating_host, "gating_host", torch.float32, (T, E))
    if correction_bias is not None:
        _need(correction_bias, "correction_bias", torch.float32, (E,))
    prob = make_problem(T, H, E, F, top_k, dt, scoring_func, renormalize, num_expert_group,
                        topk_group, routed_scaling_factor, S, activation,
                        E_l if E_l != E else 0, ep_local_offset)
    if workspace is None:
        workspace = _workspace(host_workspace_size(prob, w4), dev)
    if out_host is None:
        out_host = torch.empty((T, H), dtype=dt, pin_memory=True)
    _need_host(out_host, "out_host", dt, (T, H))
    if w4:
        rc = lib().fused_moe_fwd_w4a16_host(
            ctypes.byref(prob), _p(hidden_host), _p(gating_host), _p(w_gate_up.tiles),
            _p(w_gate_up.alpha), _p(w_down.tiles), _p(w_down.alpha), _p(correction_bias),
            _p(out_host), _p(workspace), workspace.numel(), _stream(stream))
        _check(rc, "fused_moe_fwd_w4a16_host")
    else:
        rc = lib().fused_moe_fwd_host(
            ctypes.byref(prob), _p(hidden_host), _p(gating_host), _p(w_gate_up), _p(w_down),
            _p(correction_bias), _p(shared_w_gate_up), _p(shared_w_down), _p(out_host),
            _p(workspace), workspace.numel(), _stream(stream))
        _check(rc, "fused_moe_fwd_host")
    return out_host


# ------------------------------------------------------------------------ NVFP4 (W4A16) experts
class Nvfp4Weights:
    """One projection of all (local) experts in the packed layout of moe_nvfp4_pack: `tiles`
    (uint8), the per-expert FP32 scale `alpha` [n_mats], and the matrix shape rows x K."""

    def __init__(self, tiles, alpha, n_mats, rows, K):
        self.tiles, self.alpha, self.n_mats, self.rows, self.K = tiles, alpha, n_mats, rows, K

    @property
    def device(self):
        return self.tiles.device


def nvfp4_packed_bytes(n_mats, rows, K) -> int:
    n = lib().moe_nvfp4_packed_bytes(int(n_mats), int(rows), int(K))
    if n < 0:
        raise MoeError(MOE_ERR_UNSUPPORTED, "moe_nvfp4_packed_bytes")
    return int(n)


def pack_nvfp4_weights(codes, scales, alpha, stream=None) -> Nvfp4Weights:
    """codes [n, rows, K/2] u8, scales [n, rows, K/16] u8, alpha [n] f32 -> Nvfp4Weights
    (include/moe.h: moe_nvfp4_pack)."""
    n, rows, half_k = codes.shape
    K = half_k * 2
    _need(codes, "codes", torch.uint8)
    _need(scales, "scales", torch.uint8, (n, rows, K // 16))
    _need(alpha, "alpha", torch.float32, (n,))
    tiles = torch.empty(nvfp4_packed_bytes(n, rows, K), dtype=torch.uint8, device=codes.device)
    _check(lib().moe_nvfp4_pack(n, rows, K, _p(codes), _p(scales), _p(tiles), _stream(stream)),
           "moe_nvfp4_pack")
    return Nvfp4Weights(tiles, alpha, n, rows, K)


def _need_w4(w, name, E_l, rows, K):
    if not isinstance(w, Nvfp4Weights):
        raise TypeError(f"{name} must be Nvfp4Weights (pack_nvfp4_weights)")
    if (w.n_mats, w.rows, w.K) != (E_l, rows, K):
        raise ValueError(f"{name} must hold {E_l} matrices of {rows} x {K}, "
                         f"got {w.n_mats} of {w.rows} x {w.K}")
    _need(w.tiles, name + " tiles", torch.uint8)
    _need(w.alpha, name + " alpha", torch.float32, (E_l,))


def fused_moe_fwd_w4a16(hidden_states, gating_output, w_gate_up, w_down, top_k, renormalize=True,
                        scoring_func="softmax", correction_bias=None, num_expert_group=0,
                        topk_group=0, routed_scaling_factor=1.0, out=None, workspace=None,
                        stream=None, activation="silu", ep_local_offset=0):
    """Fused MoE forward with NVFP4 routed experts (include/moe.h: fused_moe_fwd_w4a16).
    w_gate_up / w_down are Nvfp4Weights; returns out [T, H] bf16."""
    T, H = hidden_states.shape
    E = gating_output.shape[1]
    E_l = w_gate_up.n_mats
    F = w_down.K
    dt = hidden_states.dtype
    _need(hidden_states, "hidden_states", torch.bfloat16)
    _need(gating_output, "gating_output", torch.float32, (T, E))
    _need_w4(w_gate_up, "w_gate_up", E_l, gate_up_rows(activation, F), H)
    _need_w4(w_down, "w_down", E_l, H, F)
    if correction_bias is not None:
        _need(correction_bias, "correction_bias", torch.float32, (E,))
    prob = make_problem(T, H, E, F, top_k, dt, scoring_func, renormalize, num_expert_group,
                        topk_group, routed_scaling_factor, 0, activation,
                        E_l if E_l != E else 0, ep_local_offset)
    nbytes = workspace_size_w4a16(prob)
    if workspace is None:
        workspace = _workspace(nbytes, hidden_states.device)
    if out is None:
        out = torch.empty((T, H), dtype=dt, device=hidden_states.device)
    _need(out, "out", dt, (T, H))
    rc = lib().fused_moe_fwd_w4a16(ctypes.byref(prob), _p(hidden_states), _p(gating_output),
                                   _p(w_gate_up.tiles), _p(w_gate_up.alpha), _p(w_down.tiles),
                                   _p(w_down.alpha), _p(correction_bias), _p(out),
                                   _p(workspace), workspace.numel(), _stream(stream))
    _check(rc, "fused_moe_fwd_w4a16")
    return out


def moe_gemm1_w4a16(hidden_states, sorted_ids, offsets, w_gate_up, top_k, block_m=1,
                    workspace=None, stream=None, activation="silu"):
    """Grouped gate/up GEMM with NVFP4 weights + activation (include/moe.h: moe_gemm1_w4a16);
    returns act [cap, F] f16 (the type the NVFP4 GEMMs compute in)."""
    T, H = hidden_states.shape
    E_l, rows = w_gate_up.n_mats, w_gate_up.rows
    F = rows if activation == "relu2" else rows // 2
    _need(hidden_states, "hidden_states", torch.bfloat16)
    _need_w4(w_gate_up, "w_gate_up", E_l, gate_up_rows(activation, F), H)
    _need(sorted_ids, "sorted_ids", torch.int32)
    _need(offsets, "offsets", torch.int32, (E_l + 1,))
    prob = make_problem(T, H, E_l, F, top_k, torch.bfloat16, activation=activation)
    cap = sorted_capacity(prob, block_m)
    act = torch.empty((max(cap, 1), F), dtype=torch.float16, device=hidden_states.device)
    nbytes = stage_workspace_size(prob, block_m)
    if workspace is None:
        workspace = _workspace(nbytes, hidden_states.device)
    _check(lib().moe_gemm1_w4a16(ctypes.byref(prob), int(block_m), _p(hidden_states),
                                 _p(sorted_ids), _p(offsets), _p(w_gate_up.tiles),
                                 _p(w_gate_up.alpha), _p(act), _p(workspace), workspace.numel(),
                                 _stream(stream)), "moe_gemm1_w4a16")
    return act[:cap]


def moe_gemm2_w4a16(act, sorted_ids, offsets, topk_weights, w_down, T, top_k, block_m=1,
                    workspace=None, stream=None):
    """Grouped down GEMM with NVFP4 weights x route weight (include/moe.h: moe_gemm2_w4a16);
    act is f16, as moe_gemm1_w4a16 returns it; returns f32 y_route [cap, H]."""
    E_l, H, F = w_down.n_mats, w_down.rows, w_down.K
    _need_w4(w_down, "w_down", E_l, H, F)
    _need(act, "act", torch.float16)
    _need(sorted_ids, "sorted_ids", torch.int32)
    _need(offsets, "offsets", torch.int32, (E_l + 1,))
    _need(topk_weights, "topk_weights", torch.float32)
    prob = make_problem(T, H, E_l, F, top_k, torch.bfloat16)
    cap = sorted_capacity(prob, block_m)
    if act.shape[0] < cap or act.shape[1] != F:
        raise ValueError(f"act must have at least {cap} rows of {F} columns")
    y = torch.empty((max(cap, 1), H), dtype=torch.float32, device=act.device)
    nbytes = stage_workspace_size(prob, block_m)
    if workspace is None:
        workspace = _workspace(nbytes, act.device)
    _check(lib().moe_gemm2_w4a16(ctypes.byref(prob), int(block_m), _p(act), _p(sorted_ids),
                                 _p(offsets), _p(topk_weights), _p(w_down.tiles),
                                 _p(w_down.alpha), _p(y), _p(workspace), workspace.numel(),
                                 _stream(stream)), "moe_gemm2_w4a16")
    return y[:cap]


# ---------------------------------------------------------- expert-parallel building blocks
def moe_pre_permute(hidden_states, local_ids, num_local_experts, workspace=None, stream=None):
    """Rows of hidden_states in local-expert order (include/moe.h: moe_pre_permute).  Returns
    dict(permuted [T*k, H], offsets [E+1], sorted_ids [T*k], inv_route [T*k])."""
    T, H = hidden_states.shape
    k = local_ids.shape[1]
    E = int(num_local_experts)
    dt = hidden_states.dtype
    _need(hidden_states, "hidden_states", dt)
    _need(local_ids, "local_ids", torch.int32, (T, k))
    prob = make_problem(T, H, E, 8, k, dt)
    dev = hidden_states.device
    permuted = torch.empty((max(T * k, 1), H), dtype=dt, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    sorted_ids = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    inv = torch.empty(max(T * k, 1), dtype=torch.int32, device=dev)
    nbytes = workspace_size(prob)
    if workspace is None:
        workspace = _workspace(nbytes, dev)
    _check(lib().moe_pre_permute(ctypes.byref(prob), _p(hidden_states), _p(local_ids),
                                 _p(permuted), _p(offsets), _p(sorted_ids), _p(inv),
                                 _p(workspace), workspace.numel(), _stream(stream)),
           "moe_pre_permute")
    return dict(permuted=permuted[:T * k], offsets=offsets, sorted_ids=sorted_ids[:T * k],
                inv_route=inv[:T * k])


def grouped_gemm_desc(a, b, activation="none", out_f32=False) -> GroupedGemm:
    """The moe_grouped_gemm_t of a (masked [E, max_m, K] or contiguous [P, K]) and b."""
    E = b.shape[0]
    N = b.shape[1] // (2 if activation == "silu" else 1)
    K = b.shape[2]
    if activation not in ("none", "silu"):
        raise ValueError(f"unsupported grouped-GEMM activation {activation}")
    max_m = a.shape[1] if a.dim() == 3 else 0
    rows = 0 if a.dim() == 3 else a.shape[0]
    return GroupedGemm(E, N, K, max_m, rows, _DTYPES[a.dtype], 1 if activation == "silu" else 0,
                       int(bool(out_f32)))


def moe_grouped_gemm(a, b, layout_metadata, activation="none", out_f32=False, out=None,
                     workspace=None, stream=None):
    """Grouped GEMM (include/moe.h: moe_grouped_gemm).  a [E, max_m, K] with valid-row counts
    (masked layout) or a [P, K] with inclusive prefix sums (contiguous layout); b [E, N, K], or
    [E, 2N, K] with activation="silu" (silu_and_mul).  Returns out shaped like a with N cols."""
    g = grouped_gemm_desc(a, b, activation, out_f32)
    dt = a.dtype
    _need(a, "a", dt)
    _need(b, "b", dt)
    _need(layout_metadata, "layout_metadata", torch.int32, (g.E,))
    shape = tuple(a.shape[:-1]) + (g.N,)
    odt = torch.float32 if out_f32 else dt
    if out is None:
        out = torch.zeros(shape, dtype=odt, device=a.device)
    _need(out, "out", odt, shape)
    nbytes = lib().moe_grouped_gemm_workspace_size(ctypes.byref(g))
    if nbytes == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_grouped_gemm_workspace_size")
    if workspace is None:
        workspace = _workspace(int(nbytes), a.device)
    _check(lib().moe_grouped_gemm(ctypes.byref(g), _p(a), _p(b), _p(layout_metadata), _p(out),
                                  _p(workspace), workspace.numel(), _stream(stream)),
           "moe_grouped_gemm")
    return out


def moe_post_permute(rows, topk_weights, inv_route, stream=None):
    """Weighted top-k combine (include/moe.h: moe_post_permute); returns out [T, H]."""
    T, k = topk_weights.shape
    H = rows.shape[1]
    dt = rows.dtype
    _need(rows, "rows", dt)
    _need(topk_weights, "topk_weights", torch.float32, (T, k))
    _need(inv_route, "inv_route", torch.int32)
    prob = make_problem(T, H, k, 8, k, dt)
    out = torch.empty((T, H), dtype=dt, device=rows.device)
    _check(lib().moe_post_permute(ctypes.byref(prob), _p(rows), _p(topk_weights), _p(inv_route),
                                  _p(out), _stream(stream)), "moe_post_permute")
    return out


def moe_grouped_gemm_fp8(a, a_scale, b, b_scale, layout_metadata, out=None, workspace=None,
                         stream=None):
    """FP8 block-scaled grouped GEMM (include/moe.h: moe_grouped_gemm_fp8).  a: E4M3 bytes
    [E, max_m, K] (masked) or [rows, K] (contiguous), a_scale [.., K/128] f32, b [E, N, K] E4M3
    bytes, b_scale [E, N/128, K/128] f32.  Returns bf16 out shaped like a with N columns."""
    E, N, K = b.shape
    max_m = a.shape[1] if a.dim() == 3 else 0
    rows = 0 if a.dim() == 3 else a.shape[0]
    g = GroupedGemm(E, N, K, max_m, rows, MOE_BF16, 0, 0)
    _need(a, "a", torch.uint8)
    _need(a_scale, "a_scale", torch.float32, tuple(a.shape[:-1]) + (K // 128,))
    _need(b, "b", torch.uint8)
    _need(b_scale, "b_scale", torch.float32, (E, N // 128, K // 128))
    _need(layout_metadata, "layout_metadata", torch.int32, (E,))
    shape = tuple(a.shape[:-1]) + (N,)
    if out is None:
        out = torch.zeros(shape, dtype=torch.bfloat16, device=a.device)
    _need(out, "out", torch.bfloat16, shape)
    nbytes = lib().moe_grouped_gemm_workspace_size(ctypes.byref(g))
    if nbytes == 0:
        raise MoeError(MOE_ERR_INVALID_ARG, "moe_grouped_gemm_workspace_size")
    if workspace is None:
        workspace = _workspace(int(nbytes), a.device)
    _check(lib().moe_grouped_gemm_fp8(ctypes.byref(g), _p(a), _p(a_scale), _p(b), _p(b_scale),
                                      _p(layout_metadata), _p(out), _p(workspace),
                                      workspace.numel(), _stream(stream)),
           "moe_grouped_gemm_fp8")
    return out
