"""CPU oracle for the fused MoE forward pass -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` / ``--impl reference``
legs of ``bench.py`` may import this package.  The product library never loads it, and it
imports nothing from the product package.

The arithmetic lives in ``oracle.c`` (plain C, fp64, a per-token loop); this module compiles it
with gcc (``build()``), loads it with ctypes and marshals numpy arrays.  Each function cites the
passage of the source pages it follows in ``oracle.c``.

Sources: TileOPs benchmark page, "MoE" section (ops FusedMoEFwd, FusedMoESharedExpertFwd,
FusedTopKFwd, MoEPermuteAlignFwd, MoEPostPermuteFwd, MoEGroupedGemmFwd silu_and_mul,
SharedExpertMLPFwd); ROCm/aiter PR #5973 "[FlyDSL] Optimize MI308 MoE decoding (3/3)",
"Changes" (expert id -1 is a skipped padding route; the sort returns each route's sorted row).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

OK, ERR_ARG, ERR_ID = 0, 1, 6
BF16, F16 = 0, 1
SOFTMAX, SIGMOID = 0, 1
ACT_SILU, ACT_GELU_TANH, ACT_RELU2 = 0, 1, 2


def gate_up_rows(activation: int, F: int) -> int:
    """Rows per expert of w_gate_up: 2F for the gated activations, F for ReLU2."""
    return F if activation == ACT_RELU2 else 2 * F


def build(force: bool = False) -> str:
    """Compile oracle.c into oracle/_build/liboracle.so (gcc, OpenMP when available)."""
    os.makedirs(_BUILD, exist_ok=True)
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]
    try:
        subprocess.run(base + ["-fopenmp", "-o", tmp, _SRC, "-lm"], check=True,
                       capture_output=True, text=True)
    except subprocess.CalledProcessError:
        subprocess.run(base + ["-o", tmp, _SRC, "-lm"], check=True, capture_output=True, text=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
            _lib.oracle_half_bits_to_double.restype = f64
            _lib.oracle_half_bits_to_double.argtypes = [i32, ctypes.c_uint16]
            _lib.oracle_decode_array.argtypes = [i32, P, P, i64]
            _lib.oracle_exp_f32.restype = ctypes.c_float
            _lib.oracle_exp_f32.argtypes = [ctypes.c_float]
            _lib.oracle_sigmoid_key_f32.restype = ctypes.c_float
            _lib.oracle_sigmoid_key_f32.argtypes = [ctypes.c_float]
            _lib.oracle_route.argtypes = [i32, i32, i32, i32, i32, i32, i32, f64, P, P, P, P, P]
            _lib.oracle_route_select_f64.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P]
            _lib.oracle_align_sort.argtypes = [i32, i32, i32, i32, P, P, P, P, i64, P, i64, P]
            _lib.oracle_moe_tokens.argtypes = [i32, P, i32, i32, i32, i32, i32, i32, i32, P, P, P,
                                               P, P, P, i32, P, P, P, P]
            _lib.oracle_expert_act.argtypes = [i32, i32, i32, i32, i32, P, P, P, P]
            _lib.oracle_expert_down.argtypes = [i32, i32, i32, i32, P, P, P, P, P]
            _lib.oracle_combine.argtypes = [i32, i32, i32, i32, P, P, P, P]
            _lib.oracle_num_threads.restype = i32
            _lib.oracle_grouped_gemm.argtypes = [i32, i32, i32, i32, i64, i32, i32, P, P, P, P]
            _lib.oracle_grouped_gemm_fp8.argtypes = [i32, i32, i32, i32, i64, P, P, P, P, P, P]
            _lib.oracle_post_permute.argtypes = [i32, i32, i32, i32, P, P, P, P]
            _lib.oracle_e2m1_to_double.restype = f64
            _lib.oracle_e2m1_to_double.argtypes = [i32]
            _lib.oracle_e4m3_to_double.restype = f64
            _lib.oracle_e4m3_to_double.argtypes = [i32]
            _lib.oracle_nvfp4_dequant.argtypes = [i64, i32, P, P, P, i64, P]
            _lib.oracle_moe_tokens_w4.argtypes = [i32, P, i32, i32, i32, i32, i32, i32, i32,
                                                  i32, P, P, P, P, P, P, P, P, P, P, P]
            _lib.oracle_expert_act_w4.argtypes = [i32, i32, i32, i32, i32, P, P, P, P, P, P]
            _lib.oracle_expert_down_w4.argtypes = [i32, i32, i32, i32, P, P, P, P, P, P, P]
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def _bits(a):
    """Accept a uint16/int16 bit array (or a torch bf16/f16 tensor) and return uint16 bits."""
    if a is None:
        return None
    if hasattr(a, "view") and hasattr(a, "dtype") and "torch" in type(a).__module__:
        import torch
        t = a.detach().contiguous().cpu()
        return t.view(torch.int16).numpy().view(np.uint16)
    return np.ascontiguousarray(a).view(np.uint16)


def _check(rc, what):
    if rc == ERR_ID:
        raise ValueError(f"{what}: expert id out of range")
    if rc != OK:
        raise ValueError(f"{what}: invalid arguments (code {rc})")


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def half_bits_to_double(dtype: int, bits: np.ndarray) -> np.ndarray:
    b = _c(bits, np.uint16)
    out = np.empty(b.shape, np.float64)
    _load().oracle_decode_array(dtype, _ptr(b), _ptr(out), b.size)
    return out


def exp_f32(z: float) -> float:
    return float(_load().oracle_exp_f32(float(z)))


def sigmoid_key_f32(x: float) -> float:
    return float(_load().oracle_sigmoid_key_f32(float(x)))


def route(gating, top_k, scoring=SOFTMAX, renormalize=True, num_expert_group=0, topk_group=0,
          routed_scaling_factor=1.0, bias=None):
    """Return (ids int32 [T,k], weights float64 [T,k], near_tie int32 [T])."""
    g = _c(gating, np.float32)
    T, E = g.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, top_k), np.int32)
    w = np.empty((T, top_k), np.float64)
    nt = np.empty((T,), np.int32)
    rc = _load().oracle_route(T, E, top_k, scoring, int(bool(renormalize)), num_expert_group,
                              topk_group, float(routed_scaling_factor), _ptr(g), _ptr(b),
                              _ptr(ids), _ptr(w), _ptr(nt))
    _check(rc, "oracle_route")
    return ids, w, nt


def route_select_f64(gating, top_k, num_expert_group=0, topk_group=0, bias=None):
    """The sigmoid (+ correction bias, + groups) selection on the plain fp64 definition
    (oracle.c: oracle_route_select_f64).  Returns (ids int32 [T,k] in descending key order,
    boundary_gap float64 [T], order_gap float64 [T])."""
    g = _c(gating, np.float32)
    T, E = g.shape
    b = None if bias is None else _c(bias, np.float32)
    ids = np.empty((T, top_k), np.int32)
    bgap = np.empty((T,), np.float64)
    ogap = np.empty((T,), np.float64)
    rc = _load().oracle_route_select_f64(T, E, top_k, num_expert_group, topk_group, _ptr(g),
                                         _ptr(b), _ptr(ids), _ptr(bgap), _ptr(ogap))
    _check(rc, "oracle_route_select_f64")
    return ids, bgap, ogap


def align_sort(ids, E, block_m):
    """Counting sort of flat routes into expert segments padded to block_m.

    Returns dict(counts, offsets, sorted_ids, tile_expert, inv_route); sorted_ids has
    P + E*(block_m-1) slots and tile_expert that many / block_m (rounded up)."""
    i = _c(ids, np.int32)
    T, k = i.shape
    P = T * k
    sorted_len = P + E * (block_m - 1)
    tile_len = (sorted_len + block_m - 1) // block_m
    counts = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    sorted_ids = np.empty(sorted_len, np.int32)
    tile_expert = np.empty(tile_len, np.int32)
    inv = np.empty(P, np.int32)
    rc = _load().oracle_align_sort(T, k, E, block_m, _ptr(i), _ptr(counts), _ptr(offsets),
                                   _ptr(sorted_ids), sorted_len, _ptr(tile_expert), tile_len,
                                   _ptr(inv))
    _check(rc, "oracle_align_sort")
    return dict(counts=counts, offsets=offsets, sorted_ids=sorted_ids, tile_expert=tile_expert,
                inv_route=inv)


def moe_tokens(hidden, ids, weights, w_gate_up, w_down, dtype, tokens=None, expert_slot=None,
               shared_w_gate_up=None, shared_w_down=None, num_experts=None,
               activation=ACT_SILU, act_noise=False):
    """fp64 fused MoE output for the listed tokens (all tokens when ``tokens`` is None).

    hidden/w_* are 16-bit bit arrays (or torch tensors).  When ``expert_slot`` is given,
    w_gate_up/w_down hold only the slots it maps experts to and ``num_experts`` is E.
    ``activation`` is ACT_SILU, ACT_GELU_TANH (both gated: w_gate_up has 2F rows per expert) or
    ACT_RELU2 (F rows per expert).  With ``act_noise`` returns (out, noise): noise is the
    per-element scale of the error that rounding each act value to ``dtype`` before the down
    projection adds (oracle.c: oracle_moe_tokens)."""
    hb = _bits(hidden)
    T, H = hb.shape
    idv = _c(ids, np.int32)
    k = idv.shape[1]
    wv = _c(weights, np.float64)
    wgu = _bits(w_gate_up)
    wd = _bits(w_down)
    F = wd.shape[-1]
    E = num_experts if num_experts is not None else wgu.shape[0]
    slot = None if expert_slot is None else _c(expert_slot, np.int32)
    sgu = _bits(shared_w_gate_up)
    sd = _bits(shared_w_down)
    S = 0 if sd is None else sd.shape[-1]
    tl = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    out = np.empty((tl.size, H), np.float64)
    noise = np.empty((tl.size, H), np.float64) if act_noise else None
    if wgu.shape[-2] != gate_up_rows(activation, F) or (
            sgu is not None and sgu.shape[0] != gate_up_rows(activation, S)):
        raise ValueError("w_gate_up rows do not match the activation")
    rc = _load().oracle_moe_tokens(tl.size, _ptr(tl), T, H, E, F, k, dtype, activation,
                                   _ptr(hb), _ptr(idv),
                                   _ptr(wv), _ptr(wgu), _ptr(wd), _ptr(slot), S, _ptr(sgu),
                                   _ptr(sd), _ptr(out), _ptr(noise))
    _check(rc, "oracle_moe_tokens")
    return (out, noise) if act_noise else out


def expert_act(x_rows, expert_of_row, w_gate_up, dtype, activation=ACT_SILU):
    xb = _bits(x_rows)
    n, H = xb.shape
    wgu = _bits(w_gate_up)
    F = wgu.shape[1] if activation == ACT_RELU2 else wgu.shape[1] // 2
    eo = _c(expert_of_row, np.int32)
    act = np.empty((n, F), np.float64)
    _check(_load().oracle_expert_act(n, H, F, dtype, activation, _ptr(xb), _ptr(eo), _ptr(wgu),
                                     _ptr(act)), "oracle_expert_act")
    return act


def expert_down(act_rows, expert_of_row, scale, w_down, dtype):
    ab = _bits(act_rows)
    n, F = ab.shape
    wd = _bits(w_down)
    H = wd.shape[1]
    eo = _c(expert_of_row, np.int32)
    sc = _c(scale, np.float64)
    y = np.empty((n, H), np.float64)
    _check(_load().oracle_expert_down(n, H, F, dtype, _ptr(ab), _ptr(eo), _ptr(sc), _ptr(wd),
                                      _ptr(y)), "oracle_expert_down")
    return y


def combine(rows, inv_route, top_k, dtype, shared=None):
    rb = _bits(rows)
    H = rb.shape[1]
    inv = _c(inv_route, np.int32)
    T = inv.size // top_k
    sb = _bits(shared)
    out = np.empty((T, H), np.float64)
    _check(_load().oracle_combine(T, H, top_k, dtype, _ptr(rb), _ptr(inv), _ptr(sb), _ptr(out)),
           "oracle_combine")
    return out


# ---------------------------------------------------------------------------- NVFP4 weights
def e2m1_to_double(code: int) -> float:
    return _load().oracle_e2m1_to_double(int(code))


def e4m3_to_double(bits: int) -> float:
    return _load().oracle_e4m3_to_double(int(bits))


def _u8(a):
    if a is None:
        return None
    if hasattr(a, "cpu") and "torch" in type(a).__module__:
        a = a.cpu().contiguous().view(__import__("torch").uint8).numpy()
    return np.ascontiguousarray(a, dtype=np.uint8)


def _f32(a):
    if hasattr(a, "cpu") and "torch" in type(a).__module__:
        a = a.cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.float32)


def nvfp4_dequant(q, sf, alpha, rows_per_alpha=None):
    """fp64 [rows, K] from NVFP4 q [.., rows, K/2] u8, sf [.., rows, K/16] u8 and alpha (one per
    leading index, or per `rows_per_alpha` rows)."""
    qb, sb, al = _u8(q), _u8(sf), _f32(alpha).reshape(-1)
    K = qb.shape[-1] * 2
    rows = qb.size // (K // 2)
    rpa = rows_per_alpha if rows_per_alpha is not None else rows // al.size
    out = np.empty((rows, K), np.float64)
    _check(_load().oracle_nvfp4_dequant(rows, K, _ptr(qb), _ptr(sb), _ptr(al), rpa, _ptr(out)),
           "oracle_nvfp4_dequant")
    return out


def moe_tokens_w4(hidden, ids, weights, w1, w2, dtype, tokens=None, activation=ACT_SILU,
                  act_noise=False, act_dtype=None):
    """fp64 fused MoE output with NVFP4 experts.  w1 = (q [E,R1,H/2], sf [E,R1,H/16], alpha [E])
    for the gate/up projection (R1 = 2F, or F for ReLU2), w2 = (q [E,H,F/2], sf [E,H,F/16],
    alpha [E]) for the down projection.  ``act_noise``: as in moe_tokens, for act rounded to
    ``act_dtype`` (default: ``dtype``)."""
    hb = _bits(hidden)
    T, H = hb.shape
    idv = _c(ids, np.int32)
    k = idv.shape[1]
    wv = _c(weights, np.float64)
    q1, s1, a1 = _u8(w1[0]), _u8(w1[1]), _f32(w1[2])
    q2, s2, a2 = _u8(w2[0]), _u8(w2[1]), _f32(w2[2])
    E, _, F2 = q2.shape
    F = F2 * 2
    if q1.shape != (E, gate_up_rows(activation, F), H // 2):
        raise ValueError("w1 does not match the activation and shapes")
    tl = np.arange(T, dtype=np.int32) if tokens is None else _c(tokens, np.int32)
    out = np.empty((tl.size, H), np.float64)
    noise = np.empty((tl.size, H), np.float64) if act_noise else None
    adt = dtype if act_dtype is None else act_dtype
    rc = _load().oracle_moe_tokens_w4(tl.size, _ptr(tl), T, H, E, F, k, dtype, adt, activation,
                                      _ptr(hb), _ptr(idv), _ptr(wv), _ptr(q1), _ptr(s1), _ptr(a1),
                                      _ptr(q2), _ptr(s2), _ptr(a2), _ptr(out), _ptr(noise))
    _check(rc, "oracle_moe_tokens_w4")
    return (out, noise) if act_noise else out


def expert_act_w4(x_rows, expert_of_row, w1, dtype, activation=ACT_SILU):
    xb = _bits(x_rows)
    n, H = xb.shape
    q1, s1, a1 = _u8(w1[0]), _u8(w1[1]), _f32(w1[2])
    F = q1.shape[1] if activation == ACT_RELU2 else q1.shape[1] // 2
    eo = _c(expert_of_row, np.int32)
    act = np.empty((n, F), np.float64)
    _check(_load().oracle_expert_act_w4(n, H, F, dtype, activation, _ptr(xb), _ptr(eo), _ptr(q1),
                                        _ptr(s1), _ptr(a1), _ptr(act)), "oracle_expert_act_w4")
    return act


def expert_down_w4(act_rows, expert_of_row, scale, w2, dtype):
    ab = _bits(act_rows)
    n, F = ab.shape
    q2, s2, a2 = _u8(w2[0]), _u8(w2[1]), _f32(w2[2])
    H = q2.shape[1]
    eo = _c(expert_of_row, np.int32)
    sc = _c(scale, np.float64)
    y = np.empty((n, H), np.float64)
    _check(_load().oracle_expert_down_w4(n, H, F, dtype, _ptr(ab), _ptr(eo), _ptr(sc), _ptr(q2),
                                         _ptr(s2), _ptr(a2), _ptr(y)), "oracle_expert_down_w4")
    return y


# --------------------------------------------------------------- grouped GEMM and post-permute
def grouped_gemm(a, b, meta, dtype, activation=0, max_m=0):
    """fp64 grouped GEMM (oracle.c: oracle_grouped_gemm).  Masked layout when max_m > 0
    (a [E, max_m, K], meta = valid rows per group), else contiguous (a [P, K], meta = inclusive
    prefix sums).  activation 1 = silu_and_mul (b [E, 2N, K]).  Returns out [rows, N]."""
    ab = _bits(a)
    K = ab.shape[-1]
    ab = ab.reshape(-1, K)
    bb = _bits(b)
    E = bb.shape[0]
    N = bb.shape[1] // (2 if activation else 1)
    mv = _c(meta, np.int32)
    out = np.empty((ab.shape[0], N), np.float64)
    _check(_load().oracle_grouped_gemm(E, N, K, int(max_m), ab.shape[0], dtype, activation,
                                       _ptr(ab), _ptr(bb), _ptr(mv), _ptr(out)),
           "oracle_grouped_gemm")
    return out


def post_permute(rows, weights, inv, top_k, dtype):
    """fp64 weighted combine out[t] = sum_j w[t,j] rows[inv[t*k+j]] (oracle_post_permute)."""
    rb = _bits(rows)
    H = rb.shape[1]
    wv = _c(weights, np.float64).reshape(-1)
    iv = _c(inv, np.int32).reshape(-1)
    T = iv.size // top_k
    out = np.empty((T, H), np.float64)
    _check(_load().oracle_post_permute(T, H, top_k, dtype, _ptr(rb), _ptr(wv), _ptr(iv),
                                       _ptr(out)), "oracle_post_permute")
    return out


def grouped_gemm_fp8(a, a_scale, b, b_scale, meta, max_m=0):
    """fp64 FP8 block-scaled grouped GEMM (oracle_grouped_gemm_fp8).  a [E, max_m, K] (masked,
    max_m > 0) or [P, K] E4M3 bytes, a_scale [.., K/128] f32, b [E, N, K] E4M3 bytes, b_scale
    [E, N/128, K/128] f32.  Returns out [rows, N]."""
    ab = _u8(a)
    K = ab.shape[-1]
    ab = ab.reshape(-1, K)
    asv = _f32(a_scale).reshape(ab.shape[0], -1)
    bb = _u8(b)
    E, N, _ = bb.shape
    bsv = _f32(b_scale)
    mv = _c(meta, np.int32)
    out = np.empty((ab.shape[0], N), np.float64)
    _check(_load().oracle_grouped_gemm_fp8(E, N, K, int(max_m), ab.shape[0], _ptr(ab),
                                           _ptr(asv), _ptr(bb), _ptr(bsv), _ptr(mv), _ptr(out)),
           "oracle_grouped_gemm_fp8")
    return out
