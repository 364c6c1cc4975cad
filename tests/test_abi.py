"""The C-ABI library builds, loads and exports every declared symbol; host-side argument checks
(CPU only: none of these calls reaches the device)."""
import ctypes
import os
import re

import pytest

from mixture_experts_forward_moe_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = []
    inc = os.path.join(ROOT, "include")
    for fn in sorted(os.listdir(inc)):
        if not fn.endswith(".h"):
            continue
        text = open(os.path.join(inc, fn)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        for m in re.finditer(r"^[A-Za-z_][\w \*]*?\b(\w+)\s*\(", text, flags=re.M):
            if m.group(1) not in ("if", "while"):
                names.append(m.group(1))
    return names


def test_header_declares_the_binding_names():
    assert sorted(_declared_functions()) == sorted(B.EXPORTED)


def test_library_exports_every_declared_symbol():
    lib = ctypes.CDLL(B.library_path() if os.path.exists(B.library_path()) else B.lib()._name)
    for name in _declared_functions():
        assert hasattr(lib, name), name


def _prob(**kw):
    base = dict(T=32, H=256, E=16, F=128, top_k=4)
    base.update(kw)
    return B.make_problem(**base)


def test_workspace_size_and_capacity():
    L = B.lib()
    p = _prob()
    n = L.moe_workspace_size(ctypes.byref(p))
    assert n > 0 and n % 256 == 0
    assert L.moe_sorted_capacity(ctypes.byref(p), 1) == 32 * 4
    assert L.moe_sorted_capacity(ctypes.byref(p), 16) == 32 * 4 + 16 * 15
    assert L.moe_stage_workspace_size(ctypes.byref(p), 16) > n
    assert L.moe_stage_workspace_size(ctypes.byref(p), 1) == n


def _align256(n):
    return (n + 255) // 256 * 256


@pytest.mark.parametrize("kw", [
    dict(T=32, H=2048, E=128, F=768, top_k=8),                   # Qwen3-30B decode: 768 units
    dict(T=32, H=7168, E=256, F=2048, top_k=8, ep_num_local=32),  # EP8 shard: 32 local experts
    dict(T=7, H=256, E=16, F=384, top_k=2),                     # few routes: units from P
    dict(T=64, H=512, E=512, F=4096, top_k=8),                  # more than 1024 units: capped
])
def test_w4a16_workspace_adds_the_split_scratch(kw):
    """moe_workspace_size_w4a16 = moe_workspace_size + the split-K scratch its header defines:
    a counter per unit (256-byte aligned), then 2048 * round16(T) bytes per unit, for
    min(min(T*top_k, E_local) * F/128, 1024) units."""
    L = B.lib()
    p = _prob(**kw)
    base = L.moe_workspace_size(ctypes.byref(p))
    e_local = kw.get("ep_num_local", 0) or kw["E"]
    units = min(min(kw["T"] * kw["top_k"], e_local) * (kw["F"] // 128), 1024)
    scratch = _align256(4 * units) + units * 2048 * ((kw["T"] + 15) // 16 * 16)
    assert L.moe_workspace_size_w4a16(ctypes.byref(p)) == base + scratch


@pytest.mark.parametrize("kw", [dict(T=65), dict(T=512, H=256, E=16, F=128, top_k=4),
                                dict(T=0)])
def test_w4a16_workspace_has_no_scratch_past_64_tokens(kw):
    L = B.lib()
    p = _prob(**kw)
    assert L.moe_workspace_size_w4a16(ctypes.byref(p)) == L.moe_workspace_size(ctypes.byref(p))


@pytest.mark.parametrize("kw,code", [
    (dict(T=-1), B.MOE_ERR_INVALID_ARG),
    (dict(top_k=17), B.MOE_ERR_INVALID_ARG),          # top_k > E
    (dict(H=100), B.MOE_ERR_UNSUPPORTED),             # not a multiple of 8
    (dict(F=36), B.MOE_ERR_UNSUPPORTED),
    (dict(E=2048, top_k=4), B.MOE_ERR_UNSUPPORTED),   # E > 1024
    (dict(num_expert_group=3, topk_group=1, scoring_func="sigmoid"), B.MOE_ERR_INVALID_ARG),
    (dict(num_expert_group=4, topk_group=0, scoring_func="sigmoid"), B.MOE_ERR_INVALID_ARG),
    (dict(num_expert_group=8, topk_group=1, scoring_func="sigmoid", top_k=4),
     B.MOE_ERR_INVALID_ARG),                           # 1 group of 2 experts < top_k
    (dict(num_expert_group=4, topk_group=2, scoring_func="softmax"), B.MOE_ERR_UNSUPPORTED),
])
def test_invalid_problems_rejected_before_launch(kw, code):
    L = B.lib()
    p = _prob(**kw)
    assert L.moe_workspace_size(ctypes.byref(p)) == 0
    dummy = ctypes.c_void_p(16)
    rc = L.fused_moe_fwd(ctypes.byref(p), dummy, dummy, dummy, dummy, None, None, None, dummy,
                         dummy, 1 << 40, None)
    assert rc == code


def test_null_pointers_and_short_workspace_rejected():
    L = B.lib()
    p = _prob()
    d = ctypes.c_void_p(16)
    need = L.moe_workspace_size(ctypes.byref(p))
    assert L.fused_moe_fwd(ctypes.byref(p), None, d, d, d, None, None, None, d, d, need,
                           None) == B.MOE_ERR_INVALID_ARG
    assert L.fused_moe_fwd(ctypes.byref(p), d, d, d, d, None, None, None, d, None, need,
                           None) == B.MOE_ERR_INVALID_ARG
    assert L.fused_moe_fwd(ctypes.byref(p), d, d, d, d, None, None, None, d, d, need - 1,
                           None) == B.MOE_ERR_WORKSPACE_TOO_SMALL
    # shared weights must come as a pair and agree with S
    assert L.fused_moe_fwd(ctypes.byref(p), d, d, d, d, None, d, None, d, d, need,
                           None) == B.MOE_ERR_INVALID_ARG
    # correction bias only with sigmoid scoring
    assert L.fused_moe_fwd(ctypes.byref(p), d, d, d, d, d, None, None, d, d, need,
                           None) == B.MOE_ERR_UNSUPPORTED
    assert L.moe_align_sort(ctypes.byref(p), 0, d, d, d, d, None, d, d, need,
                            None) == B.MOE_ERR_INVALID_ARG
    assert L.moe_gemm1_swiglu(ctypes.byref(p), 1, d, d, d, d, d, d, 8, None) == \
        B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_shared_expert_fwd(ctypes.byref(p), d, d, d, d, d, need, None) == \
        B.MOE_ERR_INVALID_ARG  # S == 0


def test_status_strings():
    for code in range(B.MOE_ERR_F16_RANGE + 1):
        assert B.status_string(code) != "unknown status"
    assert B.status_string(99) == "unknown status"


def test_wait_limit_knob_round_trips():
    old = B.set_wait_limit_ns(12345)
    assert B.set_wait_limit_ns(old) == 12345


def test_host_entry_staging_and_argument_checks():
    """fused_moe_fwd_host: staging size, and argument errors returned before any copy or launch
    (the pointers here are never dereferenced)."""
    L = B.lib()
    p = _prob(T=32, H=256, E=16, F=128)
    stage = L.moe_host_staging_bytes(ctypes.byref(p))
    assert stage == 2 * _align256(32 * 256 * 2) + _align256(32 * 16 * 4)
    need = L.moe_workspace_size(ctypes.byref(p)) + stage
    h = ctypes.c_void_p(0x10000)
    d = ctypes.c_void_p(0x1000000)  # 256-byte aligned
    f = L.fused_moe_fwd_host
    assert f(ctypes.byref(p), None, h, d, d, None, None, None, h, d, need, None) == \
        B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(p), h, h, d, d, None, None, None, None, d, need, None) == \
        B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(p), h, h, None, d, None, None, None, h, d, need, None) == \
        B.MOE_ERR_INVALID_ARG
    assert f(ctypes.byref(p), h, h, d, d, None, None, None, h, d, need - 1, None) == \
        B.MOE_ERR_WORKSPACE_TOO_SMALL
    assert f(ctypes.byref(p), h, h, d, d, d, None, None, h, d, need, None) == \
        B.MOE_ERR_UNSUPPORTED  # correction bias with softmax scoring
    assert L.fused_moe_fwd_w4a16_host(ctypes.byref(p), h, h, d, None, d, d, None, h, d, need,
                                      None) == B.MOE_ERR_INVALID_ARG  # no alpha
    bad = _prob(T=32, H=256, E=16, F=128, top_k=0)
    assert L.moe_host_staging_bytes(ctypes.byref(bad)) == 0


@pytest.mark.parametrize("n_loc,off,code", [
    (32, 240, B.MOE_ERR_INVALID_ARG),   # the shard runs past the last expert
    (-1, 0, B.MOE_ERR_INVALID_ARG),
    (0, 8, B.MOE_ERR_INVALID_ARG),      # an offset without a shard
])
def test_combine_rejects_a_bad_shard_before_launch(n_loc, off, code):
    """moe_combine checks the problem (its expert-parallel fields choose the kernel) before it
    touches a pointer or the device."""
    p = B.make_problem(64, 256, 256, 8, 8, ep_num_local=n_loc, ep_local_offset=off)
    d = ctypes.c_void_p(16)
    assert B.lib().moe_combine(ctypes.byref(p), d, d, d, None, d, None) == code
