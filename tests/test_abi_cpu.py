"""Host-side checks of the C ABI: no GPU needed, no kernel launched.

The library must build, load, export every entry point include/moe.h declares,
and refuse bad configurations on the host, the way the Handbook says Megatron
validates them (§3.1 "Gating function": the expert bias is refused with
softmax; §3.1 "Output scale": top-1 softmax with renormalisation is refused).
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    from routing_grouped_expert_gate_gb300 import build
    build.build()
    from routing_grouped_expert_gate_gb300 import _lib
    return _lib


def _declared_symbols():
    with open(os.path.join(ROOT, "include", "moe.h")) as f:
        text = f.read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z0-9_]+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = _declared_symbols()
    assert len(names) >= 17
    lib = ctypes.CDLL(L.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    assert L.version().startswith("libmoe")


def _cfg(L, **kw):
    base = dict(T=64, d=64, E=8, k=2, F=64, F_shared=0, score="softmax", act_dtype="bf16")
    base.update(kw)
    return L.make_cfg(**base)


def test_workloads_validate(L):
    import moe_inputs as mi
    for wl in mi.WORKLOADS.values():
        cfg = L.cfg_from_workload(wl)
        assert L.check_cfg(cfg) == L.MOE_OK, wl.name
        for which in (L.MOE_WS_PERMUTE, L.MOE_WS_GROUPED, L.MOE_WS_GROUPED_BWD, L.MOE_WS_AUX,
                      L.MOE_WS_ROUTE_BWD):
            assert L.workspace_bytes(cfg, which) > 0


@pytest.mark.parametrize("kw,code", [
    (dict(k=1), "MOE_ERR_INVALID_ARG"),                     # top-1 softmax renormalised
    (dict(k=9, E=16), "MOE_ERR_UNSUPPORTED"),
    (dict(k=4, E=3), "MOE_ERR_INVALID_ARG"),                # k > E
    (dict(E=257, k=2), "MOE_ERR_UNSUPPORTED"),
    (dict(d=12), "MOE_ERR_ALIGN"),
    (dict(F=100), "MOE_ERR_ALIGN"),
    (dict(F_shared=20), "MOE_ERR_ALIGN"),
    (dict(T=-1), "MOE_ERR_INVALID_ARG"),
    (dict(d=0), "MOE_ERR_INVALID_ARG"),
])
def test_bad_configs_refused(L, kw, code):
    cfg = _cfg(L, **kw)
    assert L.check_cfg(cfg) == getattr(L, code)
    assert L.workspace_bytes(cfg, L.MOE_WS_PERMUTE) == 0


def test_top1_sigmoid_is_allowed(L):
    assert L.check_cfg(_cfg(L, k=1, score="sigmoid")) == L.MOE_OK


def test_selection_bias_with_softmax_refused_before_any_device_work(L):
    cfg = _cfg(L)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the call returns first
    rc = L.lib.moe_route_topk(ctypes.byref(cfg), fake, fake, None, fake, fake, fake, fake, None, 0,
                              None)
    assert rc == L.MOE_ERR_INVALID_ARG


def test_router_workspace_sizes_and_refusal(L):
    # tensor-core gate GEMM: three bf16 planes of W_r when x is bf16 and E % 64 == 0
    tc = _cfg(L, T=512, d=256, E=128, k=8, act_dtype="bf16")
    assert L.workspace_bytes(tc, L.MOE_WS_ROUTE) == 3 * 128 * 256 * 2
    for other in (_cfg(L, T=512, d=256, E=128, k=8, act_dtype="f32"),
                  _cfg(L, T=512, d=256, E=8, k=2, act_dtype="bf16"),
                  _cfg(L, T=512, d=256, E=96, k=8, act_dtype="bf16")):
        assert L.workspace_bytes(other, L.MOE_WS_ROUTE) == 0
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    rc = L.lib.moe_route_topk(ctypes.byref(tc), fake, fake, None, None, fake, fake, fake, fake,
                              100, None)
    assert rc == L.MOE_ERR_WORKSPACE
    assert L.lib.moe_set_router_fold(24) == L.MOE_ERR_INVALID_ARG
    assert L.lib.moe_set_router_impl(7) == L.MOE_ERR_INVALID_ARG


def test_null_and_misaligned_pointers_refused(L):
    cfg = _cfg(L)
    good = ctypes.c_void_p(0x10000)
    bad = ctypes.c_void_p(0x10008)
    rc = L.lib.moe_unpermute_combine(ctypes.byref(cfg), None, good, good, None, None, good, None)
    assert rc == L.MOE_ERR_INVALID_ARG
    rc = L.lib.moe_unpermute_combine(ctypes.byref(cfg), bad, good, good, None, None, good, None)
    assert rc == L.MOE_ERR_ALIGN
    rc = L.lib.moe_permute(ctypes.byref(cfg), good, good, good, good, good, good, good, good, 0,
                           None)
    assert rc == L.MOE_ERR_WORKSPACE


def test_status_strings_and_timeout_setter(L):
    for code in range(0, -9, -1):
        s = L.status_string(code)
        assert s and s != "unknown status"
    old = L.set_wait_timeout_ns(12345)
    assert L.set_wait_timeout_ns(old) == 12345


def test_cfg_struct_layout(L):
    # int64 T, seven int32, two floats, the activation (int32 + four floats): 64 bytes
    assert ctypes.sizeof(L.MoeCfg) == 64
    assert L.MoeCfg.scaling.offset == 36 and L.MoeCfg.aux_coeff.offset == 40


def test_activation_settings_validated(L):
    ok = [dict(act_fn="swiglu"), dict(act_fn="swiglu", glu_linear_offset=0.5),
          dict(act_fn="swiglu_clamp", act_clamp=10.0),
          dict(act_fn="situ_glu", act_gate_scale=4.0, act_linear_scale=25.0),
          dict(act_fn="situ_glu", act_gate_scale=4.0)]
    bad = [dict(act_fn="swiglu_clamp", act_clamp=0.0), dict(act_fn="swiglu_clamp", act_clamp=-1.0),
           dict(act_fn="swiglu_clamp", act_clamp=float("inf")),
           dict(act_fn="swiglu_clamp", act_clamp=10.0, glu_linear_offset=0.5),
           dict(act_fn="situ_glu", act_gate_scale=0.0),
           dict(act_fn="situ_glu", act_gate_scale=4.0, act_linear_scale=-1.0)]
    for kw in ok:
        assert L.check_cfg(_cfg(L, **kw)) == L.MOE_OK, kw
    for kw in bad:
        assert L.check_cfg(_cfg(L, **kw)) == L.MOE_ERR_INVALID_ARG, kw


def test_router_dx_placement_rules(L):
    """Few experts: the permute backward forms d_logits · W_r (the router
    backward may then skip dx_router); many experts: the router backward must
    write it and the permute backward refuses to form it. Refusals come
    before any device work."""
    few, many = _cfg(L, E=8, k=2), _cfg(L, E=64, k=8)
    assert L.router_dx_in_permute_bwd(few) and not L.router_dx_in_permute_bwd(many)
    fake = ctypes.c_void_p(0x10000)  # never dereferenced
    rc = L.lib.moe_permute_bwd(ctypes.byref(many), fake, fake, None, None, None, None, fake, fake,
                               fake, None)
    assert rc == L.MOE_ERR_UNSUPPORTED
    rc = L.lib.moe_permute_bwd(ctypes.byref(few), fake, fake, fake, None, None, None, fake, fake,
                               fake, None)
    assert rc == L.MOE_ERR_INVALID_ARG  # dx_router together with d_logits
    rc = L.lib.moe_permute_bwd(ctypes.byref(few), fake, fake, None, None, None, None, fake, None,
                               fake, None)
    assert rc == L.MOE_ERR_INVALID_ARG  # d_logits without w_router
    ws_need = L.workspace_bytes(many, L.MOE_WS_ROUTE_BWD)
    rc = L.lib.moe_route_topk_bwd(ctypes.byref(many), fake, fake, fake, fake, fake, fake, 1, None,
                                  fake, fake, ws_need, None)
    assert rc == L.MOE_ERR_INVALID_ARG
