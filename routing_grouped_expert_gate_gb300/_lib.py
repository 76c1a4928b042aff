"""ctypes binding of libmoe (include/moe.h): argument marshalling only.

Every function here has the name of the C entry point without the ``moe_``
prefix, takes torch tensors (device memory from PyTorch) or None, checks that
they are contiguous and on the current device, and calls the C function on the
current torch stream. All arithmetic runs in the library's CUDA kernels; there
is no Python or CPU fallback: if libmoe.so is missing or fails to load, the
import raises.
"""
from __future__ import annotations

import ctypes
import os
from ctypes import POINTER, c_char_p, c_float, c_int, c_int32, c_int64, c_size_t, c_uint64, c_void_p
from typing import Optional

import torch

from . import build as _build

LIB_PATH = _build.LIB

MOE_OK = 0
MOE_ERR_INVALID_ARG = -1
MOE_ERR_UNSUPPORTED = -2
MOE_ERR_ALIGN = -3
MOE_ERR_CUDA = -4
MOE_ERR_TIMEOUT = -5
MOE_ERR_DEVICE_INDEX = -6
MOE_ERR_WORKSPACE = -7
MOE_ERR_NO_DEVICE = -8

MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID = 1
MOE_SCORE_SQRT_SOFTPLUS = 2
MOE_SCORE_SOFTMAX_PRE = 3
SCORE_CODES = {"softmax": MOE_SCORE_SOFTMAX, "sigmoid": MOE_SCORE_SIGMOID,
               "sqrtsoftplus": MOE_SCORE_SQRT_SOFTPLUS, "softmax_pre": MOE_SCORE_SOFTMAX_PRE}
MOE_F32 = 0
MOE_BF16 = 1

MOE_GEMM_AUTO = 0
MOE_GEMM_CUDA_CORES = 1
MOE_GEMM_TC_SINGLE_CTA = 2
MOE_GEMM_TC_PAIRS = 3

MOE_WS_PERMUTE = 0
MOE_WS_GROUPED = 1
MOE_WS_GROUPED_BWD = 2
MOE_WS_AUX = 3
MOE_WS_ROUTE_BWD = 4
MOE_WS_ROUTE = 5
MOE_WS_Z_LOSS = 6
MOE_WS_SHARED_GATE_BWD = 7

MOE_ROUTER_AUTO = 0
MOE_ROUTER_CUDA_CORES = 1


class MoeCfg(ctypes.Structure):
    _fields_ = [("T", c_int64), ("d", c_int32), ("E", c_int32), ("k", c_int32),
                ("F", c_int32), ("F_shared", c_int32), ("score_fn", c_int32),
                ("act_dtype", c_int32), ("scaling", c_float), ("aux_coeff", c_float),
                ("act_fn", c_int32), ("act_clamp", c_float), ("act_gate_scale", c_float),
                ("act_linear_scale", c_float), ("glu_linear_offset", c_float)]


class MoeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = f"{where}: {code} ({status_string(code)})"
        if code == MOE_ERR_CUDA:
            msg += f" [{lib.moe_last_cuda_error().decode()}]"
        super().__init__(msg)


def _load():
    if not _build.up_to_date():
        try:
            _build.build()
        except Exception as e:  # no toolkit, compile error: no library, no fallback
            raise ImportError(f"libmoe.so could not be built ({LIB_PATH}): {e}") from e
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libmoe.so is missing ({LIB_PATH})")
    return ctypes.CDLL(LIB_PATH)


lib = _load()

_VP = c_void_p
_SIGS = {
    "moe_check_cfg": (c_int, [POINTER(MoeCfg)]),
    "moe_route_topk": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, c_size_t,
                               _VP]),
    "moe_permute": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, c_size_t, _VP]),
    "moe_grouped_swiglu": (c_int, [POINTER(MoeCfg), c_int32, c_int64, c_int32, _VP, _VP, _VP,
                                   _VP, _VP, _VP, _VP, _VP, c_size_t, _VP]),
    "moe_grouped_swiglu_gather": (c_int, [POINTER(MoeCfg), c_int32, c_int64, c_int32, _VP, _VP,
                                          c_int64, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_unpermute_combine": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_shared_gate": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP]),
    "moe_shared_gate_bwd": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                    c_size_t, _VP]),
    "moe_aux_loss": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, c_size_t, _VP]),
    "moe_unpermute_combine_bwd": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_grouped_swiglu_bwd": (c_int, [POINTER(MoeCfg), c_int32, c_int64, c_int32, _VP, _VP,
                                       _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                       c_size_t, _VP]),
    "moe_aux_loss_bwd": (c_int, [POINTER(MoeCfg), _VP, _VP, c_float, _VP, c_int32, _VP]),
    "moe_route_topk_bwd": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, c_int32, _VP,
                                   _VP, _VP, c_size_t, _VP]),
    "moe_permute_bwd": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP,
                                _VP]),
    "moe_router_dx_in_permute_bwd": (c_int, [POINTER(MoeCfg)]),
    "moe_workspace_bytes": (c_size_t, [POINTER(MoeCfg), c_int]),
    "moe_status_string": (c_char_p, [c_int]),
    "moe_last_cuda_error": (c_char_p, []),
    "moe_last_device_status": (c_int, [_VP, POINTER(c_int32)]),
    "moe_set_wait_timeout_ns": (c_uint64, [c_uint64]),
    "moe_selftest_wait_timeout": (c_int, [_VP]),
    "moe_version": (c_char_p, []),
    "moe_launch_count": (c_uint64, []),
    "moe_set_grouped_gemm_impl": (c_int, [c_int]),
    "moe_set_router_impl": (c_int, [c_int]),
    "moe_gate_logits": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, c_size_t, _VP]),
    "moe_route_near_ties": (c_int, [POINTER(MoeCfg), _VP, _VP, c_float, _VP, _VP]),
    "moe_quantile_route": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "moe_quantile_accumulate": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP]),
    "moe_quantile_beta_update": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, c_float, _VP]),
    "moe_z_loss": (c_int, [POINTER(MoeCfg), _VP, c_float, _VP, _VP, c_size_t, _VP]),
    "moe_z_loss_bwd": (c_int, [POINTER(MoeCfg), _VP, c_float, c_float, _VP, c_int32, _VP]),
    "moe_seq_aux_workspace_bytes": (c_size_t, [POINTER(MoeCfg), c_int64]),
    "moe_seq_aux_loss": (c_int, [POINTER(MoeCfg), _VP, _VP, c_int64, c_int32, c_float, _VP, _VP,
                                 c_size_t, _VP]),
    "moe_seq_aux_loss_bwd": (c_int, [POINTER(MoeCfg), _VP, _VP, c_int64, c_int32, c_float,
                                     c_float, _VP, c_int32, _VP, c_size_t, _VP]),
    "moe_tokens_per_expert_accumulate": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP]),
    "moe_expert_bias_update": (c_int, [POINTER(MoeCfg), _VP, _VP, c_float, _VP]),
    "moe_max_vio": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP]),
    "moe_set_router_fold": (c_int, [c_int]),
    "moe_router_uses_tensor_cores": (c_int, [POINTER(MoeCfg)]),
    "moe_router_bwd_uses_tensor_cores": (c_int, [POINTER(MoeCfg)]),
    "moe_kernel_timing": (c_int, [c_int]),
    "moe_kernel_times": (c_int, [POINTER(c_float), POINTER(c_int32)]),
    "moe_permute_noalloc": (c_int, [POINTER(MoeCfg), _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
}
for _name, (_res, _args) in _SIGS.items():
    _f = getattr(lib, _name)
    _f.restype = _res
    _f.argtypes = _args


# ------------------------------------------------------------------ helpers

def status_string(code: int) -> str:
    return lib.moe_status_string(code).decode()


def launch_count() -> int:
    return int(lib.moe_launch_count())


def set_grouped_gemm_impl(impl: int) -> int:
    """MOE_GEMM_AUTO (bf16 on tcgen05) or MOE_GEMM_CUDA_CORES; returns the previous one."""
    rc = int(lib.moe_set_grouped_gemm_impl(impl))
    if rc < 0:
        raise MoeError(rc, "moe_set_grouped_gemm_impl")
    return rc


def set_router_impl(impl: int) -> int:
    """MOE_ROUTER_AUTO (tensor cores where eligible) or MOE_ROUTER_CUDA_CORES."""
    rc = int(lib.moe_set_router_impl(impl))
    if rc < 0:
        raise MoeError(rc, "moe_set_router_impl")
    return rc


def set_router_fold(fold_k: int) -> int:
    """K elements per compensated window of the tensor-core gate GEMM."""
    rc = int(lib.moe_set_router_fold(fold_k))
    if rc < 0:
        raise MoeError(rc, "moe_set_router_fold")
    return rc


def router_uses_tensor_cores(cfg) -> bool:
    return bool(lib.moe_router_uses_tensor_cores(ctypes.byref(cfg)))


def router_bwd_uses_tensor_cores(cfg) -> bool:
    return bool(lib.moe_router_bwd_uses_tensor_cores(ctypes.byref(cfg)))


KERNEL_KINDS = ["fc1_fwd", "fc2_fwd", "fc2_dgrad", "fc1_dgrad", "fc2_wgrad", "fc1_wgrad"]


def kernel_timing(enable: bool):
    _check(lib.moe_kernel_timing(1 if enable else 0), "moe_kernel_timing")


def kernel_times():
    """{kind: (total ms, launches)} of the tcgen05 grouped GEMM kernels recorded."""
    ms = (c_float * len(KERNEL_KINDS))()
    n = (c_int32 * len(KERNEL_KINDS))()
    _check(lib.moe_kernel_times(ms, n), "moe_kernel_times")
    return {k: (float(ms[i]), int(n[i])) for i, k in enumerate(KERNEL_KINDS)}


def version() -> str:
    return lib.moe_version().decode()


MOE_ACT_SWIGLU = 0
MOE_ACT_SWIGLU_CLAMP = 1
MOE_ACT_SITU_GLU = 2
ACT_CODES = {"swiglu": MOE_ACT_SWIGLU, "swiglu_clamp": MOE_ACT_SWIGLU_CLAMP,
             "situ_glu": MOE_ACT_SITU_GLU}


def make_cfg(T, d, E, k, F, F_shared=0, score="softmax", act_dtype="bf16", scaling=1.0,
             aux_coeff=1e-3, act_fn="swiglu", act_clamp=0.0, act_gate_scale=0.0,
             act_linear_scale=0.0, glu_linear_offset=0.0) -> MoeCfg:
    return MoeCfg(T=T, d=d, E=E, k=k, F=F, F_shared=F_shared,
                  score_fn=SCORE_CODES[score],
                  act_dtype=MOE_BF16 if act_dtype == "bf16" else MOE_F32,
                  scaling=scaling, aux_coeff=aux_coeff, act_fn=ACT_CODES[act_fn],
                  act_clamp=act_clamp, act_gate_scale=act_gate_scale,
                  act_linear_scale=act_linear_scale, glu_linear_offset=glu_linear_offset)


def cfg_from_workload(wl, T: Optional[int] = None) -> MoeCfg:
    return make_cfg(wl.T if T is None else T, wl.d, wl.E, wl.k, wl.F, wl.F_shared, wl.score,
                    wl.act_dtype, wl.scaling, wl.aux_coeff, wl.act_fn, wl.act_clamp,
                    wl.act_gate_scale, wl.act_linear_scale, wl.glu_linear_offset)


def _p(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("libmoe takes contiguous tensors")
    if t.device.type != "cuda":
        raise ValueError("libmoe takes device tensors")
    return t.data_ptr()


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(rc: int, where: str):
    if rc != MOE_OK:
        raise MoeError(rc, where)


def check_cfg(cfg: MoeCfg) -> int:
    return lib.moe_check_cfg(ctypes.byref(cfg))


def workspace_bytes(cfg: MoeCfg, which: int) -> int:
    return int(lib.moe_workspace_bytes(ctypes.byref(cfg), which))


def last_device_status(stream=None):
    detail = c_int32(0)
    rc = lib.moe_last_device_status(_stream(stream), ctypes.byref(detail))
    return rc, detail.value


def set_wait_timeout_ns(ns: int) -> int:
    return int(lib.moe_set_wait_timeout_ns(ns))


def selftest_wait_timeout(stream=None):
    _check(lib.moe_selftest_wait_timeout(_stream(stream)), "moe_selftest_wait_timeout")


# ------------------------------------------------------------------ entry points

def route_topk(cfg, x, w_router, logit_bias, sel_bias, logits, idx, w, ws=None, stream=None):
    _check(lib.moe_route_topk(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias),
                              _p(sel_bias), _p(logits), _p(idx), _p(w), _p(ws),
                              0 if ws is None else ws.numel() * ws.element_size(),
                              _stream(stream)),
           "moe_route_topk")


def permute(cfg, x, idx, counts, offsets, row_of, src_tok, x_perm, ws, stream=None):
    _check(lib.moe_permute(ctypes.byref(cfg), _p(x), _p(idx), _p(counts), _p(offsets),
                           _p(row_of), _p(src_tok), _p(x_perm), _p(ws),
                           0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "moe_permute")


def permute_noalloc(cfg, x, idx, counts, offsets, row_of, src_tok, x_perm, stream=None):
    """moe_permute without a workspace: scratch lives in a fixed device array."""
    _check(lib.moe_permute_noalloc(ctypes.byref(cfg), _p(x), _p(idx), _p(counts), _p(offsets),
                                   _p(row_of), _p(src_tok), _p(x_perm), _stream(stream)),
           "moe_permute_noalloc")


def grouped_swiglu_gather(cfg, n_groups, n_rows, F, offsets, x, src_rows, w1, w2, pre_gu, h, out,
                          stream=None):
    """grouped_swiglu on the rows x[src_rows[r]], gathered inside fc1's operand load."""
    _check(lib.moe_grouped_swiglu_gather(ctypes.byref(cfg), int(n_groups), int(n_rows), int(F),
                                         _p(offsets), _p(x), int(x.shape[0]), _p(src_rows),
                                         _p(w1), _p(w2), _p(pre_gu), _p(h), _p(out),
                                         _stream(stream)),
           "moe_grouped_swiglu_gather")


def grouped_swiglu(cfg, n_groups, n_rows, F, offsets, x_rows, w1, w2, pre_gu, h, out, ws,
                   stream=None):
    _check(lib.moe_grouped_swiglu(ctypes.byref(cfg), n_groups, n_rows, F, _p(offsets),
                                  _p(x_rows), _p(w1), _p(w2), _p(pre_gu), _p(h), _p(out), _p(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream(stream)),
           "moe_grouped_swiglu")


def unpermute_combine(cfg, out_perm, row_of, w, shared_out, y, stream=None, shared_gate=None):
    _check(lib.moe_unpermute_combine(ctypes.byref(cfg), _p(out_perm), _p(row_of), _p(w),
                                     _p(shared_out), _p(shared_gate), _p(y), _stream(stream)),
           "moe_unpermute_combine")


def shared_gate(cfg, x, w_gate, gate, stream=None):
    _check(lib.moe_shared_gate(ctypes.byref(cfg), _p(x), _p(w_gate), _p(gate), _stream(stream)),
           "moe_shared_gate")


def shared_gate_bwd(cfg, x, gate, dy, shared_out, dy_shared, d_gate_logit, dw_gate, ws,
                    stream=None):
    _check(lib.moe_shared_gate_bwd(ctypes.byref(cfg), _p(x), _p(gate), _p(dy), _p(shared_out),
                                   _p(dy_shared), _p(d_gate_logit), _p(dw_gate), _p(ws),
                                   _nbytes(ws), _stream(stream)), "moe_shared_gate_bwd")


def aux_loss(cfg, logits, counts, aux, ws, stream=None):
    _check(lib.moe_aux_loss(ctypes.byref(cfg), _p(logits), _p(counts), _p(aux), _p(ws),
                            0 if ws is None else ws.numel() * ws.element_size(), _stream(stream)),
           "moe_aux_loss")


def unpermute_combine_bwd(cfg, dy, out_perm, row_of, w, d_out_perm, dw, stream=None):
    _check(lib.moe_unpermute_combine_bwd(ctypes.byref(cfg), _p(dy), _p(out_perm), _p(row_of),
                                         _p(w), _p(d_out_perm), _p(dw), _stream(stream)),
           "moe_unpermute_combine_bwd")


def grouped_swiglu_bwd(cfg, n_groups, n_rows, F, offsets, x_rows, w1, w2, pre_gu, h, d_out,
                       d_pre, dx_rows, dw1, dw2, ws, stream=None):
    _check(lib.moe_grouped_swiglu_bwd(ctypes.byref(cfg), n_groups, n_rows, F, _p(offsets),
                                      _p(x_rows), _p(w1), _p(w2), _p(pre_gu), _p(h), _p(d_out),
                                      _p(d_pre), _p(dx_rows), _p(dw1), _p(dw2), _p(ws),
                                      0 if ws is None else ws.numel() * ws.element_size(),
                                      _stream(stream)),
           "moe_grouped_swiglu_bwd")


def aux_loss_bwd(cfg, logits, counts, g_aux, d_logits, accumulate, stream=None):
    _check(lib.moe_aux_loss_bwd(ctypes.byref(cfg), _p(logits), _p(counts), float(g_aux),
                                _p(d_logits), int(accumulate), _stream(stream)),
           "moe_aux_loss_bwd")


def _nbytes(ws):
    return 0 if ws is None else ws.numel() * ws.element_size()


def gate_logits(cfg, x, w_router, logit_bias, logits, ws=None, stream=None):
    _check(lib.moe_gate_logits(ctypes.byref(cfg), _p(x), _p(w_router), _p(logit_bias),
                               _p(logits), _p(ws), _nbytes(ws), _stream(stream)),
           "moe_gate_logits")


def route_near_ties(cfg, logits, sel_bias, band, count, stream=None):
    """count[0] (device int32) = tokens whose k-th and (k+1)-th keys differ by < band."""
    _check(lib.moe_route_near_ties(ctypes.byref(cfg), _p(logits), _p(sel_bias), float(band),
                                   _p(count), _stream(stream)),
           "moe_route_near_ties")


def quantile_route(cfg, logits, beta, idx, w, alpha, beta_local=None, stream=None):
    _check(lib.moe_quantile_route(ctypes.byref(cfg), _p(logits), _p(beta), _p(idx), _p(w),
                                  _p(alpha), _p(beta_local), _stream(stream)),
           "moe_quantile_route")


def quantile_accumulate(cfg, beta_local, accum, count, stream=None):
    _check(lib.moe_quantile_accumulate(ctypes.byref(cfg), _p(beta_local), _p(accum), _p(count),
                                       _stream(stream)), "moe_quantile_accumulate")


def quantile_beta_update(cfg, beta, accum, count, ema, stream=None):
    _check(lib.moe_quantile_beta_update(ctypes.byref(cfg), _p(beta), _p(accum), _p(count),
                                        float(ema), _stream(stream)), "moe_quantile_beta_update")


def z_loss(cfg, logits, coeff, z, ws, stream=None):
    _check(lib.moe_z_loss(ctypes.byref(cfg), _p(logits), float(coeff), _p(z), _p(ws),
                          _nbytes(ws), _stream(stream)), "moe_z_loss")


def z_loss_bwd(cfg, logits, coeff, g_z, d_logits, accumulate, stream=None):
    _check(lib.moe_z_loss_bwd(ctypes.byref(cfg), _p(logits), float(coeff), float(g_z),
                              _p(d_logits), int(accumulate), _stream(stream)), "moe_z_loss_bwd")


def seq_aux_workspace_bytes(cfg, seq_len) -> int:
    return int(lib.moe_seq_aux_workspace_bytes(ctypes.byref(cfg), int(seq_len)))


def seq_aux_loss(cfg, logits, idx, seq_len, seq_major, coeff, out, ws, stream=None):
    _check(lib.moe_seq_aux_loss(ctypes.byref(cfg), _p(logits), _p(idx), int(seq_len),
                                int(seq_major), float(coeff), _p(out), _p(ws), _nbytes(ws),
                                _stream(stream)), "moe_seq_aux_loss")


def seq_aux_loss_bwd(cfg, logits, idx, seq_len, seq_major, coeff, g, d_logits, accumulate, ws,
                     stream=None):
    _check(lib.moe_seq_aux_loss_bwd(ctypes.byref(cfg), _p(logits), _p(idx), int(seq_len),
                                    int(seq_major), float(coeff), float(g), _p(d_logits),
                                    int(accumulate), _p(ws), _nbytes(ws), _stream(stream)),
           "moe_seq_aux_loss_bwd")


def tokens_per_expert_accumulate(cfg, counts, tokens_per_expert, stream=None):
    _check(lib.moe_tokens_per_expert_accumulate(ctypes.byref(cfg), _p(counts),
                                                _p(tokens_per_expert), _stream(stream)),
           "moe_tokens_per_expert_accumulate")


def expert_bias_update(cfg, tokens_per_expert, expert_bias, rate, stream=None):
    _check(lib.moe_expert_bias_update(ctypes.byref(cfg), _p(tokens_per_expert), _p(expert_bias),
                                      float(rate), _stream(stream)), "moe_expert_bias_update")


def max_vio(cfg, tokens_per_expert, out, stream=None):
    _check(lib.moe_max_vio(ctypes.byref(cfg), _p(tokens_per_expert), _p(out), _stream(stream)),
           "moe_max_vio")


def route_topk_bwd(cfg, x, w_router, logits, idx, dw, d_logits, accumulate, dx_router,
                   dw_router, ws, stream=None):
    _check(lib.moe_route_topk_bwd(ctypes.byref(cfg), _p(x), _p(w_router), _p(logits), _p(idx),
                                  _p(dw), _p(d_logits), int(accumulate), _p(dx_router),
                                  _p(dw_router), _p(ws),
                                  0 if ws is None else ws.numel() * ws.element_size(),
                                  _stream(stream)),
           "moe_route_topk_bwd")


def permute_bwd(cfg, dx_perm, row_of, dx_router, dx_shared, dx, stream=None,
                d_gate_logit=None, w_gate=None, d_logits=None, w_router=None):
    _check(lib.moe_permute_bwd(ctypes.byref(cfg), _p(dx_perm), _p(row_of), _p(dx_router),
                               _p(dx_shared), _p(d_gate_logit), _p(w_gate), _p(d_logits),
                               _p(w_router), _p(dx), _stream(stream)),
           "moe_permute_bwd")


def router_dx_in_permute_bwd(cfg) -> bool:
    """Whether permute_bwd forms d_logits · W_r itself for cfg (then route_topk_bwd
    takes dx_router=None)."""
    rc = int(lib.moe_router_dx_in_permute_bwd(ctypes.byref(cfg)))
    _check(min(rc, 0), "moe_router_dx_in_permute_bwd")
    return rc == 1
