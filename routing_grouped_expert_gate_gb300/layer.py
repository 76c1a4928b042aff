"""One token-choice MoE layer, forward and backward, as a sequence of libmoe calls.

This module only allocates device buffers (through PyTorch) and issues the C
ABI calls in order on one stream; every step of the layer runs in libmoe's
CUDA kernels:

  forward : route_topk -> permute -> grouped_swiglu (routed) [-> grouped_swiglu
            (shared) [-> shared_gate]] -> unpermute_combine -> aux_loss
  backward: unpermute_combine_bwd -> grouped_swiglu_bwd (routed) [->
            [shared_gate_bwd ->] grouped_swiglu_bwd (shared)] -> aux_loss_bwd ->
            route_topk_bwd -> permute_bwd

The shared expert's sigmoid gate is used when the parameters hold its weight
("w_gate_s", [d] fp32).

The backward returns the gradients of  <dy, y> + g_aux * aux  with respect to
x, the router weight and the expert weights.
"""
from __future__ import annotations

from typing import Dict, Optional

import torch

from . import _lib as L


def _act(cfg) -> torch.dtype:
    return torch.bfloat16 if cfg.act_dtype == L.MOE_BF16 else torch.float32


def alloc_buffers(cfg, device, backward: bool = True, alloc=None) -> Dict[str, torch.Tensor]:
    """Every intermediate and output of one forward (+ backward), allocated once.

    `alloc(shape, dtype)`, when given, makes each buffer instead of
    torch.empty on `device` (a test places guard regions after every buffer
    this way)."""
    T, d, E, k, F, Fs = cfg.T, cfg.d, cfg.E, cfg.k, cfg.F, cfg.F_shared
    A = T * k
    act = _act(cfg)
    dev = torch.device(device)
    if alloc is None:
        alloc = lambda shape, dt: torch.empty(shape, dtype=dt, device=dev)  # noqa: E731
    e = lambda *s, dt=act: alloc(s, dt)  # noqa: E731
    b = {
        "logits": e(T, E, dt=torch.float32),
        "idx": e(T, k, dt=torch.int32),
        "w": e(T, k, dt=torch.float32),
        "counts": e(E, dt=torch.int32),
        "offsets": e(E + 1, dt=torch.int32),
        "row_of": e(T, k, dt=torch.int32),
        "src_tok": e(A, dt=torch.int32),
        "x_perm": e(A, d),
        "pre_gu": e(A, 2 * F),
        "h": e(A, F),
        "out_perm": e(A, d),
        "y": e(T, d),
        "aux": e(1, dt=torch.float32),
    }
    if Fs > 0:
        b.update({"pre_gu_s": e(T, 2 * Fs), "h_s": e(T, Fs), "y_s": e(T, d),
                  "gate_s": e(T, dt=torch.float32)})
    ws = max(L.workspace_bytes(cfg, L.MOE_WS_PERMUTE), L.workspace_bytes(cfg, L.MOE_WS_GROUPED),
             L.workspace_bytes(cfg, L.MOE_WS_AUX), L.workspace_bytes(cfg, L.MOE_WS_ROUTE))
    if backward:
        b.update({
            "d_out_perm": e(A, d),
            "dw": e(T, k, dt=torch.float32),
            "d_pre": e(A, 2 * F),
            "dx_perm": e(A, d),
            "dw1": e(E, 2 * F, d),
            "dw2": e(E, d, F),
            "d_logits": e(T, E, dt=torch.float32),
            "dx_router": e(T, d, dt=torch.float32),
            "dw_router": e(E, d, dt=torch.float32),
            "dx": e(T, d),
        })
        if Fs > 0:
            b.update({"d_pre_s": e(T, 2 * Fs), "dx_s": e(T, d), "dw1_s": e(1, 2 * Fs, d),
                      "dw2_s": e(1, d, Fs), "dy_s": e(T, d),
                      "d_gate_logit_s": e(T, dt=torch.float32),
                      "dw_gate_s": e(d, dt=torch.float32)})
        ws = max(ws, L.workspace_bytes(cfg, L.MOE_WS_GROUPED_BWD),
                 L.workspace_bytes(cfg, L.MOE_WS_ROUTE_BWD),
                 L.workspace_bytes(cfg, L.MOE_WS_SHARED_GATE_BWD))
    b["ws"] = alloc((max(ws, 256),), torch.uint8)
    return b


def forward(cfg, p: Dict[str, Optional[torch.Tensor]], x: torch.Tensor,
            b: Dict[str, torch.Tensor], stream=None) -> Dict[str, torch.Tensor]:
    """S1..S7. `p` holds w_router, w1, w2 and optionally w1_s, w2_s, logit_bias, sel_bias."""
    T, k, E, F, Fs = cfg.T, cfg.k, cfg.E, cfg.F, cfg.F_shared
    ws = b["ws"]
    L.route_topk(cfg, x, p["w_router"], p.get("logit_bias"), p.get("sel_bias"), b["logits"],
                 b["idx"], b["w"], ws, stream)
    L.permute(cfg, x, b["idx"], b["counts"], b["offsets"], b["row_of"], b["src_tok"],
              b["x_perm"], ws, stream)
    L.grouped_swiglu(cfg, E, T * k, F, b["offsets"], b["x_perm"], p["w1"], p["w2"], b["pre_gu"],
                     b["h"], b["out_perm"], ws, stream)
    y_s = None
    gate = None
    if Fs > 0:
        L.grouped_swiglu(cfg, 1, T, Fs, None, x, p["w1_s"], p["w2_s"], b["pre_gu_s"], b["h_s"],
                         b["y_s"], ws, stream)
        y_s = b["y_s"]
        if p.get("w_gate_s") is not None:
            L.shared_gate(cfg, x, p["w_gate_s"], b["gate_s"], stream)
            gate = b["gate_s"]
    L.unpermute_combine(cfg, b["out_perm"], b["row_of"], b["w"], y_s, b["y"], stream,
                        shared_gate=gate)
    L.aux_loss(cfg, b["logits"], b["counts"], b["aux"], ws, stream)
    return b


def backward(cfg, p: Dict[str, Optional[torch.Tensor]], x: torch.Tensor, dy: torch.Tensor,
             b: Dict[str, torch.Tensor], g_aux: float = 1.0, stream=None) -> Dict[str, torch.Tensor]:
    """B6, B5/B4 (routed and shared), B7, B2/B1/B3, B1 (permute)."""
    T, k, E, F, Fs = cfg.T, cfg.k, cfg.E, cfg.F, cfg.F_shared
    ws = b["ws"]
    L.unpermute_combine_bwd(cfg, dy, b["out_perm"], b["row_of"], b["w"], b["d_out_perm"], b["dw"],
                            stream)
    L.grouped_swiglu_bwd(cfg, E, T * k, F, b["offsets"], b["x_perm"], p["w1"], p["w2"],
                         b["pre_gu"], b["h"], b["d_out_perm"], b["d_pre"], b["dx_perm"], b["dw1"],
                         b["dw2"], ws, stream)
    dx_s = None
    gated = Fs > 0 and p.get("w_gate_s") is not None
    if Fs > 0:
        dy_s = dy
        if gated:
            L.shared_gate_bwd(cfg, x, b["gate_s"], dy, b["y_s"], b["dy_s"], b["d_gate_logit_s"],
                              b["dw_gate_s"], ws, stream)
            dy_s = b["dy_s"]
        L.grouped_swiglu_bwd(cfg, 1, T, Fs, None, x, p["w1_s"], p["w2_s"], b["pre_gu_s"],
                             b["h_s"], dy_s, b["d_pre_s"], b["dx_s"], b["dw1_s"], b["dw2_s"], ws,
                             stream)
        dx_s = b["dx_s"]
    L.aux_loss_bwd(cfg, b["logits"], b["counts"], g_aux, b["d_logits"], 0, stream)
    # few experts: the permute backward forms the router's input gradient
    # d_logits · W_r itself, so the router backward writes no dx_router
    fused = L.router_dx_in_permute_bwd(cfg)
    L.route_topk_bwd(cfg, x, p["w_router"], b["logits"], b["idx"], b["dw"], b["d_logits"], 1,
                     None if fused else b["dx_router"], b["dw_router"], ws, stream)
    L.permute_bwd(cfg, b["dx_perm"], b["row_of"], None if fused else b["dx_router"], dx_s,
                  b["dx"], stream,
                  d_gate_logit=b["d_gate_logit_s"] if gated else None,
                  w_gate=p["w_gate_s"] if gated else None,
                  d_logits=b["d_logits"] if fused else None,
                  w_router=p["w_router"] if fused else None)
    return b


def params_from_inputs(inp: Dict[str, Optional[torch.Tensor]]) -> Dict[str, Optional[torch.Tensor]]:
    """Shape the generator's tensors for the calls: the shared expert as one group."""
    p = {k: inp.get(k) for k in ("w_router", "w1", "w2", "logit_bias", "sel_bias")}
    if inp.get("w1_s") is not None:
        p["w1_s"] = inp["w1_s"].unsqueeze(0)
        p["w2_s"] = inp["w2_s"].unsqueeze(0)
        p["w_gate_s"] = inp.get("w_gate_s")
    return p
