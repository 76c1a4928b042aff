"""Seeded synthetic inputs for one token-choice MoE layer.

This module holds none of the layer's arithmetic. It only names the workloads
(their sizes, router type and storage dtype) and draws their random tensors:
the hidden states, the router and expert weights, the optional selection bias,
the optional per-expert logit skew and the upstream gradient. The CPU oracle
(``oracle/``) and the CUDA path (tests, bench) both consume exactly the bytes
drawn here, so the two sides never share any other code.

Distributions follow the workload statements: x ~ N(0, 1), every weight
(router included) ~ N(0, 0.02), dy ~ N(0, 1), selection bias ~ U(-0.1, 0.1),
and for the imbalance stress a per-expert logit offset log(w_r) with
w_r = r^-s / sum_r' r'^-s (Zipf exponent s = 1.2, rank r = expert index + 1).
Values are drawn in fp32 and rounded (round-to-nearest-even) to the workload's
activation dtype; the router weight and both biases stay fp32.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Sequence, Dict, Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_inputs", "shrink"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    T: int            # tokens in the micro-batch
    d: int            # hidden size
    E: int            # routed experts
    k: int            # experts chosen per token
    F: int            # routed expert FFN width
    F_shared: int     # shared expert FFN width, 0 = no shared expert
    score: str        # "softmax" (renormalised over the top-k), "sigmoid", "sqrtsoftplus" or "softmax_pre"
    act_dtype: str    # "f32" or "bf16"
    backward: bool    # whether the workload runs the backward pass
    sel_bias_range: float = 0.0   # >0: selection-only expert bias ~ U(-r, r)
    zipf_s: float = 0.0           # >0: logit skew log(Zipf(s) rank weight)
    scaling: float = 1.0          # routed scaling factor
    aux_coeff: float = 1e-3       # Switch load-balancing loss coefficient
    weight_std: float = 0.02
    # expert activation: "swiglu", "swiglu_clamp" (act_clamp > 0) or "situ_glu"
    # (act_gate_scale > 0, optional act_linear_scale); glu_linear_offset is
    # added to the linear half
    act_fn: str = "swiglu"
    act_clamp: float = 0.0
    act_gate_scale: float = 0.0
    act_linear_scale: float = 0.0
    glu_linear_offset: float = 0.0
    shared_gate: bool = False     # sigmoid gate on the shared expert's output

    @property
    def A(self) -> int:
        """Token-expert assignments, T*k."""
        return self.T * self.k

    @property
    def torch_act_dtype(self) -> torch.dtype:
        return torch.float32 if self.act_dtype == "f32" else torch.bfloat16

    def grouped_flops_fwd(self) -> float:
        """Algorithmic FLOPs of the routed + shared expert GEMMs, forward."""
        return 6.0 * self.A * self.d * self.F + 6.0 * self.T * self.d * self.F_shared

    def router_flops_fwd(self) -> float:
        return 2.0 * self.T * self.d * self.E


WORKLOADS: Dict[str, Workload] = {
    w.name: w
    for w in [
        Workload("tiny_fp32", T=256, d=64, E=8, k=2, F=128, F_shared=0,
                 score="softmax", act_dtype="f32", backward=False),
        Workload("mixtral_style", T=4096, d=4096, E=8, k=2, F=14336, F_shared=0,
                 score="softmax", act_dtype="bf16", backward=True),
        Workload("fine_grained_64e", T=8192, d=2048, E=64, k=8, F=1408, F_shared=1408,
                 score="softmax", act_dtype="bf16", backward=True),
        Workload("deepseek_v3_shaped", T=8192, d=7168, E=256, k=8, F=2048, F_shared=2048,
                 score="sigmoid", act_dtype="bf16", backward=False, sel_bias_range=0.1),
        Workload("zipf_imbalance", T=16384, d=2048, E=128, k=8, F=768, F_shared=0,
                 score="softmax", act_dtype="bf16", backward=True, zipf_s=1.2),
    ]
}


def shrink(w: Workload, **changes) -> Workload:
    """A smaller (or otherwise changed) copy of a workload, for parity tests."""
    name = changes.pop("name", w.name + "_small")
    return dataclasses.replace(w, name=name, **changes)


# Order of the independent per-tensor streams; a tensor's stream never
# depends on which other tensors a workload has.
_STREAMS = ["x", "w_router", "w1", "w2", "w1_s", "w2_s", "sel_bias", "dy", "w_gate_s"]


def _gen(seed: int, name: str, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1_000_003 + _STREAMS.index(name) * 7919 + 17)
    return g


def _normal(shape, std: float, g: torch.Generator, device, out_dtype) -> torch.Tensor:
    """N(0, std) drawn in fp32 in slabs along dim 0, rounded to out_dtype."""
    out = torch.empty(shape, dtype=out_dtype, device=device)
    rows = shape[0]
    per_row = 1
    for s in shape[1:]:
        per_row *= s
    slab = max(1, (1 << 26) // max(per_row, 1))
    for r0 in range(0, rows, slab):
        r1 = min(rows, r0 + slab)
        v = torch.randn((r1 - r0,) + tuple(shape[1:]), generator=g, device=device,
                        dtype=torch.float32)
        if std != 1.0:
            v.mul_(std)
        out[r0:r1].copy_(v)
    return out


def zipf_logit_offset(E: int, s: float) -> torch.Tensor:
    """log of the Zipf(s) weight of rank e+1 among E ranks, rounded to fp32."""
    z = sum((r ** -s) for r in range(1, E + 1))
    return torch.tensor([math.log((r ** -s) / z) for r in range(1, E + 1)],
                        dtype=torch.float64).to(torch.float32)


def make_inputs(w: Workload, seed: int = 0, device="cpu",
                with_dy: Optional[bool] = None,
                only: Optional[Sequence[str]] = None) -> Dict[str, Optional[torch.Tensor]]:
    """Draw every input tensor of the workload on `device`.

    Returns a dict with keys x [T,d], w_router [E,d] fp32, w1 [E,2F,d],
    w2 [E,d,F], w1_s [2F_s,d] / w2_s [d,F_s] (None without a shared expert),
    sel_bias [E] fp32 (or None), logit_bias [E] fp32 (or None), dy [T,d]
    (or None), w_gate_s [d] fp32 (the shared expert's gate weight, or None).
    Rows [0,F) of each w1[e] are the gate, rows [F,2F) the up part.
    `only` restricts the draw to the named tensors among x, w_router, w1, w2
    (the others come back None); every tensor has its own generator, so the
    values drawn do not depend on which others are drawn.
    """
    device = torch.device(device)
    act = w.torch_act_dtype
    std = w.weight_std
    out: Dict[str, Optional[torch.Tensor]] = {}

    def want(name):
        return only is None or name in only

    out["x"] = _normal((w.T, w.d), 1.0, _gen(seed, "x", device), device, act) if want("x") else None
    out["w_router"] = (_normal((w.E, w.d), std, _gen(seed, "w_router", device), device,
                               torch.float32) if want("w_router") else None)
    out["w1"] = (_normal((w.E, 2 * w.F, w.d), std, _gen(seed, "w1", device), device, act)
                 if want("w1") else None)
    out["w2"] = (_normal((w.E, w.d, w.F), std, _gen(seed, "w2", device), device, act)
                 if want("w2") else None)
    if w.F_shared > 0 and want("w1") and want("w2"):
        out["w1_s"] = _normal((2 * w.F_shared, w.d), std, _gen(seed, "w1_s", device),
                              device, act)
        out["w2_s"] = _normal((w.d, w.F_shared), std, _gen(seed, "w2_s", device),
                              device, act)
    else:
        out["w1_s"] = None
        out["w2_s"] = None
    # the shared expert's sigmoid gate weight [d], fp32 like the router's
    out["w_gate_s"] = (_normal((w.d,), std, _gen(seed, "w_gate_s", device), device,
                               torch.float32)
                       if w.F_shared > 0 and w.shared_gate and want("w1") else None)
    if w.sel_bias_range > 0:
        g = _gen(seed, "sel_bias", device)
        r = w.sel_bias_range
        out["sel_bias"] = (torch.rand((w.E,), generator=g, device=device,
                                      dtype=torch.float32) * (2 * r) - r)
    else:
        out["sel_bias"] = None
    out["logit_bias"] = zipf_logit_offset(w.E, w.zipf_s).to(device) if w.zipf_s > 0 else None
    if with_dy is None:
        with_dy = w.backward
    out["dy"] = (_normal((w.T, w.d), 1.0, _gen(seed, "dy", device), device, act)
                 if with_dy and only is None else None)
    return out
