"""Out-of-bounds writes: every buffer of one forward + backward, inputs
included, sits in front of a guard region filled with a byte pattern. After
the layer has run on ragged sizes (d = 200, token counts that are no multiple
of the 128-row tile, experts that receive no token) and on every form of the
grouped GEMM, each guard must hold its pattern and each input its values.
A memory sanitizer is not used here; this test is what checks the kernels'
store bounds instead.
"""
import dataclasses

import pytest
import torch

import moe_inputs as mi
from tests.test_parity_gpu import SMALL, _wl

pytestmark = pytest.mark.gpu

GUARD_BYTES = 8192
PATTERN = 0xA5


class Guarded:
    """An allocator for layer.alloc_buffers: each tensor is the head of a
    larger byte buffer whose tail (right after the tensor's last byte) holds
    PATTERN."""

    def __init__(self, device):
        self.device = device
        self.items = []

    def __call__(self, shape, dt):
        n = 1
        for s in shape:
            n *= int(s)
        nbytes = n * torch.empty((), dtype=dt).element_size()
        raw = torch.empty(nbytes + GUARD_BYTES, dtype=torch.uint8, device=self.device)
        raw[nbytes:].fill_(PATTERN)
        self.items.append((raw, nbytes))
        return raw[:nbytes].view(dt).view(tuple(shape))

    def copy_of(self, t):
        if t is None:
            return None
        g = self(t.shape, t.dtype)
        g.copy_(t)
        return g

    def intact(self):
        return [i for i, (raw, n) in enumerate(self.items)
                if not bool((raw[n:] == PATTERN).all())]


CASES = [("ragged_d_small", "native", "tcgen05"), ("ragged_d_small", "native", "tcgen05_1cta"),
         ("ragged_d_small", "native", "tcgen05_pairs"), ("ragged_d_small", "native", "cudacores"),
         ("ragged_d_small", "f32", "cudacores"),
         ("zipf_small", "native", "tcgen05"), ("zipf_small", "native", "tcgen05_pairs"),
         ("fine_grained_small", "native", "tcgen05"), ("fine_grained_small", "native",
                                                       "tcgen05_1cta"),
         ("mixtral_f4096_small", "native", "tcgen05"),
         ("mixtral_d4096_small", "native", "tcgen05"),
         ("presoftmax_top1_small", "native", "tcgen05"),
         ("gated_shared_small", "native", "tcgen05"), ("few_shared_small", "native", "tcgen05"),
         ("tiny_fp32", "native", "cudacores")]


@pytest.mark.parametrize("name,dt,impl", CASES)
def test_no_write_past_any_buffer(name, dt, impl):
    from routing_grouped_expert_gate_gb300 import build
    build.build()
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    from routing_grouped_expert_gate_gb300 import layer
    wl = SMALL[name] if dt == "native" else _wl(name, dt)
    if name == "tiny_fp32":
        wl = dataclasses.replace(wl, backward=True)
    src = mi.make_inputs(wl, seed=1, device="cuda", with_dy=True)
    g = Guarded("cuda")
    inp = {k: g.copy_of(v) for k, v in src.items()}
    cfg = moe.cfg_from_workload(wl)
    p = layer.params_from_inputs(inp)
    b = layer.alloc_buffers(cfg, "cuda", backward=True, alloc=g)
    for k, v in b.items():  # outputs start as NaN / -7 so that nothing relies on zeros
        if k != "ws":
            v.fill_(float("nan") if v.is_floating_point() else -7)
    old = L.set_grouped_gemm_impl({"tcgen05": L.MOE_GEMM_AUTO,
                                   "tcgen05_1cta": L.MOE_GEMM_TC_SINGLE_CTA,
                                   "tcgen05_pairs": L.MOE_GEMM_TC_PAIRS,
                                   "cudacores": L.MOE_GEMM_CUDA_CORES}[impl])
    old_r = L.set_router_impl(L.MOE_ROUTER_CUDA_CORES if impl == "cudacores"
                              else L.MOE_ROUTER_AUTO)
    try:
        layer.forward(cfg, p, inp["x"], b)
        layer.backward(cfg, p, inp["x"], inp["dy"], b)
        torch.cuda.synchronize()
    finally:
        L.set_grouped_gemm_impl(old)
        L.set_router_impl(old_r)
    assert L.last_device_status()[0] == 0
    bad = g.intact()
    assert not bad, f"guard regions overwritten after buffers {bad} of {len(g.items)}"
    for k, v in src.items():
        if v is not None:
            assert torch.equal(inp[k], v), f"input {k} was modified"
