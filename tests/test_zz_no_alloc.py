"""moe_permute_noalloc, the dispatch entry point that allocates nothing.

Some callers cannot allocate device memory themselves: their device memory
belongs to a host framework's pool, or they run where a cudaMalloc is not
allowed. They cannot hand moe_permute a workspace, so this entry point keeps
its scratch in a fixed device array inside the library. Its results must be
those of moe_permute, bit for bit (indices, counts and copied rows are exact
integer and byte work). The GPU test makes two calls in a row with different
routings and sizes, so the second call runs on the first call's leftovers in
the shared array. This file is collected last on purpose.
"""
import ctypes

import pytest
import torch


def _lib():
    from routing_grouped_expert_gate_gb300 import build
    build.build()
    from routing_grouped_expert_gate_gb300 import _lib as L
    return L


def _routing(T, E, k, gen):
    # k distinct experts per token, from random keys (an input, not the method)
    keys = torch.rand(T, E, generator=gen, device="cuda")
    return keys.argsort(dim=1)[:, :k].to(torch.int32).contiguous()


@pytest.mark.gpu
def test_noalloc_matches_permute_on_two_calls():
    L = _lib()
    gen = torch.Generator(device="cuda")
    gen.manual_seed(1234)
    for T, d, E, k, dt in [(1000, 256, 64, 8, "bf16"), (3000, 192, 128, 4, "f32")]:
        cfg = L.make_cfg(T=T, d=d, E=E, k=k, F=64, act_dtype=dt)
        tdt = torch.bfloat16 if dt == "bf16" else torch.float32
        x = torch.randn(T, d, generator=gen, device="cuda").to(tdt)
        idx = _routing(T, E, k, gen)
        outs = []
        for use_noalloc in (False, True):
            counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
            offsets = torch.full((E + 1,), -7, dtype=torch.int32, device="cuda")
            row_of = torch.full((T, k), -7, dtype=torch.int32, device="cuda")
            src = torch.full((T * k,), -7, dtype=torch.int32, device="cuda")
            xp = torch.full((T * k, d), -7.0, dtype=tdt, device="cuda")
            if use_noalloc:
                L.permute_noalloc(cfg, x, idx, counts, offsets, row_of, src, xp)
            else:
                ws = torch.empty(L.workspace_bytes(cfg, L.MOE_WS_PERMUTE), dtype=torch.uint8,
                                 device="cuda")
                L.permute(cfg, x, idx, counts, offsets, row_of, src, xp, ws)
            torch.cuda.synchronize()
            assert L.last_device_status()[0] == 0
            outs.append((counts, offsets, row_of, src, xp))
        for a, b in zip(outs[0], outs[1]):
            assert torch.equal(a, b)
        assert int(outs[1][1][-1]) == T * k


def test_noalloc_rejects_sizes_beyond_its_scratch():
    L = _lib()
    fake = ctypes.c_void_p(0x10000)  # never dereferenced: the size check comes first
    # ceil(T / 128) * E * 4 bytes must fit in the 1 MiB array: T = 131072 fits at E = 256
    ok = L.make_cfg(T=131072, d=64, E=256, k=8, F=64)
    too_big = L.make_cfg(T=131073, d=64, E=256, k=8, F=64)
    assert L.workspace_bytes(ok, L.MOE_WS_PERMUTE) <= 1 << 20
    rc = L.lib.moe_permute_noalloc(ctypes.byref(too_big), fake, fake, fake, fake, fake, fake,
                                   fake, None)
    assert rc == L.MOE_ERR_UNSUPPORTED
