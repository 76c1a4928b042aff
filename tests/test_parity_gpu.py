"""GPU parity: every stage of the layer, through the C ABI, against the oracle.

Sizes are small enough for the float64 oracle to finish in seconds yet span
several GEMM tiles with ragged tails (T, F and d not multiples of the tiles),
empty experts (E = 128/256 with few tokens, a Zipf-skewed router) and both
router types. Each bf16 workload also runs as fp32, where every float output
must agree to 1e-4.
"""
import dataclasses

import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as O
from tests.parity import (TOL_AUX, TOL_F32, act_tol, assert_close, gpu_choice_on_near_ties,
                          record, routing_checks, to_np)

pytestmark = pytest.mark.gpu

W = mi.WORKLOADS
SMALL = {
    "tiny_fp32": dataclasses.replace(W["tiny_fp32"], backward=True),
    "mixtral_small": mi.shrink(W["mixtral_style"], name="mixtral_small", T=300, d=256, F=320),
    "fine_grained_small": mi.shrink(W["fine_grained_64e"], name="fine_grained_small", T=517,
                                    d=320, F=192, F_shared=128),
    "deepseek_small": mi.shrink(W["deepseek_v3_shaped"], name="deepseek_small", T=256, d=512,
                                F=128, F_shared=192, backward=True),
    "zipf_small": mi.shrink(W["zipf_imbalance"], name="zipf_small", T=1024, d=192, F=136),
    # router variants (Handbook §3.1): sqrt(softplus) with the selection bias and a
    # routed scaling factor; pre-softmax at top-1 and at top-4 with a skewed router
    "sqrtsoftplus_small": mi.shrink(W["deepseek_v3_shaped"], name="sqrtsoftplus_small",
                                    score="sqrtsoftplus", T=384, d=256, E=64, k=6, F=96,
                                    F_shared=64, scaling=2.5, backward=True),
    "presoftmax_top1_small": mi.shrink(W["fine_grained_64e"], name="presoftmax_top1_small",
                                       score="softmax_pre", T=333, d=192, E=16, k=1, F=128,
                                       F_shared=0),
    "presoftmax_small": mi.shrink(W["zipf_imbalance"], name="presoftmax_small",
                                  score="softmax_pre", T=257, d=128, E=32, k=4, F=64),
    # expert activations (Handbook §3.4 "Activation") and the gated shared expert:
    # a clamp value that clips about a sixth of the gate inputs (a bf16 value, so
    # that the clip decisions on the stored bf16 pre-activations are unambiguous);
    # SiTU-GLU with scales inside the activations' range and a linear offset
    "clamp_small": mi.shrink(W["mixtral_style"], name="clamp_small", T=300, d=256, F=320,
                             act_fn="swiglu_clamp", act_clamp=0.3125),
    "situ_small": mi.shrink(W["fine_grained_64e"], name="situ_small", T=517, d=320, F=192,
                            F_shared=128, act_fn="situ_glu", act_gate_scale=0.25,
                            act_linear_scale=0.2, glu_linear_offset=0.1),
    "gated_shared_small": mi.shrink(W["fine_grained_64e"], name="gated_shared_small", T=517,
                                    d=320, F=192, F_shared=128, shared_gate=True),
    # d = 4096: fc2's data gradient applies the SwiGLU derivative in its
    # epilogue (at smaller d a separate pass does)
    "mixtral_d4096_small": mi.shrink(W["mixtral_style"], name="mixtral_d4096_small", T=320,
                                     d=4096, F=192),
    # F = 4096: fc2 forward and fc1 dgrad with K >= 4096, where CTA pairs run a
    # segment's last tile of <= 128 rows as an M = 128 tile
    "mixtral_f4096_small": mi.shrink(W["mixtral_style"], name="mixtral_f4096_small", T=160,
                                     d=256, F=4096),
    # d = 200: no multiple of the 64-wide K block or of the 32-column store box
    # (router, fc1 and the weight gradients read a zero-filled last K block; fc2
    # and the data gradients store a ragged last column box)
    "ragged_d_small": mi.shrink(W["deepseek_v3_shaped"], name="ragged_d_small", T=200, d=200,
                                E=64, k=6, F=96, F_shared=64, backward=True),
    # few experts with a gated shared expert, top-4, d = 1288 (a 1024-column
    # slice and a ragged 264-column one): the permute backward that forms
    # d_logits · W_r streams k + 1 row slices per token through its ring
    "few_shared_small": mi.shrink(W["mixtral_style"], name="few_shared_small", T=2999, d=1288,
                                  E=12, k=4, F=96, F_shared=64, shared_gate=True),
    # few experts with sigmoid scores and a selection bias, fwd + bwd: the
    # top-k in 16-lane groups, the per-token scores backward and the grouped
    # aux-loss partials on their sigmoid branches
    "sigmoid_few_small": mi.shrink(W["deepseek_v3_shaped"], name="sigmoid_few_small", T=321,
                                   d=256, E=12, k=3, F=96, F_shared=64, backward=True),
    "sqrtsoftplus_few_small": mi.shrink(W["deepseek_v3_shaped"], name="sqrtsoftplus_few_small",
                                        score="sqrtsoftplus", T=263, d=192, E=8, k=2, F=64,
                                        F_shared=0, backward=True),
}
# bf16 workloads run on the tcgen05 kernels (the default) and, as a cross-check,
# on the CUDA-core kernels; fp32 workloads run on the CUDA-core kernels.
CASES = ([(n, "native", "tcgen05") for n in SMALL if n != "tiny_fp32"]
         + [(n, "native", "tcgen05_1cta") for n in SMALL if n != "tiny_fp32"]
         + [(n, "native", "tcgen05_pairs") for n in SMALL if n != "tiny_fp32"]
         + [(n, "native", "cudacores") for n in SMALL]
         + [(n, "f32", "cudacores") for n in SMALL if n != "tiny_fp32"])


def _wl(name, dt):
    wl = SMALL[name]
    if dt == "f32":
        wl = dataclasses.replace(wl, act_dtype="f32", name=wl.name + "_f32")
    return wl


def run_gpu(wl, seed=0, backward=True, impl="tcgen05"):
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    from routing_grouped_expert_gate_gb300 import layer
    inp = mi.make_inputs(wl, seed=seed, device="cuda", with_dy=backward)
    cfg = moe.cfg_from_workload(wl)
    p = layer.params_from_inputs(inp)
    b = layer.alloc_buffers(cfg, "cuda", backward=backward)
    old = L.set_grouped_gemm_impl({"tcgen05": L.MOE_GEMM_AUTO,
                                   "tcgen05_1cta": L.MOE_GEMM_TC_SINGLE_CTA,
                                   "tcgen05_pairs": L.MOE_GEMM_TC_PAIRS,
                                   "cudacores": L.MOE_GEMM_CUDA_CORES}[impl])
    # the CUDA-core run also takes the router's gate GEMM off the tensor cores
    old_r = L.set_router_impl(L.MOE_ROUTER_CUDA_CORES if impl == "cudacores"
                              else L.MOE_ROUTER_AUTO)
    try:
        layer.forward(cfg, p, inp["x"], b)
        if backward:
            layer.backward(cfg, p, inp["x"], inp["dy"], b)
        torch.cuda.synchronize()
    finally:
        L.set_grouped_gemm_impl(old)
        L.set_router_impl(old_r)
    rc, detail = moe._lib.last_device_status()
    assert rc == 0, f"device status {rc} ({moe.status_string(rc)}) detail {detail}"
    return inp, b


@pytest.fixture(scope="module")
def built():
    from routing_grouped_expert_gate_gb300 import build
    build.build()
    import routing_grouped_expert_gate_gb300  # noqa: F401


def oracle_on_gpu_selection(wl, ref, b, report):
    """The oracle's forward and backward for the comparisons.

    Routing is checked first against the oracle's own selection (bit-exact
    outside near ties). Where near-tie tokens exist, the GPU's choice on them
    is checked to be a valid one and the oracle is re-run on it, so that
    every remaining output and gradient is compared in full; the number of
    near-tie tokens goes into the run's parity summary."""
    f0 = O.layer_forward(wl, ref)
    routing_checks(wl, b, f0, report)
    if report["near_tie_tokens"] == 0:
        f = f0
        report["oracle_selection"] = "own"
    else:
        f = O.layer_forward(wl, ref, idx=gpu_choice_on_near_ties(wl, b, f0))
        report["oracle_selection"] = "GPU choice on near ties"
    # with the same selection, the dispatch is identical everywhere
    for key in ("counts", "offsets", "row_of", "src_tok"):
        got = b[key].cpu().numpy().astype(np.int64)
        assert np.array_equal(got, f[key]), f"{key} differs from the oracle's"
    return f


@pytest.mark.parametrize("name,dt,impl", CASES)
def test_layer_parity(built, request, name, dt, impl):
    wl = _wl(name, dt)
    inp, b = run_gpu(wl, backward=True, impl=impl)
    ref = {k: O.as_f64(v) for k, v in inp.items()}
    report = {}
    f = oracle_on_gpu_selection(wl, ref, b, report)
    g = O.layer_backward(wl, ref, f, ref["dy"])
    tol = act_tol(wl)
    compared = []

    def check(name, gpu, want, t):
        assert_close(name, gpu, want, t)
        compared.append(name)

    # S1/S2: logits and weights are fp32 results of exact inputs
    check("logits", b["logits"], f["logits"], TOL_F32)
    assert float(np.max(np.abs(to_np(b["logits"]) - f["logits"]))) < 1e-6, \
        "logit error must stay far below the near-tie band"
    check("w", b["w"], f["w"], TOL_F32)

    # S3: the row copy is exact
    xp = to_np(b["x_perm"])
    assert np.array_equal(xp, f["x_perm"])
    compared.append("x_perm (exact)")

    # S4/S5
    F = wl.F
    pre = to_np(b["pre_gu"])
    check("gate", pre[:, :F], f["g"], tol)
    check("up", pre[:, F:], f["u"], tol)
    check("h", b["h"], f["h"], tol)
    check("out_perm", b["out_perm"], f["out_perm"], tol)
    if wl.F_shared:
        check("y_shared", b["y_s"], f["y_s"], tol)
    if inp.get("w_gate_s") is not None:
        check("shared gate", b["gate_s"], f["gate_s"], TOL_F32)
    # S6, S7
    check("y", b["y"], f["y"], tol)
    aux = float(b["aux"].item())
    assert abs(aux - f["aux"]) <= TOL_AUX * abs(f["aux"]), (aux, f["aux"])
    compared.append("aux")

    # backward (bf16 workloads: everything here is downstream of bf16 activations)
    check("d_out_perm", b["d_out_perm"], g["d_out_perm"], tol)
    check("dw", b["dw"], g["dw"], tol)
    check("d_pre", b["d_pre"], g["d_pre"], tol)
    check("dx_perm", b["dx_perm"], g["dx_perm"], tol)
    check("dW1", b["dw1"], g["dW1"], tol)
    check("dW2", b["dw2"], g["dW2"], tol)
    check("d_logits", b["d_logits"], g["d_logits"], tol)
    check("dW_r", b["dw_router"], g["dW_r"], tol)
    check("dx", b["dx"], g["dx"], tol)
    if wl.F_shared:
        check("dW1_s", b["dw1_s"][0], g["dW1_s"], tol)
        check("dW2_s", b["dw2_s"][0], g["dW2_s"], tol)
    if inp.get("w_gate_s") is not None:
        check("d shared-gate logit", b["d_gate_logit_s"], g["d_gate_logit_s"], tol)
        check("dW_gate_s", b["dw_gate_s"], g["dW_gate_s"], tol)
        check("dy_s", b["dy_s"], g["dy_s"], tol)
    # experts that received no rows get an exactly zero weight gradient
    empty = np.nonzero(f["counts"] == 0)[0]
    for e in empty:
        assert float(b["dw1"][e].abs().max()) == 0.0 and float(b["dw2"][e].abs().max()) == 0.0
    record(request.node.name, near_tie_tokens=report["near_tie_tokens"],
           oracle_selection=report["oracle_selection"], compared=len(compared),
           backward_compared=all(n in compared for n in ("dW1", "dW2", "d_logits", "dW_r", "dx")))


@pytest.mark.parametrize("name", ["mixtral_small", "zipf_small"])
@pytest.mark.parametrize("impl", ["tcgen05", "tcgen05_pairs"])
def test_grouped_bwd_minimal_workspace(built, request, name, impl):
    """The grouped backward with a minimal workspace: the SwiGLU derivative in fc2's
    data-gradient epilogue, and the weight gradients' expert tails zeroed in
    shared memory instead of read through per-expert tensor maps. Same
    oracle checks as the layer test."""
    from routing_grouped_expert_gate_gb300 import _lib as L
    import routing_grouped_expert_gate_gb300 as moe
    wl = SMALL[name]
    inp, b = run_gpu(wl, backward=True, impl=impl)
    cfg = moe.cfg_from_workload(wl)
    T, k, E, F = wl.T, wl.k, wl.E, wl.F
    out = {n: torch.full_like(b[n], float("nan")) for n in ("d_pre", "dx_perm", "dw1", "dw2")}
    small_ws = torch.empty(256, dtype=torch.uint8, device="cuda")  # room for neither
    old = L.set_grouped_gemm_impl(L.MOE_GEMM_TC_PAIRS if impl == "tcgen05_pairs"
                                  else L.MOE_GEMM_AUTO)
    try:
        L.grouped_swiglu_bwd(cfg, E, T * k, F, b["offsets"], b["x_perm"], inp["w1"], inp["w2"],
                             b["pre_gu"], b["h"], b["d_out_perm"], out["d_pre"], out["dx_perm"],
                             out["dw1"], out["dw2"], small_ws)
        torch.cuda.synchronize()
    finally:
        L.set_grouped_gemm_impl(old)
    assert L.last_device_status()[0] == 0
    ref = {kk: O.as_f64(v) for kk, v in inp.items()}
    report = {}
    f = oracle_on_gpu_selection(wl, ref, b, report)
    g = O.layer_backward(wl, ref, f, ref["dy"])
    tol = act_tol(wl)
    assert_close("d_pre", out["d_pre"], g["d_pre"], tol)
    assert_close("dx_perm", out["dx_perm"], g["dx_perm"], tol)
    assert_close("dW1", out["dw1"], g["dW1"], tol)
    assert_close("dW2", out["dw2"], g["dW2"], tol)
    record(request.node.name, near_tie_tokens=report["near_tie_tokens"],
           oracle_selection=report["oracle_selection"], compared=4, backward_compared=True)
    # dW2 (same inputs as in the layer run) does not depend on which way the
    # expert tails were cleared; dW1 follows d_pre, whose derivative here ran
    # on the fp32 accumulators instead of a bf16 dh
    assert torch.equal(out["dw2"], b["dw2"])


@pytest.mark.parametrize("name", ["fine_grained_small", "deepseek_small", "zipf_small"])
@pytest.mark.parametrize("fold_k", [16, 32, 64])
def test_router_gate_gemm_paths(built, name, fold_k):
    """The tensor-core gate GEMM (three bf16 planes of W_r, compensated folds
    every fold_k elements) and the CUDA-core one both keep every logit within
    1e-6 of the float64 oracle and select the oracle's experts."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = SMALL[name]
    inp = mi.make_inputs(wl, seed=3, device="cuda")
    cfg = moe.cfg_from_workload(wl)
    ref = {k: O.as_f64(v) for k, v in inp.items() if v is not None}
    r = O.route(ref["x"], ref["w_router"], wl.k, wl.score, wl.scaling, ref.get("logit_bias"),
                ref.get("sel_bias"))
    ws = torch.empty(max(L.workspace_bytes(cfg, L.MOE_WS_ROUTE), 256), dtype=torch.uint8,
                     device="cuda")
    old_f = L.set_router_fold(fold_k)
    try:
        for impl in (L.MOE_ROUTER_AUTO, L.MOE_ROUTER_CUDA_CORES):
            old = L.set_router_impl(impl)
            try:
                assert L.router_uses_tensor_cores(cfg) == (impl == L.MOE_ROUTER_AUTO)
                logits = torch.full((wl.T, wl.E), float("nan"), device="cuda")
                idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
                w = torch.empty(wl.T, wl.k, device="cuda")
                L.route_topk(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"),
                             inp.get("sel_bias"), logits, idx, w, ws)
                torch.cuda.synchronize()
            finally:
                L.set_router_impl(old)
            assert L.last_device_status()[0] == 0
            err = float(np.max(np.abs(to_np(logits) - r["logits"])))
            assert err < 1e-6, (impl, fold_k, err)
            decided = r["gap"] >= 1e-6
            assert np.array_equal(to_np(idx)[decided], r["idx"][decided])
            assert_close("w", to_np(w)[decided], r["w"][decided], TOL_F32)
    finally:
        L.set_router_fold(old_f)


@pytest.mark.parametrize("E,d", [(8, 4096), (8, 8704), (16, 4096), (16, 8704), (16, 2048),
                                 (8, 200), (12, 1032)])
def test_small_router_hidden_sizes(built, E, d):
    """The few-expert gate GEMM (E <= 16) on its forms: W_r resident in shared
    memory with one warp per token group (E·d·4 <= 160 KB, including hidden
    sizes that are no multiple of the lanes' 512-element stride), and, for
    larger W_r, CTAs that split d over their warps with one fp32 chunk per
    lane (d <= 8192) or 32-element chunks folded into compensated pairs; a
    ragged token count. Logits within 1e-6 of the float64 oracle, the
    oracle's experts selected."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = mi.shrink(W["mixtral_style"], name=f"router_e{E}_d{d}", T=37, d=d, E=E, F=64)
    inp = mi.make_inputs(wl, seed=5, device="cuda", with_dy=False)
    cfg = moe.cfg_from_workload(wl)
    ref = {k: O.as_f64(v) for k, v in inp.items() if v is not None}
    r = O.route(ref["x"], ref["w_router"], wl.k, wl.score, wl.scaling, ref.get("logit_bias"),
                ref.get("sel_bias"))
    ws = torch.empty(max(L.workspace_bytes(cfg, L.MOE_WS_ROUTE), 256), dtype=torch.uint8,
                     device="cuda")
    logits = torch.full((wl.T, wl.E), float("nan"), device="cuda")
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.k, device="cuda")
    L.route_topk(cfg, inp["x"], inp["w_router"], None, None, logits, idx, w, ws)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    err = float(np.max(np.abs(to_np(logits) - r["logits"])))
    assert err < 1e-6, err
    decided = r["gap"] >= 1e-6
    assert np.array_equal(to_np(idx)[decided], r["idx"][decided])


@pytest.mark.parametrize("E,d,T", [(8, 264, 9741), (16, 520, 5003), (3, 1024, 4865),
                                   (8, 4096, 1000)])
def test_streamed_router_many_blocks(built, E, d, T):
    """The few-expert gate GEMM with bf16 x streamed through the shared-memory
    ring: more token blocks than CTAs (each CTA walks several blocks and the
    ring wraps many times), a last 256-column slice that is partly past d, E
    below the lane layout's expert count, and a ragged last block. Logits
    within 1e-6 of the float64 oracle, the oracle's experts selected."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = mi.shrink(W["mixtral_style"], name=f"router_stream_e{E}_d{d}_t{T}", T=T, d=d, E=E,
                   k=min(2, E), F=64)
    inp = mi.make_inputs(wl, seed=17, device="cuda", with_dy=False)
    cfg = moe.cfg_from_workload(wl)
    ref = {k: O.as_f64(v) for k, v in inp.items() if v is not None}
    r = O.route(ref["x"], ref["w_router"], wl.k, wl.score, wl.scaling, ref.get("logit_bias"),
                ref.get("sel_bias"))
    ws = torch.empty(max(L.workspace_bytes(cfg, L.MOE_WS_ROUTE), 256), dtype=torch.uint8,
                     device="cuda")
    logits = torch.full((wl.T, wl.E), float("nan"), device="cuda")
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.k, device="cuda")
    L.route_topk(cfg, inp["x"], inp["w_router"], None, None, logits, idx, w, ws)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    err = float(np.max(np.abs(to_np(logits) - r["logits"])))
    assert err < 1e-6, err
    decided = r["gap"] >= 1e-6
    assert np.array_equal(to_np(idx)[decided], r["idx"][decided])


@pytest.mark.parametrize("E,d,T", [(64, 200, 333), (128, 456, 129), (256, 1032, 257)])
def test_router_gate_gemm_ragged_shapes(built, E, d, T):
    """The tensor-core gate GEMM where d is no multiple of the 64-wide K block
    (the last block's columns past d arrive as zeros) and T no multiple of
    the 128-token tile: logits within 1e-6 of the float64 oracle, the
    oracle's experts selected."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = mi.shrink(W["deepseek_v3_shaped"], name=f"router_tc_e{E}_d{d}_t{T}", T=T, d=d, E=E,
                   F=64, F_shared=0)
    inp = mi.make_inputs(wl, seed=11, device="cuda", with_dy=False)
    cfg = moe.cfg_from_workload(wl)
    assert L.router_uses_tensor_cores(cfg)
    ref = {k: O.as_f64(v) for k, v in inp.items() if v is not None}
    r = O.route(ref["x"], ref["w_router"], wl.k, wl.score, wl.scaling, ref.get("logit_bias"),
                ref.get("sel_bias"))
    ws = torch.empty(max(L.workspace_bytes(cfg, L.MOE_WS_ROUTE), 256), dtype=torch.uint8,
                     device="cuda")
    logits = torch.full((wl.T, wl.E), float("nan"), device="cuda")
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.k, device="cuda")
    L.route_topk(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), inp.get("sel_bias"),
                 logits, idx, w, ws)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    err = float(np.max(np.abs(to_np(logits) - r["logits"])))
    assert err < 1e-6, err
    decided = r["gap"] >= 1e-6
    assert np.array_equal(to_np(idx)[decided], r["idx"][decided])
    assert_close("w", to_np(w)[decided], r["w"][decided], TOL_F32)


@pytest.mark.parametrize("name", ["mixtral_small", "deepseek_small", "tiny_fp32"])
def test_layer_replays_from_cuda_graph(built, name):
    """Every call of the layer can be captured into a CUDA graph (no host
    synchronisation, no allocation, launch parameters fixed at the call): the
    forward and backward replayed from a graph write exactly what the same
    calls write on a stream, starting from buffers filled with NaN / -7."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import layer
    wl = SMALL[name]
    inp = mi.make_inputs(wl, seed=4, device="cuda", with_dy=True)
    cfg = moe.cfg_from_workload(wl)
    p = layer.params_from_inputs(inp)
    b = layer.alloc_buffers(cfg, "cuda", backward=True)

    def step():
        layer.forward(cfg, p, inp["x"], b)
        layer.backward(cfg, p, inp["x"], inp["dy"], b)

    def poison():
        for k, v in b.items():
            if k != "ws":
                v.fill_(float("nan") if v.is_floating_point() else -7)

    step()  # first calls: one-time function attributes and occupancy queries
    poison()
    step()
    torch.cuda.synchronize()
    ref = {k: v.clone() for k, v in b.items() if k != "ws"}
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step()
    poison()
    g.replay()
    torch.cuda.synchronize()
    assert moe._lib.last_device_status()[0] == 0
    for k, v in ref.items():
        got = b[k]
        same = (got == v) | (torch.isnan(got) & torch.isnan(v)) if v.is_floating_point() \
            else (got == v)
        assert bool(same.all()), k


def test_zero_load_experts_exist_in_skewed_case(built):
    wl = SMALL["zipf_small"]
    inp = mi.make_inputs(wl, seed=0)
    ref = {k: O.as_f64(v) for k, v in inp.items()}
    r = O.route(ref["x"], ref["w_router"], wl.k, wl.score, 1.0, ref["logit_bias"], None)
    counts = O.dispatch(r["idx"], wl.E)["counts"]
    assert (counts == 0).sum() >= 1 and counts.max() > 3 * counts.mean()


@pytest.mark.parametrize("impl", ["tcgen05", "tcgen05_1cta", "tcgen05_pairs", "cudacores"])
def test_deterministic_bytes(built, impl):
    wl = SMALL["fine_grained_small"]
    _, b1 = run_gpu(wl, backward=True, impl=impl)
    _, b2 = run_gpu(wl, backward=True, impl=impl)
    for key in ("logits", "idx", "w", "row_of", "x_perm", "pre_gu", "out_perm", "y", "aux",
                "d_pre", "dw1", "dw2", "dw_router", "dx"):
        assert torch.equal(b1[key], b2[key]), key


def test_mixture_example_through_gpu(built):
    """The 0.75/0.25 mixture (LeCompute, 'An expert transforms numbers inside
    the model') embedded in d = F = 8 and run through the fp32 path."""
    import json
    import os
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import layer
    with open(os.path.join(os.path.dirname(__file__), "golden", "mixture_075_025.json")) as fh:
        gold = json.load(fh)
    c = gold["construction"]
    d = F = 8
    dev = "cuda"
    x = torch.zeros(1, d, device=dev)
    x[0, :2] = torch.tensor(c["x"])
    wr = torch.zeros(2, d, device=dev)
    wr[:, :2] = torch.tensor(c["w_router"])
    w1 = torch.zeros(2, 2 * F, d, device=dev)
    w2 = torch.zeros(2, d, F, device=dev)
    for e in range(2):
        w1[e, 0, :2] = torch.tensor(c["w1"][e][0])      # gate row 0
        w1[e, F, :2] = torch.tensor(c["w1"][e][1])      # up row 0
        w2[e, :2, 0] = torch.tensor([r[0] for r in c["w2"][e]])
    cfg = moe.make_cfg(T=1, d=d, E=2, k=2, F=F, act_dtype="f32", aux_coeff=0.0)
    b = layer.alloc_buffers(cfg, dev, backward=False)
    layer.forward(cfg, {"w_router": wr, "w1": w1, "w2": w2}, x, b)
    torch.cuda.synchronize()
    np.testing.assert_allclose(b["w"].cpu().numpy()[0],
                               [gold["page_values"]["weight_A"], gold["page_values"]["weight_B"]],
                               atol=1e-7)
    np.testing.assert_allclose(b["y"].cpu().numpy()[0, :2], gold["expected_y"], atol=1e-6)


def test_zero_tokens(built):
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import layer
    wl = mi.shrink(SMALL["mixtral_small"], T=0)
    inp = mi.make_inputs(wl, device="cuda", with_dy=True)
    cfg = moe.cfg_from_workload(wl)
    p = layer.params_from_inputs(inp)
    b = layer.alloc_buffers(cfg, "cuda", backward=True)
    layer.forward(cfg, p, inp["x"], b)
    layer.backward(cfg, p, inp["x"], inp["dy"], b)
    torch.cuda.synchronize()
    assert int(b["offsets"].abs().sum()) == 0 and int(b["counts"].abs().sum()) == 0
    assert float(b["aux"].item()) == 0.0
    assert float(b["dw1"].abs().max()) == 0.0 and float(b["dw_router"].abs().max()) == 0.0


def test_out_of_range_index_is_reported_not_faulted(built):
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    T, d, E, k = 64, 64, 8, 2
    cfg = moe.make_cfg(T=T, d=d, E=E, k=k, F=64)
    dev = "cuda"
    x = torch.randn(T, d, device=dev).to(torch.bfloat16)
    idx = torch.stack([torch.arange(T) % E, (torch.arange(T) + 1) % E], 1).to(torch.int32).to(dev)
    idx[5, 1] = E  # one bad entry
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = torch.empty(T, k, dtype=torch.int32, device=dev)
    src = torch.zeros(T * k, dtype=torch.int32, device=dev)
    xp = torch.zeros(T * k, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(L.workspace_bytes(cfg, L.MOE_WS_PERMUTE), dtype=torch.uint8, device=dev)
    L.last_device_status()
    L.permute(cfg, x, idx, counts, offsets, row_of, src, xp, ws)
    rc, detail = L.last_device_status()
    assert rc == L.MOE_ERR_DEVICE_INDEX and detail == 5
    assert int(offsets[-1]) == T * k - 1  # the bad assignment was skipped
    assert int(row_of[5, 1]) == -1
    # the combine refuses the bad row instead of reading out of bounds
    y = torch.empty(T, d, dtype=torch.bfloat16, device=dev)
    w = torch.ones(T, k, device=dev)
    L.unpermute_combine(cfg, xp, row_of, w, None, y)
    rc, detail = L.last_device_status()
    assert rc == L.MOE_ERR_DEVICE_INDEX and detail == 5
    assert L.last_device_status()[0] == 0  # reading clears it


@pytest.mark.parametrize("E", [8, 32])
def test_repeated_expert_is_reported(built, E):
    """A token that names the same expert twice is recorded as a bad index
    (its repeat counts once, the other rows stay consistent); no fault."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    T, d, k = 64, 64, 2
    cfg = moe.make_cfg(T=T, d=d, E=E, k=k, F=64)
    dev = "cuda"
    x = torch.randn(T, d, device=dev).to(torch.bfloat16)
    idx = torch.stack([torch.arange(T) % E, (torch.arange(T) + 1) % E], 1).to(torch.int32).to(dev)
    idx[9, 1] = idx[9, 0]  # token 9 repeats its first expert
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    offsets = torch.empty(E + 1, dtype=torch.int32, device=dev)
    row_of = torch.empty(T, k, dtype=torch.int32, device=dev)
    src = torch.zeros(T * k, dtype=torch.int32, device=dev)
    xp = torch.zeros(T * k, d, dtype=torch.bfloat16, device=dev)
    ws = torch.empty(L.workspace_bytes(cfg, L.MOE_WS_PERMUTE), dtype=torch.uint8, device=dev)
    L.last_device_status()
    L.permute(cfg, x, idx, counts, offsets, row_of, src, xp, ws)
    rc, detail = L.last_device_status()
    assert rc == L.MOE_ERR_DEVICE_INDEX and detail == 9
    assert int(offsets[-1]) == T * k - 1  # the repeat counted once
    assert L.last_device_status()[0] == 0


def test_bounded_wait_reports_timeout(built):
    from routing_grouped_expert_gate_gb300 import _lib as L
    old = L.set_wait_timeout_ns(2_000_000)  # 2 ms
    try:
        L.last_device_status()
        L.selftest_wait_timeout()
        rc, detail = L.last_device_status()
        assert rc == L.MOE_ERR_TIMEOUT and detail == 1
        # the context is still usable afterwards
        assert float(torch.ones(4, device="cuda").sum()) == 4.0
    finally:
        L.set_wait_timeout_ns(old)


@pytest.mark.parametrize("name", ["mixtral_small", "deepseek_small", "zipf_small",
                                  "sqrtsoftplus_small", "presoftmax_small"])
def test_near_tie_count(built, name):
    """moe_route_near_ties counts the tokens whose k-th and (k+1)-th fp32
    selection keys differ by less than the band: it agrees with the float64
    keys computed from the same logits, up to tokens within a few fp32 ulps of
    the band's edge."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = SMALL[name]
    inp = mi.make_inputs(wl, seed=0, device="cuda", with_dy=False)
    cfg = moe.cfg_from_workload(wl)
    ws = torch.empty(max(L.workspace_bytes(cfg, L.MOE_WS_ROUTE), 256), dtype=torch.uint8,
                     device="cuda")
    logits = torch.empty(wl.T, wl.E, device="cuda")
    idx = torch.empty(wl.T, wl.k, dtype=torch.int32, device="cuda")
    w = torch.empty(wl.T, wl.k, device="cuda")
    L.route_topk(cfg, inp["x"], inp["w_router"], inp.get("logit_bias"), inp.get("sel_bias"),
                 logits, idx, w, ws)
    sb = inp.get("sel_bias")
    keys = O.selection_keys(to_np(logits), wl.score, None if sb is None else to_np(sb))
    srt = -np.sort(-keys, axis=1)
    gap = srt[:, wl.k - 1] - srt[:, wl.k]
    cnt = torch.full((1,), -5, dtype=torch.int32, device="cuda")
    margin = 2e-6
    for band in (0.0, 1e-6, 1e-3, 3e-2, 1e9):
        L.route_near_ties(cfg, logits, sb, band, cnt)
        n = int(cnt.item())
        lo = int((gap < band - margin).sum())
        hi = int((gap < band + margin).sum()) if band > 0 else 0
        assert lo <= n <= hi, (band, lo, n, hi)
    assert n == wl.T  # every token is a near tie for an unbounded band
    assert L.last_device_status()[0] == 0


@pytest.mark.parametrize("T,E,k", [(1, 8, 2), (127, 8, 2), (4096, 8, 2), (5000, 8, 1),
                                   (999, 12, 1), (32767, 16, 2), (40000, 8, 2), (3001, 12, 4),
                                   (2051, 64, 8), (20608, 256, 4), (16384, 128, 8),
                                   (33024, 256, 4)])
def test_permute_index_paths(built, T, E, k):
    """The dispatch on both of its index paths: per-block counts followed by a
    rank + copy kernel that turns them into base rows itself, while there are
    at most 16384 (128-token block, expert) cells (k = 1 to 8, E = 8 to 128),
    and beyond that (T = 20608 and 33024 at E = 256) separate count, scan,
    rank and copy launches. counts, offsets, row_of and src_tok bit-exact
    against the oracle's dispatch; every copied row equal to its token's row."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    d = 64
    # (top-1 softmax is refused, so k = 1 routes with sigmoid scores)
    cfg = moe.make_cfg(T=T, d=d, E=E, k=k, F=64, score="softmax" if k > 1 else "sigmoid")
    g = torch.Generator(device="cuda")
    g.manual_seed(T * 31 + E)
    # k distinct experts per token, skewed towards the low indices
    keys = torch.rand(T, E, generator=g, device="cuda") * torch.linspace(1.0, 0.2, E,
                                                                         device="cuda")
    idx = torch.topk(keys, k, dim=1).indices.to(torch.int32).contiguous()
    x = torch.randn(T, d, generator=g, device="cuda").to(torch.bfloat16)
    counts = torch.full((E,), -1, dtype=torch.int32, device="cuda")
    offsets = torch.full((E + 1,), -1, dtype=torch.int32, device="cuda")
    row_of = torch.full((T, k), -1, dtype=torch.int32, device="cuda")
    src = torch.full((T * k,), -1, dtype=torch.int32, device="cuda")
    xp = torch.zeros(T * k, d, dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(max(L.workspace_bytes(cfg, L.MOE_WS_PERMUTE), 256), dtype=torch.uint8,
                     device="cuda")
    L.permute(cfg, x, idx, counts, offsets, row_of, src, xp, ws)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    ref = O.dispatch(idx.cpu().numpy().astype(np.int64), E)
    for key, got in (("counts", counts), ("offsets", offsets), ("row_of", row_of),
                     ("src_tok", src)):
        assert np.array_equal(got.cpu().numpy().astype(np.int64), ref[key]), key
    assert torch.equal(xp, x[src.long()])


@pytest.mark.parametrize("name", ["mixtral_small", "presoftmax_top1_small", "tiny_fp32",
                                  "mixtral_d4096_small", "few_shared_small"])
def test_router_dx_formed_in_permute_bwd_is_bitwise_the_same(built, name):
    """Few experts: the permute backward forms d_logits · W_r itself (for
    bf16 rows streaming them through its shared-memory ring, W_r's columns in
    registers). Its dx equals, bit for bit, the dx of the other order of work
    (the router backward writing dx_router in fp32, the permute backward
    adding it), with and without a gated shared expert."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = SMALL[name]
    cfg = moe.cfg_from_workload(wl)
    assert L.router_dx_in_permute_bwd(cfg)
    inp, b = run_gpu(wl, backward=True)
    dx_fused = b["dx"].clone()
    # d_logits rebuilt as the layer builds it (aux part, then the scores part)
    # with the router backward now writing dx_router
    L.aux_loss_bwd(cfg, b["logits"], b["counts"], 1.0, b["d_logits"], 0)
    L.route_topk_bwd(cfg, inp["x"], inp["w_router"], b["logits"], b["idx"], b["dw"],
                     b["d_logits"], 1, b["dx_router"], b["dw_router"], b["ws"])
    dx2 = torch.empty_like(b["dx"])
    gated = wl.F_shared > 0 and wl.shared_gate
    L.permute_bwd(cfg, b["dx_perm"], b["row_of"], b["dx_router"],
                  b["dx_s"] if wl.F_shared > 0 else None, dx2,
                  d_gate_logit=b["d_gate_logit_s"] if gated else None,
                  w_gate=inp["w_gate_s"] if gated else None)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    assert torch.equal(dx2, dx_fused)


@pytest.mark.parametrize("name", ["deepseek_small", "fine_grained_small", "ragged_d_small",
                                  "mixtral_small", "zipf_small"])
def test_gathered_fc1_equals_explicit_permute(built, name):
    """fc1 reading its rows straight from x through src_tok (the dispatch copy
    fused into the operand load) computes what the explicit x_perm path
    computes, bit for bit: gate|up, h and fc2's output. The dispatch run
    without x_perm produces the same index outputs."""
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import _lib as L
    wl = SMALL[name]
    inp, b = run_gpu(wl, backward=False)
    cfg = moe.cfg_from_workload(wl)
    T, k, E, F = wl.T, wl.k, wl.E, wl.F
    # index outputs only
    idx_only = {n: torch.full_like(b[n], -3) for n in ("counts", "offsets", "row_of", "src_tok")}
    L.permute(cfg, None, b["idx"], idx_only["counts"], idx_only["offsets"], idx_only["row_of"],
              idx_only["src_tok"], None, b["ws"])
    pre = torch.full_like(b["pre_gu"], float("nan"))
    h = torch.full_like(b["h"], float("nan"))
    out = torch.full_like(b["out_perm"], float("nan"))
    L.grouped_swiglu_gather(cfg, E, T * k, F, b["offsets"], inp["x"], b["src_tok"], inp["w1"],
                            inp["w2"], pre, h, out)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    for n, v in idx_only.items():
        assert torch.equal(v, b[n]), n
    assert torch.equal(pre, b["pre_gu"])
    assert torch.equal(h, b["h"])
    assert torch.equal(out, b["out_perm"])
