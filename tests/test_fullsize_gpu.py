"""Parity at the full sizes of the five workloads, in the launch configuration
the bench times (tcgen05 grouped GEMMs for bf16).

The float64 oracle cannot run the whole layer at these sizes, so:
  * routing, dispatch and the aux loss (integer or cheap) run in full: indices
    and the permutation must match bit for bit outside near ties; on near-tie
    tokens the GPU's choice must be a valid one, and the oracle then takes it,
    so that the whole dispatch matches bit for bit and the aux loss to 1e-5;
  * the row copy is checked in full on the device (x_perm == x[src_tok]);
  * outputs and gradients are checked on sampled tokens, each evaluated on its
    own by the oracle (a token's output needs only its own routing), and on
    sampled FFN columns of a few experts for the weight gradients (each column
    needs only that expert's rows);
  * the router weight gradient, a reduction over every token, is checked through
    the identity dW_r = d_logitsᵀ x (float64 on the device) plus the sampled
    d_logits rows against the oracle.
"""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as O
from tests.parity import (NEAR_TIE, TOL_AUX, TOL_F32, act_tol, assert_close,
                          gpu_choice_on_near_ties, record, routing_checks)

pytestmark = pytest.mark.gpu


class LazyExperts:
    """float64 copies of single experts' weights, made when first indexed."""

    def __init__(self, t):
        self.t = t
        self.cache = {}

    def __getitem__(self, e):
        e = int(e)
        if e not in self.cache:
            self.cache[e] = O.as_f64(self.t[e])
        return self.cache[e]


def _sample_tokens(T, counts, src_tok, offsets, ties):
    cand = [0, 1, T // 3, T // 2, T - 2, T - 1]
    order = np.argsort(-counts)
    for e in (order[0], order[len(order) // 2]):
        if counts[e] > 0:
            cand.append(int(src_tok[offsets[e]]))
            cand.append(int(src_tok[offsets[e + 1] - 1]))
    nz = np.nonzero(counts)[0]
    smallest = nz[np.argmin(counts[nz])]
    cand.append(int(src_tok[offsets[smallest]]))
    cand += [int(t) for t in ties[:2]]
    return sorted(set(t for t in cand if 0 <= t < T))


@pytest.mark.parametrize("name", list(mi.WORKLOADS))
def test_fullsize_parity(name):
    import routing_grouped_expert_gate_gb300 as moe
    from routing_grouped_expert_gate_gb300 import layer
    wl = mi.WORKLOADS[name]
    backward = wl.backward
    inp = mi.make_inputs(wl, seed=0, device="cuda", with_dy=backward)
    cfg = moe.cfg_from_workload(wl)
    p = layer.params_from_inputs(inp)
    b = layer.alloc_buffers(cfg, "cuda", backward=backward)
    layer.forward(cfg, p, inp["x"], b)
    if backward:
        layer.backward(cfg, p, inp["x"], inp["dy"], b)
    torch.cuda.synchronize()
    rc, detail = moe._lib.last_device_status()
    assert rc == 0, (rc, detail)
    tol = act_tol(wl)

    # ---- full routing, dispatch and aux loss in float64
    x64 = O.as_f64(inp["x"])
    ref = {"x": x64, "w_router": O.as_f64(inp["w_router"]),
           "logit_bias": O.as_f64(inp["logit_bias"]), "sel_bias": O.as_f64(inp["sel_bias"]),
           "w1": LazyExperts(inp["w1"]), "w2": LazyExperts(inp["w2"]),
           "w1_s": O.as_f64(inp["w1_s"]), "w2_s": O.as_f64(inp["w2_s"])}
    r0 = O.route(x64, ref["w_router"], wl.k, wl.score, wl.scaling, ref["logit_bias"],
                 ref["sel_bias"])
    f0 = dict(r0)
    f0.update(O.dispatch(r0["idx"], wl.E))
    report = {}
    assert_close("logits", b["logits"], r0["logits"], TOL_F32)
    assert float(np.max(np.abs(O.as_f64(b["logits"]) - r0["logits"]))) < 1e-6
    # indices and permutation bit-exact outside near ties; on near-tie tokens
    # the GPU's choice must be a valid one, and the oracle continues from it
    routing_checks(wl, b, f0, report)
    ties = np.nonzero(r0["gap"] < NEAR_TIE)[0]
    if ties.size:
        r = O.route(x64, ref["w_router"], wl.k, wl.score, wl.scaling, ref["logit_bias"],
                    ref["sel_bias"], idx=gpu_choice_on_near_ties(wl, b, f0))
    else:
        r = r0
    dsp = O.dispatch(r["idx"], wl.E)
    for key in ("counts", "offsets", "row_of", "src_tok"):
        got = b[key].cpu().numpy().astype(np.int64)
        assert np.array_equal(got, dsp[key]), f"{key} differs from the oracle's"
    assert_close("w", b["w"], r["w"], TOL_F32)
    aux = O.aux_loss(r["logits"], dsp["counts"], wl.k, wl.aux_coeff, wl.score)
    assert abs(float(b["aux"].item()) - aux) <= TOL_AUX * abs(aux)
    src_gpu = b["src_tok"].long()
    assert torch.equal(b["x_perm"], inp["x"][src_gpu])
    if wl.zipf_s:
        # the imbalance stress does what it is for (Handbook §3.3 "Cost of
        # imbalance"): the busiest expert takes over 10x the mean load and
        # at least one expert receives no token
        c = dsp["counts"]
        assert c.max() > 10 * c.mean() and int((c == 0).sum()) >= 1, (c.max(), c.mean())
    record(f"fullsize[{name}]", near_tie_tokens=int(ties.size),
           oracle_selection="GPU choice on near ties" if ties.size else "own",
           backward_compared=True)

    # ---- sampled tokens (near-tie tokens among them): outputs and gradients
    toks = _sample_tokens(wl.T, dsp["counts"], dsp["src_tok"], dsp["offsets"], ties)
    tf = O.tokens_forward(wl, ref, toks, routing=r)
    assert_close("y[sampled]", O.as_f64(b["y"][toks]), tf["y"], tol)
    if not backward:
        return
    dy64 = O.as_f64(inp["dy"][toks])
    tb = O.tokens_backward(wl, ref, toks, r, dsp["counts"], dy64)
    assert_close("dw[sampled]", O.as_f64(b["dw"][toks]), tb["dw"], tol)
    assert_close("d_logits[sampled]", O.as_f64(b["d_logits"][toks]), tb["d_logits"], tol)
    assert_close("dx[sampled]", O.as_f64(b["dx"][toks]), tb["dx"], tol)

    # ---- weight gradients on sampled FFN columns of three experts
    F = wl.F
    cols = sorted(set([0, 1, F // 2, F - 1]))
    order = np.argsort(-dsp["counts"])
    nz = [e for e in order if dsp["counts"][e] > 0]
    dy_full = inp["dy"]
    for e in (nz[0], nz[len(nz) // 2], nz[-1]):
        lo, hi = dsp["offsets"][e], dsp["offsets"][e + 1]
        rows_tok = dsp["src_tok"][lo:hi]
        wsel = np.array([r["w"][t, list(r["idx"][t]).index(e)] for t in rows_tok])
        d_out = wsel[:, None] * O.as_f64(dy_full[torch.from_numpy(rows_tok).cuda()])
        cg = O.expert_grad_columns(x64[rows_tok], d_out, ref["w1"][e], ref["w2"][e], cols)
        assert_close(f"dW2[{e}] cols", O.as_f64(b["dw2"][e][:, cols]), cg["dW2_cols"], tol)
        assert_close(f"dW1[{e}] gate rows", O.as_f64(b["dw1"][e][cols]), cg["dW1_gate"], tol)
        assert_close(f"dW1[{e}] up rows", O.as_f64(b["dw1"][e][[F + c for c in cols]]),
                     cg["dW1_up"], tol)
    empty = np.nonzero(dsp["counts"] == 0)[0]
    for e in empty[:4]:
        assert float(b["dw1"][e].abs().max()) == 0.0 and float(b["dw2"][e].abs().max()) == 0.0
    if wl.F_shared:
        Fs = wl.F_shared
        cs = sorted(set([0, Fs // 3, Fs - 1]))
        cg = O.expert_grad_columns(x64, O.as_f64(dy_full), ref["w1_s"], ref["w2_s"], cs)
        assert_close("dW2_s cols", O.as_f64(b["dw2_s"][0][:, cs]), cg["dW2_cols"], tol)
        assert_close("dW1_s gate rows", O.as_f64(b["dw1_s"][0][cs]), cg["dW1_gate"], tol)

    # ---- router weight gradient: identity over every token, in float64 on the device
    dwr = b["d_logits"].double().T @ inp["x"].double()
    assert_close("dW_r = d_logitsᵀ x", b["dw_router"], dwr.cpu().numpy(), TOL_F32)
