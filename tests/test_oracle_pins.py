"""Pins of the CPU oracle to facts fixed by the pages and by mathematics.

Each test would fail on a plausible mistake in the oracle: a gate/up swap, a
wrong tie rule, a dropped or mis-signed gradient term, a wrong aux-loss
normalisation, an unstable permutation. None of them runs the CUDA path.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _tiny(score="softmax", E=4, k=2, F=6, d=8, T=16, F_shared=0, sel=0.0, zipf=0.0,
          scaling=1.0, coeff=1e-2, seed=0, **act):
    wl = mi.Workload("pin", T=T, d=d, E=E, k=k, F=F, F_shared=F_shared, score=score,
                     act_dtype="f32", backward=True, sel_bias_range=sel, zipf_s=zipf,
                     scaling=scaling, aux_coeff=coeff, weight_std=0.5, **act)
    inp = {kk: O.as_f64(v) for kk, v in mi.make_inputs(wl, seed=seed).items()}
    return wl, inp


# ---------------------------------------------------------------- worked examples

def test_mixture_example_075_025():
    g = _load("mixture_075_025.json")
    c = g["construction"]
    x = np.array([c["x"]])
    w_router = np.array(c["w_router"])
    r = O.route(x, w_router, k=2, score="softmax")
    # the page's weights, exactly
    assert r["idx"][0].tolist() == [0, 1]
    np.testing.assert_allclose(r["w"][0], [g["page_values"]["weight_A"],
                                           g["page_values"]["weight_B"]], rtol=0, atol=1e-15)
    w1 = np.array(c["w1"])
    w2 = np.array(c["w2"])
    np.testing.assert_allclose(O.swiglu_ffn(x, w1[0], w2[0])["out"][0], c["out_A"], atol=1e-12)
    np.testing.assert_allclose(O.swiglu_ffn(x, w1[1], w2[1])["out"][0], c["out_B"], atol=1e-12)
    wl = mi.Workload("mix", T=1, d=2, E=2, k=2, F=1, F_shared=0, score="softmax",
                     act_dtype="f32", backward=False)
    f = O.layer_forward(wl, {"x": x, "w_router": w_router, "w1": w1, "w2": w2})
    np.testing.assert_allclose(f["y"][0], g["expected_y"], rtol=0, atol=1e-12)


def _four_gpu_idx(T):
    # tokens 0..3071 pick expert 0 first, then 1, 2 or 3 (1024 tokens each);
    # tokens 3072..3583 pick {4, 5}, tokens 3584..4095 pick {6, 7}
    idx = np.zeros((T, 2), dtype=np.int64)
    for t in range(T):
        if t < 3072:
            idx[t] = [0, 1 + t // 1024]
        elif t < 3584:
            idx[t] = [4, 5]
        else:
            idx[t] = [6, 7]
    return idx


def test_four_gpu_scenario_counts_and_maxvio():
    g = _load("four_gpu_loads.json")
    idx = _four_gpu_idx(g["T"])
    dsp = O.dispatch(idx, g["E"])
    assert dsp["counts"].tolist() == g["expert_loads"]
    assert int(dsp["counts"].sum()) == g["assignments"] == g["T"] * g["k"]
    per_gpu = dsp["counts"].reshape(-1, g["experts_per_gpu"]).sum(axis=1)
    assert per_gpu.tolist() == g["device_totals"]
    assert O.max_vio(dsp["counts"]) == g["max_vio"]
    assert int(dsp["offsets"][-1]) * g["hidden"] * g["bytes_per_value"] == g["permuted_bytes"]


def test_max_vio_all_on_one_expert():
    g = _load("handbook_counts.json")["max_vio_all_on_one"]
    T = 512
    # every token picks experts 0..7: expert 0 (the busiest) receives every token
    idx = np.tile(np.arange(g["k"]), (T, 1))
    counts = O.dispatch(idx, g["E"])["counts"]
    assert counts[0] == T
    assert O.max_vio(counts) == g["max_vio"]


def test_parameter_count_matches_weight_layout():
    g = _load("handbook_counts.json")["parameter_count"]
    d, F = g["hidden"], g["expert_width"]
    wl = mi.Workload("pc", T=1, d=d, E=1, k=1, F=F, F_shared=0, score="softmax",
                     act_dtype="f32", backward=False)
    w1 = np.zeros((2 * wl.F, wl.d))
    w2 = np.zeros((wl.d, wl.F))
    out = O.swiglu_ffn(np.zeros((1, d)), w1, w2)
    assert out["out"].shape == (1, d) and out["h"].shape == (1, F)
    assert w1.size + w2.size == g["per_expert"]
    assert g["experts_chosen"] * g["per_expert"] == g["chosen_total"] == 3 * d * g["dense_width"]


# ---------------------------------------------------------------- top-k

def _brute_topk(keys_row, k):
    """The sorted top-k by definition: among all k-subsets, the one whose every
    member outranks every non-member; members listed by descending key. Rank is
    (fp32 key descending, then index ascending)."""
    E = len(keys_row)
    key32 = keys_row.astype(np.float32)

    def outranks(a, b):
        return key32[a] > key32[b] or (key32[a] == key32[b] and a < b)

    found = []
    n_subsets = 0
    for S in itertools.combinations(range(E), k):
        n_subsets += 1
        rest = [e for e in range(E) if e not in S]
        if all(outranks(a, b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    members = list(found[0])
    # order members: a precedes b iff a outranks b
    ordered = sorted(members, key=lambda e: sum(outranks(o, e) for o in members))
    return ordered, n_subsets


def test_subset_enumerator_counts():
    g = _load("handbook_counts.json")["subset_counts"]
    assert sum(1 for _ in itertools.combinations(range(32), 4)) == g["choose_4_of_32"]
    assert sum(1 for _ in itertools.combinations(range(31), 3)) == g["choose_3_of_31"]
    _, n = _brute_topk(np.arange(10, dtype=np.float64), 4)
    assert n == math.comb(10, 4)


@pytest.mark.parametrize("E,k", [(4, 1), (5, 2), (8, 2), (8, 3), (10, 4), (6, 6)])
def test_topk_matches_brute_force_with_ties(E, k):
    rng = np.random.default_rng(E * 10 + k)
    for trial in range(40):
        if trial % 2:
            keys = rng.integers(0, 4, size=(1, E)).astype(np.float64)  # many exact ties
        else:
            keys = rng.standard_normal((1, E))
        got = O.topk_sorted(keys, k)[0].tolist()
        want, _ = _brute_topk(keys[0], k)
        assert got == want, (keys, got, want)


def test_kth_gap_definition():
    keys = np.array([[0.5, 2.0, 1.0, 1.0 + 5e-7]])
    assert O.kth_gap(keys, 2)[0] == pytest.approx((1.0 + 5e-7) - 1.0, abs=1e-15)
    assert O.kth_gap(keys, 4)[0] == np.inf


# ---------------------------------------------------------------- weights

def test_softmax_weights_are_renormalised_softmax_of_full_distribution():
    rng = np.random.default_rng(1)
    logits = rng.standard_normal((50, 12)) * 2
    idx = O.topk_sorted(logits, 3)
    w = O.mixing_weights(logits, idx, "softmax", 1.0)
    full = np.exp(logits) / np.exp(logits).sum(axis=1, keepdims=True)
    chosen = np.take_along_axis(full, idx, axis=1)
    np.testing.assert_allclose(w, chosen / chosen.sum(axis=1, keepdims=True), rtol=1e-13)
    np.testing.assert_allclose(w.sum(axis=1), 1.0, rtol=1e-14)
    # weights follow the sorted order
    assert np.all(np.diff(w, axis=1) <= 1e-15)


def test_sigmoid_weights_sum_to_scaling_and_shared_share():
    g = _load("handbook_counts.json")["shared_share"]
    rng = np.random.default_rng(2)
    logits = rng.standard_normal((40, 16))
    idx = O.topk_sorted(O.sigmoid(logits), 8)
    w = O.mixing_weights(logits, idx, "sigmoid", g["scaling"])
    np.testing.assert_allclose(w.sum(axis=1), g["scaling"], rtol=1e-14)
    share = 1.0 / (1.0 + w.sum(axis=1))
    assert np.all(np.round(100 * share) == g["share_percent_rounded"])


def test_softmax_top1_weight_is_one_and_router_gets_no_gradient():
    wl, inp = _tiny(k=1, coeff=0.0)
    f = O.layer_forward(wl, inp)
    np.testing.assert_allclose(f["w"], 1.0, rtol=0, atol=0)
    b = O.layer_backward(wl, inp, f, inp["dy"], g_aux=0.0)
    assert np.all(b["d_logits"] == 0.0) and np.all(b["dW_r"] == 0.0)


def test_selection_bias_changes_selection_only():
    wl, inp = _tiny(score="sigmoid", E=8, k=3, sel=0.3, T=64)
    r_b = O.route(inp["x"], inp["w_router"], wl.k, "sigmoid", 1.0, None, inp["sel_bias"])
    r_0 = O.route(inp["x"], inp["w_router"], wl.k, "sigmoid", 1.0, None, None)
    same = np.all(np.sort(r_b["idx"], 1) == np.sort(r_0["idx"], 1), axis=1)
    assert same.any() and (~same).any()
    for t in np.nonzero(same)[0]:
        for j, e in enumerate(r_b["idx"][t]):
            j0 = list(r_0["idx"][t]).index(e)
            assert r_b["w"][t, j] == pytest.approx(r_0["w"][t, j0], rel=1e-14)
    # a shift shared by every bias changes no selection and no weight
    r_s = O.route(inp["x"], inp["w_router"], wl.k, "sigmoid", 1.0, None, inp["sel_bias"] + 0.25)
    assert np.array_equal(r_s["idx"], r_b["idx"])
    np.testing.assert_array_equal(r_s["w"], r_b["w"])


def test_selection_bias_refused_with_softmax():
    with pytest.raises(ValueError):
        O.selection_keys(np.zeros((1, 4)), "softmax", np.zeros(4))


# ---------------------------------------------------------------- dispatch

def test_dispatch_is_stable_and_invertible():
    rng = np.random.default_rng(3)
    T, E, k = 300, 7, 3
    idx = np.array([rng.choice(E, size=k, replace=False) for _ in range(T)])
    d = O.dispatch(idx, E)
    assert d["counts"].sum() == T * k and d["offsets"][-1] == T * k
    assert np.all(d["offsets"][1:] - d["offsets"][:-1] == d["counts"])
    for t in range(T):
        for j in range(k):
            r = d["row_of"][t, j]
            assert d["src_tok"][r] == t
            assert d["offsets"][idx[t, j]] <= r < d["offsets"][idx[t, j] + 1]
    for e in range(E):
        seg = d["src_tok"][d["offsets"][e]:d["offsets"][e + 1]]
        assert np.all(np.diff(seg) > 0)  # ascending token order within an expert
    # the permutation touches every row exactly once
    assert sorted(d["row_of"].ravel().tolist()) == list(range(T * k))


def test_permute_then_unpermute_identity():
    rng = np.random.default_rng(4)
    T, E, k, d = 64, 6, 3, 5
    idx = np.array([rng.choice(E, size=k, replace=False) for _ in range(T)])
    x = rng.standard_normal((T, d))
    dsp = O.dispatch(idx, E)
    xp = O.permute_rows(x, dsp["src_tok"])
    y = O.combine(xp, dsp["row_of"], np.ones((T, k)))
    np.testing.assert_allclose(y, k * x, rtol=1e-15)
    np.testing.assert_allclose(O.permute_backward(xp, dsp["row_of"]), k * x, rtol=1e-15)


# ---------------------------------------------------------------- aux loss

def test_aux_loss_uniform_routing_equals_coeff():
    T, E, k, coeff = 64, 8, 2, 0.37
    logits = np.zeros((T, E))            # P = 1/E for every token
    counts = np.full(E, T * k // E)      # perfectly even load
    assert O.aux_loss(logits, counts, k, coeff, "softmax") == pytest.approx(coeff, rel=1e-14)
    assert O.aux_loss(logits, counts, k, coeff, "sigmoid") == pytest.approx(coeff, rel=1e-14)


def test_sigmoid_aux_reading_hand_worked():
    """The sigmoid router's aux probabilities, read as s / sum_e s (the pages
    give no form), on two tokens and two experts worked by hand: logits
    (0, ln 3) and (-ln 3, ln 3) give scores (1/2, 3/4) and (1/4, 3/4), so
    P = (2/5, 3/5) and (1/4, 3/4); top-1 sends both tokens to expert 1
    (counts 0, 2) and aux = coeff * 2 / (1 * 2^2) * 2 * (3/5 + 3/4)
    = 1.35 coeff. A softmax over all experts would give 1.65 coeff and the
    unnormalised scores 1.5 coeff."""
    l3 = np.log(3.0)
    logits = np.array([[0.0, l3], [-l3, l3]])
    idx = O.topk_sorted(O.sigmoid(logits), 1)
    assert idx[:, 0].tolist() == [1, 1]
    counts = O.dispatch(idx, 2)["counts"]
    assert counts.tolist() == [0, 2]
    np.testing.assert_allclose(O.aux_probs(logits, "sigmoid"), [[0.4, 0.6], [0.25, 0.75]],
                               rtol=1e-15)
    assert O.aux_loss(logits, counts, 1, 0.1, "sigmoid") == pytest.approx(0.135, rel=1e-14)
    assert O.aux_loss(logits, counts, 1, 0.1, "softmax") == pytest.approx(0.165, rel=1e-14)


def test_aux_loss_single_expert_is_one():
    g = _load("handbook_counts.json")["single_expert_aux"]
    rng = np.random.default_rng(5)
    T = 33
    logits = rng.standard_normal((T, 1))
    idx = O.topk_sorted(logits, 1)
    counts = O.dispatch(idx, 1)["counts"]
    assert O.aux_loss(logits, counts, 1, 1.0, "softmax") == pytest.approx(
        g["load_balancing_loss_over_coeff"], rel=1e-14)


def test_aux_loss_is_sensitive_to_skewed_load():
    T, E, k = 64, 4, 1
    rng = np.random.default_rng(6)
    logits = rng.standard_normal((T, E))
    even = np.full(E, T // E)
    skew = np.array([T, 0, 0, 0])
    P = O.softmax_rows(logits)
    want = E / (k * T * T) * np.sum(skew * P.sum(0))
    assert O.aux_loss(logits, skew, k, 1.0, "softmax") == pytest.approx(want, rel=1e-14)
    assert O.aux_loss(logits, skew, k, 1.0, "softmax") != pytest.approx(
        O.aux_loss(logits, even, k, 1.0, "softmax"))


# ---------------------------------------------------------------- experts

def test_single_expert_top1_equals_dense_swiglu():
    """Handbook §2.5: a 1-expert top-1 MoE computes the dense FFN it came from.
    Checked against torch's own linear/silu in float64 (a different library)."""
    wl, inp = _tiny(E=1, k=1, coeff=0.0, F=10, d=12, T=20)
    f = O.layer_forward(wl, inp)
    x = torch.from_numpy(inp["x"])
    w1 = torch.from_numpy(inp["w1"][0])
    w2 = torch.from_numpy(inp["w2"][0])
    gate, up = torch.nn.functional.linear(x, w1).chunk(2, dim=-1)
    dense = torch.nn.functional.linear(torch.nn.functional.silu(gate) * up, w2)
    np.testing.assert_allclose(f["y"], dense.numpy(), rtol=1e-12, atol=1e-13)
    # swapping the gate and up halves must change the result
    swapped = torch.nn.functional.linear(torch.nn.functional.silu(up) * gate, w2)
    assert not np.allclose(f["y"], swapped.numpy(), rtol=1e-3)


def test_grouped_matches_per_token_evaluation():
    wl, inp = _tiny(E=5, k=2, F_shared=7, T=40)
    f = O.layer_forward(wl, inp)
    tf = O.tokens_forward(wl, inp, list(range(wl.T)))
    np.testing.assert_array_equal(tf["idx"], f["idx"])
    np.testing.assert_allclose(tf["y"], f["y"], rtol=1e-12, atol=1e-12)


def test_given_selection_on_exact_ties():
    """Where the k-th and (k+1)-th keys tie exactly, either expert is a valid
    choice (by default the lower index wins). The oracle takes a given
    selection and continues with the same definitions: the output of each tied
    token equals its per-token evaluation under that selection (a separate
    code path: one FFN per chosen expert, weighted sum), the weights are the
    softmax over the chosen logits, the counts move by one per tie, and a
    selection that repeats an expert is refused."""
    wl, inp = _tiny(E=4, k=2, T=24, seed=2)
    inp["w_router"][2] = inp["w_router"][1]  # experts 1 and 2 tie on every token
    f = O.layer_forward(wl, inp)
    ties = np.nonzero(f["gap"] == 0.0)[0]
    assert ties.size >= 2
    given = f["idx"].copy()
    for t in ties:
        assert 1 in given[t] and 2 not in given[t]  # the lower index won
        given[t][given[t] == 1] = 2
    g = O.layer_forward(wl, inp, idx=given)
    np.testing.assert_array_equal(g["idx"], given)
    np.testing.assert_allclose(g["w"], f["w"], rtol=0, atol=1e-15)
    tf = O.tokens_forward(wl, inp, list(ties), routing={"idx": given, "w": g["w"]})
    np.testing.assert_allclose(g["y"][ties], tf["y"], rtol=1e-12, atol=1e-12)
    assert np.max(np.abs(g["y"][ties] - f["y"][ties])) > 1e-3  # the choice matters
    assert g["counts"][2] == f["counts"][2] + ties.size
    assert g["counts"][1] == f["counts"][1] - ties.size
    bad = given.copy()
    bad[0] = [0, 0]
    with pytest.raises(ValueError):
        O.layer_forward(wl, inp, idx=bad)


# ---------------------------------------------------------------- gradients

def _fd_check(wl, inp, keys, eps=1e-6, rtol=2e-6, atol=1e-9):
    dy = inp["dy"]
    f = O.layer_forward(wl, inp)
    assert np.min(f["gap"]) > 1e-3  # no near ties: selection is locally constant
    b = O.layer_backward(wl, inp, f, dy)
    grad_of = {"x": "dx", "w_router": "dW_r", "w1": "dW1", "w2": "dW2",
               "w1_s": "dW1_s", "w2_s": "dW2_s", "w_gate_s": "dW_gate_s"}
    for name in keys:
        base = inp[name]
        g_an = b[grad_of[name]]
        g_fd = np.zeros_like(base)
        it = np.nditer(base, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            old = base[i]
            base[i] = old + eps
            lp = O.layer_loss(wl, inp, dy)
            base[i] = old - eps
            lm = O.layer_loss(wl, inp, dy)
            base[i] = old
            g_fd[i] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g_an, g_fd, rtol=rtol, atol=atol, err_msg=name)


def test_finite_differences_softmax_with_shared_expert():
    wl, inp = _tiny(E=4, k=2, F=3, d=4, T=6, F_shared=2, coeff=0.5, seed=1)
    _fd_check(wl, inp, ["x", "w_router", "w1", "w2", "w1_s", "w2_s"])


def test_finite_differences_sigmoid_with_bias_and_scaling():
    wl, inp = _tiny(score="sigmoid", E=5, k=3, F=3, d=4, T=6, sel=0.2, scaling=2.5,
                    coeff=0.5, seed=2)
    _fd_check(wl, inp, ["x", "w_router", "w1", "w2"])


def test_finite_differences_sigmoid_top1_with_logit_skew():
    wl, inp = _tiny(score="sigmoid", E=4, k=1, F=3, d=4, T=6, zipf=1.2, coeff=0.5, seed=3)
    _fd_check(wl, inp, ["x", "w_router", "w1"])


def test_aux_gradient_finite_differences():
    rng = np.random.default_rng(7)
    T, E, k = 9, 5, 2
    for score in ("softmax", "sigmoid"):
        logits = rng.standard_normal((T, E))
        counts = np.array([5, 0, 7, 3, 3])
        g = O.aux_loss_backward(logits, counts, k, 0.3, score)
        fd = np.zeros_like(logits)
        for t in range(T):
            for e in range(E):
                lp = logits.copy(); lp[t, e] += 1e-6
                lm = logits.copy(); lm[t, e] -= 1e-6
                fd[t, e] = (O.aux_loss(lp, counts, k, 0.3, score)
                            - O.aux_loss(lm, counts, k, 0.3, score)) / 2e-6
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-10)  # FD roundoff floor ~ |L| eps / h


def test_per_token_and_per_column_backward_match_full_backward():
    wl, inp = _tiny(E=4, k=2, F=6, d=5, T=30, F_shared=3, coeff=0.2, seed=4)
    f = O.layer_forward(wl, inp)
    b = O.layer_backward(wl, inp, f, inp["dy"])
    toks = [0, 7, 29]
    tb = O.tokens_backward(wl, inp, toks, f, f["counts"], inp["dy"][toks])
    np.testing.assert_allclose(tb["dw"], b["dw"][toks], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(tb["d_logits"], b["d_logits"][toks], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(tb["dx"], b["dx"][toks], rtol=1e-12, atol=1e-13)
    e = 2
    r0, r1 = f["offsets"][e], f["offsets"][e + 1]
    cols = [1, 4]
    cg = O.expert_grad_columns(f["x_perm"][r0:r1], b["d_out_perm"][r0:r1], inp["w1"][e],
                               inp["w2"][e], cols)
    np.testing.assert_allclose(cg["dW2_cols"], b["dW2"][e][:, cols], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(cg["dW1_gate"], b["dW1"][e][cols], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(cg["dW1_up"], b["dW1"][e][[wl.F + c for c in cols]],
                               rtol=1e-12, atol=1e-14)
