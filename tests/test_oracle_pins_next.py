"""Pins of the oracle's router variants and load-balance bookkeeping: sqrt(softplus)
and pre-softmax scores, the router z-loss, the sequence-wise aux loss, the
expert-bias sign update and the int64 token counts. Each check would fail on a
plausible slip (a wrong derivative, a missing 1/B, a float comparison where the
pages compare integers, a renormalisation where there is none)."""
import json
import math
import os

import numpy as np
import pytest

import moe_inputs as mi
from oracle import moe_oracle as O
from tests.test_oracle_pins import _fd_check, _tiny

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
G = json.load(open(os.path.join(GOLDEN, "router_variants.json")))


# ---------------------------------------------------------------- score functions

def test_gating_functions_rank_experts_alike():
    rng = np.random.default_rng(11)
    logits = rng.standard_normal((200, 16)) * 3
    ref = O.topk_sorted(O.selection_keys(logits, "softmax", None), 4)
    for score in ("sigmoid", "sqrtsoftplus", "softmax_pre"):
        np.testing.assert_array_equal(O.topk_sorted(O.selection_keys(logits, score, None), 4),
                                      ref, err_msg=score)


def test_sqrtsoftplus_closed_form():
    s = O.scores(np.array([[0.0, 30.0, -30.0]]), "sqrtsoftplus")[0]
    assert s[0] == pytest.approx(math.sqrt(math.log(2.0)), rel=1e-15)
    assert s[1] == pytest.approx(math.sqrt(30.0 + math.log1p(math.exp(-30.0))), rel=1e-15)
    assert s[2] == pytest.approx(math.sqrt(math.log1p(math.exp(-30.0))), rel=1e-12)
    # its derivative against central differences
    l = np.linspace(-6, 6, 25)[None, :]
    fd = (O.scores(l + 1e-6, "sqrtsoftplus") - O.scores(l - 1e-6, "sqrtsoftplus")) / 2e-6
    np.testing.assert_allclose(O.score_derivative(l, "sqrtsoftplus"), fd, rtol=1e-7)


def test_weight_ratio_limits_of_the_three_gating_functions():
    g = G["sqrtsoftplus_ratio_limit"]
    idx = np.array([[0, 1]])
    prev = None
    for scale in (0.5, 2.0, 10.0, 1e4):
        logits = np.array([[g["logit_ratio"] * scale, scale]])
        w = O.mixing_weights(logits, idx, "sqrtsoftplus", 1.0)[0]
        err = abs(w[0] / w[1] - g["weight_ratio_limit"])
        # approaches the limit as the scale grows
        assert prev is None or err < prev or err < 1e-12
        prev = err
    assert prev < 1e-12
    logits = np.array([[40.0, 10.0]])
    ws = O.mixing_weights(logits, idx, "sigmoid", 1.0)[0]
    assert ws[0] / ws[1] == pytest.approx(1.0, abs=1e-4)  # sigmoid saturates
    wm = O.mixing_weights(logits, idx, "softmax", 1.0)[0]
    assert wm[0] / wm[1] > 1e12  # softmax: the top expert takes nearly everything


def test_pre_softmax_weights_are_not_renormalised():
    # two experts whose logits differ by ln 3: full-softmax probabilities 3/4 and 1/4
    logits = np.array([[math.log(3.0), 0.0, -50.0]])
    r1 = O.mixing_weights(logits, np.array([[0]]), "softmax_pre", 1.0)
    assert r1[0, 0] == pytest.approx(0.75, rel=1e-12)
    assert O.mixing_weights(logits, np.array([[0]]), "softmax", 1.0)[0, 0] == 1.0
    r2 = O.mixing_weights(logits, np.array([[0, 1]]), "softmax_pre", 2.5)
    np.testing.assert_allclose(r2[0], [2.5 * 0.75, 2.5 * 0.25], rtol=1e-10)
    rng = np.random.default_rng(12)
    lg = rng.standard_normal((50, 8))
    idx = O.topk_sorted(O.selection_keys(lg, "softmax_pre", None), 3)
    w = O.mixing_weights(lg, idx, "softmax_pre", 1.0)
    mass = np.take_along_axis(O.softmax_rows(lg), idx, axis=1).sum(axis=1)
    np.testing.assert_allclose(w.sum(axis=1), mass, rtol=1e-14)
    assert np.all(w.sum(axis=1) < 1.0)


def test_selection_bias_refused_with_pre_softmax():
    with pytest.raises(ValueError):
        O.selection_keys(np.zeros((1, 4)), "softmax_pre", np.zeros(4))
    O.selection_keys(np.zeros((1, 4)), "sqrtsoftplus", np.zeros(4))  # accepted


def test_finite_differences_pre_softmax_top1_router_gets_a_gradient():
    wl, inp = _tiny(score="softmax_pre", E=4, k=1, F=3, d=4, T=6, coeff=0.5, seed=21)
    _fd_check(wl, inp, ["x", "w_router", "w1"])
    f = O.layer_forward(wl, inp)
    b = O.layer_backward(wl, inp, f, inp["dy"], g_aux=0.0)
    assert np.abs(b["dW_r"]).max() > 1e-6
    # every logit gets a gradient, not only the chosen one
    assert np.count_nonzero(np.abs(b["d_logits"]) > 0) == wl.T * wl.E


def test_finite_differences_pre_softmax_top2():
    wl, inp = _tiny(score="softmax_pre", E=5, k=2, F=3, d=4, T=6, coeff=0.5, scaling=1.7,
                    seed=22)
    _fd_check(wl, inp, ["x", "w_router", "w1", "w2"])


def test_finite_differences_sqrtsoftplus_with_bias_and_scaling():
    wl, inp = _tiny(score="sqrtsoftplus", E=5, k=3, F=3, d=4, T=6, sel=0.2, scaling=2.5,
                    coeff=0.5, seed=23)
    _fd_check(wl, inp, ["x", "w_router", "w1", "w2"])


def test_finite_differences_sqrtsoftplus_top1():
    wl, inp = _tiny(score="sqrtsoftplus", E=4, k=1, F=3, d=4, T=6, coeff=0.5, seed=24)
    _fd_check(wl, inp, ["x", "w_router"])


# ---------------------------------------------------------------- z-loss

def test_z_loss_closed_forms():
    T, E, c = 7, 16, 0.3
    logits = np.full((T, E), c)
    assert O.z_loss(logits, 1e-3) == pytest.approx(1e-3 * (c + math.log(E)) ** 2, rel=1e-14)
    g = G["z_loss_logged_value"]
    # logits whose logsumexp is sqrt(20.9) for every token: the logged value is 20.9
    lse = math.sqrt(g["logged_value"])
    logits = np.full((T, E), lse - math.log(E))
    coeff = 1e-3
    assert O.z_loss(logits, coeff) / coeff == pytest.approx(g["logged_value"], rel=1e-13)
    assert round(math.sqrt(g["logged_value"]), 1) == g["rms_logsumexp_about"]
    # the logsumexp, not the max: shifting one logit changes it
    l2 = logits.copy()
    l2[:, 0] -= 5.0
    assert O.z_loss(l2, coeff) < O.z_loss(logits, coeff)


def test_z_loss_gradient_finite_differences():
    rng = np.random.default_rng(25)
    logits = rng.standard_normal((6, 5)) * 2
    g = O.z_loss_backward(logits, 0.7, g=1.3)
    fd = np.zeros_like(logits)
    for t in range(6):
        for e in range(5):
            lp = logits.copy(); lp[t, e] += 1e-6
            lm = logits.copy(); lm[t, e] -= 1e-6
            fd[t, e] = 1.3 * (O.z_loss(lp, 0.7) - O.z_loss(lm, 0.7)) / 2e-6
    np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-10)


# ---------------------------------------------------------------- sequence-wise aux loss

def _routing(T, E, k, seed, score="softmax"):
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((T, E)) * 2
    idx = O.topk_sorted(O.selection_keys(logits, score, None), k)
    return logits, idx


def test_seq_aux_with_one_sequence_is_the_batch_aux_loss():
    for score in ("softmax", "sigmoid", "sqrtsoftplus"):
        logits, idx = _routing(48, 6, 2, 26, score)
        counts = O.dispatch(idx, 6)["counts"]
        assert O.seq_aux_loss(logits, idx, 48, 2, 0.1, score) == pytest.approx(
            O.aux_loss(logits, counts, 2, 0.1, score), rel=1e-13)


def test_seq_aux_is_the_mean_of_per_sequence_losses():
    S, B, E, k = 16, 3, 5, 2
    logits, idx = _routing(S * B, E, k, 27)
    per = []
    for b in range(B):
        rows = slice(b * S, (b + 1) * S)
        per.append(O.aux_loss(logits[rows], O.dispatch(idx[rows], E)["counts"], k, 0.2,
                              "softmax"))
    assert O.seq_aux_loss(logits, idx, S, k, 0.2, "softmax") == pytest.approx(np.mean(per),
                                                                               rel=1e-13)
    # it differs from the loss over the whole micro-batch (the scope matters)
    whole = O.aux_loss(logits, O.dispatch(idx, E)["counts"], k, 0.2, "softmax")
    assert abs(whole - np.mean(per)) > 1e-6


def test_seq_aux_uniform_routing_is_the_coefficient():
    S, B, E, k = 8, 4, 4, 2
    logits = np.zeros((S * B, E))
    idx = np.array([[(2 * t) % E, (2 * t + 1) % E] for t in range(S * B)])
    assert O.seq_aux_loss(logits, idx, S, k, 0.37, "softmax") == pytest.approx(0.37, rel=1e-14)


def test_seq_aux_layouts_agree():
    S, B, E, k = 10, 3, 6, 2
    logits, idx = _routing(S * B, E, k, 28)
    # batch-major token b*S+s  <->  sequence-major token s*B+b
    perm = np.array([(t % S) * B + t // S for t in range(S * B)])
    lm = np.empty_like(logits); lm[perm] = logits
    im = np.empty_like(idx); im[perm] = idx
    a = O.seq_aux_loss(logits, idx, S, k, 0.1, "softmax", seq_major=False)
    b = O.seq_aux_loss(lm, im, S, k, 0.1, "softmax", seq_major=True)
    assert a == pytest.approx(b, rel=1e-14)
    ga = O.seq_aux_loss_backward(logits, idx, S, k, 0.1, "softmax", seq_major=False)
    gb = O.seq_aux_loss_backward(lm, im, S, k, 0.1, "softmax", seq_major=True)
    np.testing.assert_allclose(gb[perm], ga, rtol=1e-14)


def test_seq_aux_gradient_finite_differences():
    S, B, E, k = 5, 2, 4, 2
    for score in ("softmax", "sqrtsoftplus"):
        logits, idx = _routing(S * B, E, k, 29, score)
        g = O.seq_aux_loss_backward(logits, idx, S, k, 0.4, score, g=0.9)
        fd = np.zeros_like(logits)
        for t in range(S * B):
            for e in range(E):
                lp = logits.copy(); lp[t, e] += 1e-6
                lm = logits.copy(); lm[t, e] -= 1e-6
                fd[t, e] = 0.9 * (O.seq_aux_loss(lp, idx, S, k, 0.4, score)
                                  - O.seq_aux_loss(lm, idx, S, k, 0.4, score)) / 2e-6
        np.testing.assert_allclose(g, fd, rtol=1e-6, atol=1e-10)


# ---------------------------------------------------------------- expert bias, counts

def test_bias_update_rule_on_the_pages_form():
    g = G["bias_update_rule"]
    new = O.expert_bias_update(np.array(g["counts"]), np.full(4, 0.25), 1e-3)
    np.testing.assert_allclose(new, 0.25 + 1e-3 * np.array(g["direction"]), rtol=0, atol=1e-15)
    # exactly at the mean: no move
    np.testing.assert_array_equal(O.expert_bias_update(np.array([2, 2, 2]), np.zeros(3), 1.0),
                                  np.zeros(3))


def test_bias_update_compares_integers_not_a_float_mean():
    # total 2^54 over two experts: counts 2^53 + 1 and 2^53 - 1. As doubles both
    # round to 2^53 = the mean and would not move; the integer rule moves both.
    c = np.array([2 ** 53 + 1, 2 ** 53 - 1], dtype=np.int64)
    np.testing.assert_array_equal(O.expert_bias_update(c, np.zeros(2), 1.0), [-1.0, 1.0])
    assert float(c[0]) == float(2 ** 53)  # the float mean cannot tell them apart


def test_token_counts_accumulate_over_micro_batches():
    E = 7
    acc = np.zeros(E, dtype=np.int64)
    all_idx = []
    for seed in range(3):
        _, idx = _routing(40, E, 3, 30 + seed)
        acc = O.accumulate_tokens_per_expert(acc, O.dispatch(idx, E)["counts"])
        all_idx.append(idx)
    np.testing.assert_array_equal(acc, O.dispatch(np.concatenate(all_idx), E)["counts"])
    assert acc.dtype == np.int64


# ---------------------------------------------------------------- quantile balancing

def test_quantile_route_selects_top_k_of_scores_minus_beta():
    rng = np.random.default_rng(31)
    T, E, k = 48, 8, 2
    logits = rng.standard_normal((T, E))
    beta = rng.standard_normal(E) * 0.3
    r = O.quantile_route(logits, beta, k, "softmax")
    v = (logits.astype(np.float32) - beta.astype(np.float32)).astype(np.float64)
    for t in range(T):
        ranked = sorted(range(E), key=lambda e: (-v[t, e], e))
        assert list(r["idx"][t]) == ranked[:k]
        assert r["alpha"][t] == v[t, ranked[k]]
    # the weights ignore beta: the same as plain routing with those experts
    np.testing.assert_allclose(r["w"], O.mixing_weights(logits, r["idx"], "softmax", 1.0))


def test_quantile_solution_by_brute_force():
    rng = np.random.default_rng(32)
    T, E, k = 12, 4, 2  # col_target = 6
    logits = rng.standard_normal((T, E))
    beta = np.zeros(E)
    r = O.quantile_route(logits, beta, k, "sigmoid")
    s32 = O.scores(logits, "sigmoid").astype(np.float32)
    for e in range(E):
        col = [float(np.float32(s32[t, e] - np.float32(r["alpha"][t]))) for t in range(T)]
        col.sort(reverse=True)
        assert r["beta_local"][e] == col[T * k // E]  # the 7th largest
    with pytest.raises(ValueError):
        O.quantile_route(logits[:11], beta, k, "sigmoid")  # 11 * 2 not divisible by 4


def test_quantile_balancing_evens_the_load_faster_than_the_sign_update():
    g = G["quantile_balancing"]
    rng = np.random.default_rng(33)
    T, E, k = 512, 16, 2
    skew = np.log(np.arange(1, E + 1, dtype=np.float64) ** -1.2)
    logits = rng.standard_normal((T, E)) + 2.0 * skew[None, :]
    target = T * k // E
    beta = np.zeros(E)
    bias = np.zeros(E)
    for _ in range(g["steps"]):
        r = O.quantile_route(logits, beta, k, "sigmoid")
        beta = O.quantile_beta_update(beta, r["beta_local"], 1, ema=0.0)
        keys = O.selection_keys(logits, "sigmoid", bias)
        counts = O.dispatch(O.topk_sorted(keys, k), E)["counts"]
        bias = O.expert_bias_update(counts, bias, 1e-3)
    q_counts = O.dispatch(O.quantile_route(logits, beta, k, "sigmoid", solve=False)["idx"],
                          E)["counts"]
    s_counts = O.dispatch(O.topk_sorted(O.selection_keys(logits, "sigmoid", bias), k),
                          E)["counts"]
    assert q_counts.sum() == s_counts.sum() == T * k
    assert O.max_vio(q_counts) < 0.25
    assert O.max_vio(q_counts) < 0.25 * O.max_vio(s_counts)
    assert abs(q_counts - target).max() < abs(s_counts - target).max()


def test_quantile_beta_update_ema_and_centring():
    beta = np.array([0.5, -0.25, 1.0, 0.0])
    accum = np.array([1.0, 2.0, 3.0, 6.0])
    nb = O.quantile_beta_update(beta, accum, 2, ema=0.75)
    want = 0.75 * beta + 0.25 * accum / 2
    np.testing.assert_allclose(nb, want - want.mean(), rtol=1e-15)
    assert abs(nb.mean()) < 1e-15
    np.testing.assert_allclose(O.quantile_beta_update(beta, accum, 0, ema=1.0),
                               beta - beta.mean())


# ---------------------------------------------------------------- expert activations

GA = json.load(open(os.path.join(GOLDEN, "expert_activations.json")))


def _gu(seed=40, n=400):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, 7)) * 12, rng.standard_normal((n, 7)) * 12


def test_clamp_validation_follows_the_pages():
    c = GA["swiglu_clamp_value"]["clamp"]
    O.GluAct("swiglu_clamp", clamp=c).check()
    for bad in (0.0, -1.0, math.inf, math.nan):
        with pytest.raises(ValueError):
            O.GluAct("swiglu_clamp", clamp=bad).check()
    with pytest.raises(ValueError):
        O.GluAct("swiglu_clamp", clamp=c, offset=0.5).check()


def test_clamped_swiglu_limits_and_bound():
    g, u = _gu()
    c = GA["swiglu_clamp_value"]["clamp"]
    plain = O.glu_forward(g, u, O.SWIGLU)
    # a limit no activation reaches changes nothing
    np.testing.assert_array_equal(O.glu_forward(g, u, O.GluAct("swiglu_clamp", clamp=1e9)),
                                  plain)
    h = O.glu_forward(g, u, O.GluAct("swiglu_clamp", clamp=c))
    # the point of the clamp: |h| <= silu(c) * c, while plain SwiGLU exceeds it here
    bound = c * c / (1.0 + math.exp(-c))
    assert np.abs(h).max() <= bound * (1 + 1e-15)
    assert np.abs(plain).max() > bound
    # inside the box the two agree
    inside = (g <= c) & (np.abs(u) <= c)
    np.testing.assert_array_equal(h[inside], plain[inside])


def test_situ_glu_limits_and_bound():
    g, u = _gu(41)
    sg, sl = GA["situ_glu"]["gate_scale"], GA["situ_glu"]["linear_scale"]
    # a huge scale is SwiGLU: s tanh(x / s) -> x
    big = O.glu_forward(g, u, O.GluAct("situ_glu", gate_scale=1e7))
    np.testing.assert_allclose(big, O.glu_forward(g, u, O.SWIGLU), rtol=1e-9, atol=1e-12)
    # the smooth cap: the gate stays below s, the linear half below s_l
    act = O.GluAct("situ_glu", gate_scale=sg, linear_scale=sl)
    h = O.glu_forward(g, u, act)
    gate_only = O.glu_forward(g, np.ones_like(u), O.GluAct("situ_glu", gate_scale=sg))
    assert np.abs(gate_only).max() < sg
    lin_only = O.glu_forward(np.full_like(g, 50.0), u,
                             O.GluAct("situ_glu", gate_scale=1e7, linear_scale=sl)) / 50.0
    assert np.abs(lin_only).max() < sl
    assert np.abs(h).max() < sg * sl


@pytest.mark.parametrize("act", [
    {"act_fn": "swiglu_clamp", "act_clamp": 0.6},
    {"act_fn": "situ_glu", "act_gate_scale": 0.8, "act_linear_scale": 0.9},
    {"act_fn": "situ_glu", "act_gate_scale": 1.5},
    {"act_fn": "swiglu", "glu_linear_offset": 0.3},
])
def test_finite_differences_expert_activations(act):
    wl, inp = _tiny(E=4, k=2, F=3, d=4, T=6, F_shared=2, coeff=0.5, seed=42, **act)
    if act["act_fn"] == "swiglu_clamp":
        # some inputs are clipped, none sits on the edge (where the derivative jumps)
        f = O.layer_forward(wl, inp)
        c = act["act_clamp"]
        g = np.concatenate([f["g"].ravel(), f["g_s"].ravel()])
        u = np.concatenate([f["u"].ravel(), f["u_s"].ravel()])
        assert np.any(g > c) and np.any(np.abs(u) > c)
        assert np.min(np.abs(g - c)) > 1e-4 and np.min(np.abs(np.abs(u) - c)) > 1e-4
    _fd_check(wl, inp, ["x", "w_router", "w1", "w2", "w1_s", "w2_s"])


def test_shared_gate_half_at_zero_weight_and_gradients():
    wl, inp = _tiny(E=4, k=2, F=3, d=4, T=6, F_shared=2, coeff=0.5, seed=43, shared_gate=True)
    assert inp["w_gate_s"] is not None and inp["w_gate_s"].shape == (4,)
    f = O.layer_forward(wl, inp)
    ungated = dict(inp, w_gate_s=None)
    f0 = O.layer_forward(wl, ungated)
    zero = dict(inp, w_gate_s=np.zeros(4))
    fz = O.layer_forward(wl, zero)
    routed = f0["y"] - f0["y_s"]
    np.testing.assert_allclose(fz["y"], routed + 0.5 * f0["y_s"], rtol=1e-14, atol=1e-15)
    assert not np.allclose(f["y"], f0["y"])
    _fd_check(wl, inp, ["x", "w_router", "w1_s", "w2_s", "w_gate_s"])
