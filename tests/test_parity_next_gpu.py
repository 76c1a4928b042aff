"""GPU parity of the router z-loss, the sequence-wise aux loss and the
load-balance bookkeeping against the float64 oracle (the router variants
themselves run through the whole-layer parity cases)."""
import numpy as np
import pytest
import torch

import moe_inputs as mi
from oracle import moe_oracle as O
from tests.parity import TOL_AUX, TOL_F32, assert_close, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def L():
    from routing_grouped_expert_gate_gb300 import build
    build.build()
    from routing_grouped_expert_gate_gb300 import _lib
    return _lib


def _logits_and_idx(T, E, k, score, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    logits = (torch.randn(T, E, generator=g, device="cuda") * 2.0).contiguous()
    l64 = O.as_f64(logits)
    idx = O.topk_sorted(O.selection_keys(l64, score, None), k)
    return logits, torch.from_numpy(idx.astype(np.int32)).cuda(), l64, idx


@pytest.mark.parametrize("T,E", [(1, 8), (300, 64), (4100, 256)])
def test_z_loss(L, T, E):
    cfg = L.make_cfg(T=T, d=64, E=E, k=2, F=64)
    logits, _, l64, _ = _logits_and_idx(T, E, 2, "softmax", 40 + T)
    ws = torch.empty(L.workspace_bytes(cfg, L.MOE_WS_Z_LOSS), dtype=torch.uint8, device="cuda")
    z = torch.empty(1, device="cuda")
    coeff = 1e-3
    L.z_loss(cfg, logits, coeff, z, ws)
    ref = O.z_loss(l64, coeff)
    assert abs(float(z.item()) - ref) <= TOL_AUX * abs(ref)
    # backward, overwrite then accumulate
    d = torch.full((T, E), 7.0, device="cuda")
    L.z_loss_bwd(cfg, logits, coeff, 1.5, d, 0)
    g = O.z_loss_backward(l64, coeff, 1.5)
    assert_close("dz/dlogits", d, g, TOL_F32)
    L.z_loss_bwd(cfg, logits, coeff, 1.5, d, 1)
    assert_close("dz/dlogits accumulated", d, 2 * g, TOL_F32)
    # deterministic
    z2 = torch.empty(1, device="cuda")
    L.z_loss(cfg, logits, coeff, z2, ws)
    assert torch.equal(z, z2)
    assert L.last_device_status()[0] == 0


@pytest.mark.parametrize("score", ["softmax", "sigmoid", "sqrtsoftplus", "softmax_pre"])
@pytest.mark.parametrize("T,S,seq_major", [(512, 128, 0), (512, 128, 1), (600, 200, 0),
                                           (600, 200, 1), (96, 96, 0), (4096, 1024, 1),
                                           (8, 1, 0)])
def test_seq_aux_loss(L, score, T, S, seq_major):
    E, k, coeff = 32, 4, 1e-3
    cfg = L.make_cfg(T=T, d=64, E=E, k=k, F=64, score=score)
    logits, idx, l64, idx64 = _logits_and_idx(T, E, k, score, 50 + T + S)
    ws = torch.empty(max(L.seq_aux_workspace_bytes(cfg, S), 256), dtype=torch.uint8,
                     device="cuda")
    out = torch.empty(1, device="cuda")
    L.seq_aux_loss(cfg, logits, idx, S, seq_major, coeff, out, ws)
    ref = O.seq_aux_loss(l64, idx64, S, k, coeff, score, seq_major=bool(seq_major))
    assert abs(float(out.item()) - ref) <= TOL_AUX * abs(ref), (float(out.item()), ref)
    d = torch.zeros(T, E, device="cuda")
    L.seq_aux_loss_bwd(cfg, logits, idx, S, seq_major, coeff, 0.7, d, 1, ws)
    g = O.seq_aux_loss_backward(l64, idx64, S, k, coeff, score, g=0.7,
                                seq_major=bool(seq_major))
    assert_close("d seq_aux / d logits", d, g, TOL_F32)
    assert L.last_device_status()[0] == 0
    # one sequence: the micro-batch aux loss
    if S == T and score == "softmax":
        counts = torch.from_numpy(np.bincount(idx64.reshape(-1), minlength=E).astype(np.int32))
        aux = torch.empty(1, device="cuda")
        wsa = torch.empty(L.workspace_bytes(cfg, L.MOE_WS_AUX), dtype=torch.uint8,
                          device="cuda")
        L.aux_loss(L.make_cfg(T=T, d=64, E=E, k=k, F=64, aux_coeff=coeff), logits,
                   counts.cuda(), aux, wsa)
        assert abs(float(aux.item()) - float(out.item())) <= 1e-6 * abs(float(aux.item()))


def test_seq_len_must_divide_tokens(L):
    cfg = L.make_cfg(T=100, d=64, E=8, k=2, F=64)
    logits = torch.zeros(100, 8, device="cuda")
    idx = torch.zeros(100, 2, dtype=torch.int32, device="cuda")
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    out = torch.empty(1, device="cuda")
    assert L.seq_aux_workspace_bytes(cfg, 30) == 0
    with pytest.raises(L.MoeError):
        L.seq_aux_loss(cfg, logits, idx, 30, 0, 1e-3, out, ws)


def test_token_counts_bias_update_and_max_vio(L):
    E, k = 64, 8
    cfg = L.make_cfg(T=1, d=64, E=E, k=k, F=64, score="sigmoid")
    acc = torch.zeros(E, dtype=torch.int64, device="cuda")
    acc_ref = np.zeros(E, dtype=np.int64)
    rng = np.random.default_rng(60)
    for _ in range(3):
        counts = rng.integers(0, 5000, size=E).astype(np.int32)
        L.tokens_per_expert_accumulate(cfg, torch.from_numpy(counts).cuda(), acc)
        acc_ref = O.accumulate_tokens_per_expert(acc_ref, counts)
    assert np.array_equal(acc.cpu().numpy(), acc_ref)
    bias0 = (rng.standard_normal(E) * 0.05).astype(np.float32)
    bias = torch.from_numpy(bias0.copy()).cuda()
    rate = np.float32(1e-3)
    L.expert_bias_update(cfg, acc, bias, float(rate))
    # the oracle gives the direction; the bias itself is fp32 (bias + dir * rate in fp32)
    direction = O.expert_bias_update(acc_ref, np.zeros(E), 1.0).astype(np.float32)
    want = bias0 + direction * rate
    assert np.array_equal(bias.cpu().numpy(), want)
    mv = torch.empty(1, device="cuda")
    L.max_vio(cfg, acc, mv)
    assert float(mv.item()) == np.float32(O.max_vio(acc_ref))
    assert L.last_device_status()[0] == 0


def test_bias_update_compares_integers_on_the_device(L):
    cfg = L.make_cfg(T=1, d=64, E=2, k=1, F=64, score="sigmoid")
    acc = torch.tensor([2 ** 53 + 1, 2 ** 53 - 1], dtype=torch.int64, device="cuda")
    bias = torch.zeros(2, device="cuda")
    L.expert_bias_update(cfg, acc, bias, 0.5)
    assert bias.cpu().tolist() == [-0.5, 0.5]
    even = torch.tensor([7, 7], dtype=torch.int64, device="cuda")
    L.expert_bias_update(cfg, even, bias, 0.5)
    assert bias.cpu().tolist() == [-0.5, 0.5]


def test_max_vio_all_on_one_expert(L):
    # Handbook §3.3 "Cost of imbalance": top-8 of 64, every token on the busiest
    # expert -> MaxVio 7
    E, k, T = 64, 8, 1000
    cfg = L.make_cfg(T=T, d=64, E=E, k=k, F=64)
    tpe = torch.zeros(E, dtype=torch.int64, device="cuda")
    tpe[0] = T
    tpe[1:8] = T
    out = torch.empty(1, device="cuda")
    L.max_vio(cfg, tpe, out)
    assert float(out.item()) == 7.0


# ---------------------------------------------------------------- quantile balancing

def _quantile_inputs(T, E, seed, skew=0.0):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    logits = torch.randn(T, E, generator=g, device="cuda") * 2.0
    if skew:
        off = torch.log(torch.arange(1, E + 1, device="cuda", dtype=torch.float32) ** -1.2)
        logits = logits + skew * off[None, :]
    beta = (torch.randn(E, generator=g, device="cuda") * 0.3).contiguous()
    return logits.contiguous(), beta


def _run_quantile(L, cfg, logits, beta, solve=True):
    T, E, k = cfg.T, cfg.E, cfg.k
    idx = torch.empty(T, k, dtype=torch.int32, device="cuda")
    w = torch.empty(T, k, device="cuda")
    alpha = torch.empty(T, device="cuda")
    bl = torch.empty(E, device="cuda") if solve else None
    L.quantile_route(cfg, logits, beta, idx, w, alpha, bl)
    torch.cuda.synchronize()
    assert L.last_device_status()[0] == 0
    return idx, w, alpha, bl


@pytest.mark.parametrize("T,E,k", [(4096, 64, 4), (1000, 8, 2), (256, 256, 8)])
def test_quantile_route_softmax_is_exact(L, T, E, k):
    cfg = L.make_cfg(T=T, d=64, E=E, k=k, F=64, score="softmax")
    logits, beta = _quantile_inputs(T, E, 70 + T)
    idx, w, alpha, bl = _run_quantile(L, cfg, logits, beta)
    r = O.quantile_route(O.as_f64(logits), O.as_f64(beta), k, "softmax")
    # the keys are fp32 differences of the same fp32 inputs on both sides
    assert np.array_equal(idx.cpu().numpy(), r["idx"])
    assert np.array_equal(alpha.cpu().numpy().astype(np.float64), r["alpha"])
    assert np.array_equal(bl.cpu().numpy().astype(np.float64), r["beta_local"])
    assert_close("w", w, r["w"], TOL_F32)


@pytest.mark.parametrize("score", ["sigmoid", "sqrtsoftplus"])
def test_quantile_route_sigmoid_like(L, score):
    T, E, k = 2048, 32, 4
    cfg = L.make_cfg(T=T, d=64, E=E, k=k, F=64, score=score)
    logits, beta = _quantile_inputs(T, E, 80)
    idx, w, alpha, bl = _run_quantile(L, cfg, logits, beta)
    r = O.quantile_route(O.as_f64(logits), O.as_f64(beta), k, score)
    decided = r["gap"] >= 1e-6
    assert np.array_equal(idx.cpu().numpy()[decided], r["idx"][decided])
    assert np.max(np.abs(alpha.cpu().numpy() - r["alpha"])) < 1e-6
    assert np.max(np.abs(bl.cpu().numpy() - r["beta_local"])) < 1e-6
    assert_close("w", to_np(w)[decided], r["w"][decided], TOL_F32)


def test_quantile_accumulate_and_update(L):
    E = 64
    cfg = L.make_cfg(T=1024, d=64, E=E, k=4, F=64, score="sigmoid")
    accum = torch.zeros(E, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    beta = torch.zeros(E, device="cuda")
    sols = []
    for seed in range(3):
        logits, _ = _quantile_inputs(1024, E, 90 + seed, skew=1.0)
        _, _, _, bl = _run_quantile(L, cfg, logits, beta)
        L.quantile_accumulate(cfg, bl, accum, count)
        sols.append(O.as_f64(bl))
    beta0 = torch.linspace(-0.1, 0.2, E, device="cuda")
    beta.copy_(beta0)
    L.quantile_beta_update(cfg, beta, accum, count, 0.9)
    want = O.quantile_beta_update(O.as_f64(beta0), np.sum(sols, axis=0), 3, 0.9)
    assert np.max(np.abs(O.as_f64(beta) - want)) < 1e-6
    assert int(count.item()) == 0 and float(accum.abs().max()) == 0.0
    assert abs(float(beta.double().mean())) < 1e-6


def test_quantile_balancing_loop_evens_the_load(L):
    T, E, k = 4096, 32, 4
    cfg = L.make_cfg(T=T, d=64, E=E, k=k, F=64, score="sigmoid")
    logits, _ = _quantile_inputs(T, E, 100, skew=2.0)
    beta = torch.zeros(E, device="cuda")
    accum = torch.zeros(E, device="cuda")
    count = torch.zeros(1, dtype=torch.int32, device="cuda")
    first = None
    for _ in range(5):
        idx, _, _, bl = _run_quantile(L, cfg, logits, beta)
        c = np.bincount(idx.cpu().numpy().reshape(-1), minlength=E)
        first = O.max_vio(c) if first is None else first
        L.quantile_accumulate(cfg, bl, accum, count)
        L.quantile_beta_update(cfg, beta, accum, count, 0.0)
    idx, _, _, _ = _run_quantile(L, cfg, logits, beta, solve=False)
    c = np.bincount(idx.cpu().numpy().reshape(-1), minlength=E)
    assert c.sum() == T * k
    assert O.max_vio(c) < 0.25 < first


def test_quantile_refusals(L):
    logits = torch.zeros(10, 8, device="cuda")
    beta = torch.zeros(8, device="cuda")
    idx = torch.empty(10, 3, dtype=torch.int32, device="cuda")
    w = torch.empty(10, 3, device="cuda")
    alpha = torch.empty(10, device="cuda")
    bl = torch.empty(8, device="cuda")
    with pytest.raises(L.MoeError):  # 10 * 3 is not divisible by 8
        L.quantile_route(L.make_cfg(T=10, d=64, E=8, k=3, F=64, score="sigmoid"), logits, beta,
                         idx, w, alpha, bl)
    with pytest.raises(L.MoeError):  # pre-softmax is not a quantile score
        L.quantile_route(L.make_cfg(T=10, d=64, E=8, k=3, F=64, score="softmax_pre"), logits,
                         beta, idx, w, alpha, None)
