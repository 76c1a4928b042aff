"""CPU oracle for one token-choice MoE layer, forward and backward, in float64.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
this module: only the tests, ``__graft_entry__.smoke()`` and ``bench.py``'s
CPU-baseline leg (and its ``--impl reference`` arm) use it. It shares no code
with the CUDA path; its inputs come from ``moe_inputs`` (random tensors only).

It is the plain definition of the layer, written with numpy loops and numpy
matrix products, in the order the pages state the steps:

  S1  gate GEMM          The Ultimate MoE Training Handbook, §3.1 "Router scoring",
                         part "Precision" (router GEMM computed in fp32, weight [E, d])
  S2  scores + top-k     same section, parts "Gating function" and "Output scale"
                         (top-k on logits then softmax over the chosen; or sigmoid,
                         selection bias added for selection only, renormalised with
                         +1e-20, times the routed scaling factor); §3.2 "Who selects"
                         (sorted top-k)
  S3  dispatch           MoE training cluster: routing, load balancing (LeCompute),
                         "Read the timeline before blaming the network" (group rows by
                         expert, restore order later); "Four GPUs, with one holding up
                         the group" (per-expert assignment counts)
  S4/S5 SwiGLU experts   Handbook §3.4 "Experts", parts "Count and size" (fc1 is twice
                         the FFN width, fc2 maps F back to d) and "Activation" (the gate
                         is the first half of fc1's output); §2.5 (bias-free experts)
  S5s shared expert      Handbook §3.4 "Shared experts" (added at weight 1)
  S6  combine            LeCompute, "An expert transforms numbers inside the model"
                         (y = sum of chosen outputs times their weights)
  S7  Switch aux loss    Handbook §3.3 "Load balancing", part "Aux loss"
                         (coeff * E / (k * T^2) * sum_e count_e * sum_t P[t, e])

Backward: the chain rule applied to the same definitions (LeCompute, "How the
router learns without an expert-selection answer key": the gradient reaches the
router only through the mixing weights of the chosen experts; the discrete
choice itself has no derivative).

Readings where the pages leave a step open (each is also listed in the design
notes of the repository):
  * top-k ties: descending key, equal keys go to the lower expert index; the
    decision is taken on the key rounded once to fp32, the router's dtype
  * aux-loss probabilities: the softmax over all E logits (no bias); for the
    sigmoid router, s / sum_e s (parity unpinned there except by invariants
    and a case of the reading worked by hand)
  * counts come from the final selection (bias included) and carry no gradient
  * the combine and every reduction are exact sums in float64

Every function takes float64 numpy arrays (exact widenings of the bf16/fp32
inputs) and returns float64 / int64 arrays.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, Optional, Sequence

import numpy as np

SIGMOID_RENORM_EPS = 1e-20  # Handbook §3.1 "Output scale": sum of chosen scores + 1e-20


# ----------------------------------------------------------------------------
# helpers
# ----------------------------------------------------------------------------

def as_f64(t) -> Optional[np.ndarray]:
    """Widen a torch tensor (bf16/fp32, any device) or array to float64 numpy."""
    if t is None:
        return None
    if hasattr(t, "detach"):
        return t.detach().to("cpu").double().numpy()
    return np.asarray(t, dtype=np.float64)


def sigmoid(z: np.ndarray) -> np.ndarray:
    """1 / (1 + exp(-z)), evaluated without overflow for either sign."""
    z = np.asarray(z, dtype=np.float64)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def silu(z: np.ndarray) -> np.ndarray:
    return z * sigmoid(z)


def softplus(z: np.ndarray) -> np.ndarray:
    """log(1 + exp(z)), evaluated without overflow for either sign."""
    return np.logaddexp(0.0, np.asarray(z, dtype=np.float64))


def logsumexp_rows(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def softmax_rows(z: np.ndarray) -> np.ndarray:
    m = z.max(axis=-1, keepdims=True)
    e = np.exp(z - m)
    return e / e.sum(axis=-1, keepdims=True)


# ----------------------------------------------------------------------------
# S1 + S2: router
# ----------------------------------------------------------------------------

def gate_logits(x: np.ndarray, w_router: np.ndarray,
                logit_bias: Optional[np.ndarray] = None) -> np.ndarray:
    """S1: logits[t, e] = sum_c x[t, c] * w_router[e, c]  (+ logit_bias[e]).

    Handbook §3.1 "Precision": the router GEMM takes the input and the [E, d]
    router weight in the router dtype. The logit bias is how a workload adds a
    fixed per-expert skew to the logits; it moves selection and weights alike.
    """
    logits = x @ w_router.T
    if logit_bias is not None:
        logits = logits + logit_bias[None, :]
    return logits


SCORE_FUNCTIONS = ("softmax", "sigmoid", "sqrtsoftplus", "softmax_pre")


def scores(logits: np.ndarray, score: str) -> np.ndarray:
    """Per-expert scores before selection.

    Handbook §3.1 "Gating function": softmax routing selects on the logits
    themselves (the softmax over the chosen comes after the top-k); with the
    pre-softmax setting ("Output scale": --moe-router-pre-softmax) the softmax
    over all E experts comes first and the top-k ranks its probabilities;
    sigmoid routing selects on sigmoid(logits); sqrt(softplus) routing on
    sqrt(log(1 + exp(logits))).
    """
    if score == "softmax":
        return logits.copy()
    if score == "softmax_pre":
        return softmax_rows(logits)
    if score == "sigmoid":
        return sigmoid(logits)
    if score == "sqrtsoftplus":
        return np.sqrt(softplus(logits))
    raise ValueError(score)


def score_derivative(logits: np.ndarray, score: str) -> np.ndarray:
    """d score / d logit, elementwise, for the sigmoid-like score functions."""
    if score == "sigmoid":
        s = sigmoid(logits)
        return s * (1.0 - s)
    if score == "sqrtsoftplus":
        # d/dl sqrt(softplus(l)) = sigmoid(l) / (2 sqrt(softplus(l)))
        return sigmoid(logits) / (2.0 * np.sqrt(softplus(logits)))
    raise ValueError(score)


def selection_keys(logits: np.ndarray, score: str,
                   sel_bias: Optional[np.ndarray]) -> np.ndarray:
    """The values the top-k ranks: scores, plus the expert bias when there is one.

    Handbook §3.3 "Loss-free bias": the bias is added to the score before the
    top-k and is used only to pick experts.
    """
    s = scores(logits, score)
    if sel_bias is not None:
        if score in ("softmax", "softmax_pre"):
            raise ValueError("the selection bias is refused with softmax scores "
                             "(Handbook §3.1, Gating function)")
        s = s + sel_bias[None, :]
    return s


def topk_sorted(keys: np.ndarray, k: int) -> np.ndarray:
    """Indices of the k largest keys per row, in descending key order.

    Handbook §3.2 "Who selects": top-k sorted while training. Equal keys are
    ordered by ascending expert index (the pages leave tie order open). The
    comparison is made on the keys rounded to fp32, the router's precision.
    """
    keys32 = keys.astype(np.float32)
    order = np.argsort(-keys32, axis=1, kind="stable")
    return order[:, :k].astype(np.int64)


def kth_gap(keys: np.ndarray, k: int) -> np.ndarray:
    """Per token: (k-th largest key) - ((k+1)-th largest key), in float64.

    Tokens whose gap is below 1e-6 are near ties: their selection depends on
    rounding and they are excluded from exact index comparisons.
    """
    T, E = keys.shape
    if k >= E:
        return np.full(T, np.inf)
    srt = -np.sort(-keys, axis=1)
    return srt[:, k - 1] - srt[:, k]


def mixing_weights(logits: np.ndarray, idx: np.ndarray, score: str,
                   scaling: float) -> np.ndarray:
    """Weights of the chosen experts.

    Handbook §3.1 "Gating function" and "Output scale": softmax routing takes
    the softmax over the k chosen logits (the renormalised softmax); with the
    pre-softmax setting the weights are the chosen experts' probabilities
    under the softmax over all E, not renormalised; sigmoid and sqrt(softplus)
    routing divide each chosen score by their sum plus 1e-20 when k > 1 (the
    expert bias never enters); then everything is multiplied by the routed
    scaling factor.
    """
    k = idx.shape[1]
    sel_logits = np.take_along_axis(logits, idx, axis=1)
    if score == "softmax":
        p = softmax_rows(sel_logits)
    elif score == "softmax_pre":
        p = np.take_along_axis(softmax_rows(logits), idx, axis=1)
    else:
        s = scores(sel_logits, score)
        p = s / (s.sum(axis=1, keepdims=True) + SIGMOID_RENORM_EPS) if k > 1 else s
    return p * scaling


def route(x, w_router, k: int, score: str, scaling: float = 1.0,
          logit_bias=None, sel_bias=None, idx=None) -> Dict[str, np.ndarray]:
    """S1 + S2 for every token: logits, sorted indices, weights, near-tie gaps.

    `idx` [T, k], when given, is taken as the selection instead of the top-k of
    the keys (a token whose k-th and (k+1)-th keys tie to within rounding may
    be decided either way; everything after the choice follows the same
    definitions). Each row must hold k distinct experts.
    """
    logits = gate_logits(x, w_router, logit_bias)
    keys = selection_keys(logits, score, sel_bias)
    if idx is None:
        idx = topk_sorted(keys, k)
    else:
        idx = np.asarray(idx, dtype=np.int64)
        E = logits.shape[1]
        if idx.shape != (logits.shape[0], k) or np.any((idx < 0) | (idx >= E)) or any(
                len(set(r)) != k for r in idx.tolist()):
            raise ValueError("a given selection needs k distinct experts per token")
    w = mixing_weights(logits, idx, score, scaling)
    return {"logits": logits, "keys": keys, "idx": idx, "w": w, "gap": kth_gap(keys, k)}


# ----------------------------------------------------------------------------
# S3: dispatch
# ----------------------------------------------------------------------------

def dispatch(idx: np.ndarray, E: int) -> Dict[str, np.ndarray]:
    """Histogram, exclusive scan and stable permutation of the assignments.

    LeCompute, "Four GPUs, with one holding up the group": counts[e] is the
    number of token-expert assignments of expert e (they sum to T*k).
    LeCompute, "Read the timeline before blaming the network": the rows are
    grouped by expert (expert-contiguous), and the grouping is undone later.
    Within one expert, rows follow ascending token index (the stable order).
    """
    T, k = idx.shape
    counts = np.zeros(E, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            counts[idx[t, j]] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):
        offsets[e + 1] = offsets[e] + counts[e]
    cursor = offsets[:E].copy()
    row_of = np.zeros((T, k), dtype=np.int64)
    src_tok = np.zeros(T * k, dtype=np.int64)
    for t in range(T):
        for j in range(k):
            e = idx[t, j]
            row_of[t, j] = cursor[e]
            src_tok[cursor[e]] = t
            cursor[e] += 1
    return {"counts": counts, "offsets": offsets, "row_of": row_of, "src_tok": src_tok}


def permute_rows(x: np.ndarray, src_tok: np.ndarray) -> np.ndarray:
    """x_perm[r] = x[src_tok[r]]: one copy of the token per chosen expert."""
    return x[src_tok]


def max_vio(counts: np.ndarray) -> float:
    """MaxVio = (busiest expert's load - mean load) / mean load.

    Handbook §3.2 "Who selects" and LeCompute, "Which tokens are supposed to
    balance?".
    """
    counts = np.asarray(counts, dtype=np.float64)
    mean = counts.mean()
    return float((counts.max() - mean) / mean)


# ----------------------------------------------------------------------------
# GLU activations of the experts
# ----------------------------------------------------------------------------

@dataclasses.dataclass(frozen=True)
class GluAct:
    """The expert activation applied to fc1's [gate | linear] halves.

    Handbook §3.4 "Experts", part "Activation" and its code: glu() computes
    act(x_glu) * (x_linear + glu_linear_offset) with SiLU; a clamp value c
    clips x_glu from above at c and x_linear to [-c, c] first (SwiGLU with a
    hard clamp; c must be finite and > 0, and the offset zero); SiTU-GLU
    replaces the gate by situ(x, s) = s tanh(x / s) sigmoid(x) and, with a
    linear scale, soft-clamps x_linear to s_l tanh(x_linear / s_l).
    """
    kind: str = "swiglu"        # "swiglu" | "swiglu_clamp" | "situ_glu"
    clamp: float = 0.0
    gate_scale: float = 0.0
    linear_scale: float = 0.0   # 0: the linear half is not soft-clamped
    offset: float = 0.0

    def check(self) -> "GluAct":
        if self.kind == "swiglu_clamp":
            if not (math.isfinite(self.clamp) and self.clamp > 0):
                raise ValueError("the SwiGLU clamp value must be finite and > 0")
            if self.offset != 0.0:
                raise ValueError("glu_linear_offset must be 0 with the SwiGLU clamp")
        elif self.kind == "situ_glu":
            if not self.gate_scale > 0:
                raise ValueError("SiTU-GLU needs a gate scale > 0")
        elif self.kind != "swiglu":
            raise ValueError(self.kind)
        return self


SWIGLU = GluAct()


def act_of(wl) -> GluAct:
    """The activation a workload asks for (SwiGLU when it names none)."""
    return GluAct(getattr(wl, "act_fn", "swiglu"), getattr(wl, "act_clamp", 0.0),
                  getattr(wl, "act_gate_scale", 0.0), getattr(wl, "act_linear_scale", 0.0),
                  getattr(wl, "glu_linear_offset", 0.0)).check()


def glu_forward(g: np.ndarray, u: np.ndarray, act: GluAct = SWIGLU) -> np.ndarray:
    if act.kind == "swiglu":
        return silu(g) * (u + act.offset)
    if act.kind == "swiglu_clamp":
        c = act.clamp
        return silu(np.minimum(g, c)) * np.clip(u, -c, c)
    s = act.gate_scale
    gate = s * np.tanh(g / s) * sigmoid(g)
    lin = act.linear_scale * np.tanh(u / act.linear_scale) if act.linear_scale > 0 else u
    return gate * (lin + act.offset)


def glu_backward(g: np.ndarray, u: np.ndarray, dh: np.ndarray, act: GluAct = SWIGLU,
                 decide=None):
    """(dg, du) of h = glu_forward(g, u). A clipped input passes no gradient
    (the clip is the identity, derivative 1, on [-c, c] ends included).

    `decide` = (g', u'): the values the clip decisions are taken on, when
    they must be those of a lower-precision copy (a bf16 layer keeps its
    pre-activations in bf16 for the backward)."""
    sg = sigmoid(g)
    if act.kind == "swiglu":
        dsilu = sg * (1.0 + g * (1.0 - sg))
        return dh * (u + act.offset) * dsilu, dh * (g * sg)
    if act.kind == "swiglu_clamp":
        c = act.clamp
        gd, ud = (g, u) if decide is None else decide
        gc = np.minimum(g, c)
        uc = np.clip(u, -c, c)
        sgc = sigmoid(gc)
        dg = dh * uc * sgc * (1.0 + gc * (1.0 - sgc)) * (gd <= c)
        du = dh * (gc * sgc) * ((ud >= -c) & (ud <= c))
        return dg, du
    s = act.gate_scale
    th = np.tanh(g / s)
    gate = s * th * sg
    dgate = (1.0 - th * th) * sg + s * th * sg * (1.0 - sg)
    if act.linear_scale > 0:
        tl = np.tanh(u / act.linear_scale)
        lin = act.linear_scale * tl
        dlin = 1.0 - tl * tl
    else:
        lin = u
        dlin = np.ones_like(u)
    return dh * (lin + act.offset) * dgate, dh * gate * dlin


# ----------------------------------------------------------------------------
# S4 / S5: SwiGLU experts
# ----------------------------------------------------------------------------

def swiglu_ffn(xs: np.ndarray, w1: np.ndarray, w2: np.ndarray,
               act: GluAct = SWIGLU) -> Dict[str, np.ndarray]:
    """One bias-free SwiGLU expert on the rows xs [n, d].

    Handbook §3.4 "Count and size": fc1 has twice the FFN width, fc2 maps the
    FFN width F back to d; "Activation": fc1's output is split in two halves,
    the first is the gate (through SiLU), the second the linear part, and the
    two are multiplied (glu_forward: SiLU by default, or a clamped / SiTU
    variant). w1 is [2F, d], w2 is [d, F].
    """
    F = w2.shape[1]
    gu = xs @ w1.T
    g = gu[:, :F]
    u = gu[:, F:]
    h = glu_forward(g, u, act)
    out = h @ w2.T
    return {"g": g, "u": u, "h": h, "out": out}


def grouped_swiglu(x_perm: np.ndarray, offsets: np.ndarray, w1: np.ndarray,
                   w2: np.ndarray, act: GluAct = SWIGLU) -> Dict[str, np.ndarray]:
    """Each expert e runs its FFN on its own contiguous segment of rows."""
    A = x_perm.shape[0]
    E, twoF, _ = w1.shape
    F = twoF // 2
    d = w2.shape[1]
    g = np.zeros((A, F))
    u = np.zeros((A, F))
    h = np.zeros((A, F))
    out = np.zeros((A, d))
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue
        res = swiglu_ffn(x_perm[r0:r1], w1[e], w2[e], act)
        g[r0:r1], u[r0:r1], h[r0:r1], out[r0:r1] = res["g"], res["u"], res["h"], res["out"]
    return {"g": g, "u": u, "h": h, "out": out}


# ----------------------------------------------------------------------------
# S6: combine
# ----------------------------------------------------------------------------

def shared_gate(x: np.ndarray, w_gate: np.ndarray) -> np.ndarray:
    """Handbook §3.4 "Shared experts" (--moe-shared-expert-gate): a sigmoid
    gate on the shared expert's output, sigmoid(x · w_gate) per token, from a
    [d] gate weight."""
    return sigmoid(x @ w_gate)


def combine(out_perm: np.ndarray, row_of: np.ndarray, w: np.ndarray,
            y_shared: Optional[np.ndarray] = None) -> np.ndarray:
    """y[t] = sum_j w[t, j] * out_perm[row_of[t, j]]  (+ y_shared[t]).

    LeCompute, "An expert transforms numbers inside the model": with weights
    0.75 and 0.25 the block returns 0.75 * output_A + 0.25 * output_B, one
    coordinate at a time. Handbook §3.4 "Shared experts": the shared expert's
    output is added at weight 1.
    """
    T, k = row_of.shape
    y = np.zeros((T, out_perm.shape[1]))
    for j in range(k):
        y += w[:, j:j + 1] * out_perm[row_of[:, j]]
    if y_shared is not None:
        y = y + y_shared
    return y


# ----------------------------------------------------------------------------
# S7: Switch load-balancing loss
# ----------------------------------------------------------------------------

def aux_probs(logits: np.ndarray, score: str) -> np.ndarray:
    """Router probabilities the aux loss averages: softmax over all E experts.

    For sigmoid and sqrt(softplus) scores the pages give no form; the reading
    here normalises the scores over all experts, s / sum_e s.
    """
    if score in ("softmax", "softmax_pre"):
        return softmax_rows(logits)
    s = scores(logits, score)
    return s / s.sum(axis=1, keepdims=True)


def aux_loss(logits: np.ndarray, counts: np.ndarray, k: int, coeff: float,
             score: str) -> float:
    """Handbook §3.3 "Aux loss": coeff * E / (k * T^2) * sum_e counts[e] * sum_t P[t, e]."""
    T, E = logits.shape
    P = aux_probs(logits, score)
    col = P.sum(axis=0)
    return float(np.sum(col * counts.astype(np.float64)) * (E * coeff / (k * T * T)))


# ----------------------------------------------------------------------------
# router z-loss
# ----------------------------------------------------------------------------

def z_loss(logits: np.ndarray, coeff: float) -> float:
    """Handbook §3.1 "Router scoring", part "Precision" (z_loss_func): the mean over tokens of
    the squared logsumexp of each token's logits, times the coefficient. (The
    value Megatron logs is this divided by the coefficient, the mean squared
    logsumexp.)"""
    T = logits.shape[0]
    if T == 0:
        return 0.0
    lse = logsumexp_rows(logits)
    return float(coeff * np.mean(lse * lse))


def z_loss_backward(logits: np.ndarray, coeff: float, g: float = 1.0,
                    T_total: Optional[int] = None) -> np.ndarray:
    """d(g * z_loss)/d(logits) = g * coeff * 2 * lse_t * softmax(l_t) / T."""
    n = logits.shape[0]
    T = n if T_total is None else T_total
    lse = logsumexp_rows(logits)
    return (g * coeff * 2.0 / T) * lse[:, None] * softmax_rows(logits)


# ----------------------------------------------------------------------------
# load-balance bookkeeping: sequence-wise aux loss, expert bias update
# ----------------------------------------------------------------------------

def sequence_of_tokens(T: int, seq_len: int, seq_major: bool) -> np.ndarray:
    """Sequence index of every token of a micro-batch of T = B * seq_len tokens.

    Batch-major storage (seq_major False): token t = b * seq_len + s. Sequence-
    major storage, the [seq, batch] order Megatron's activations use: token
    t = s * B + b.
    """
    B = T // seq_len
    t = np.arange(T)
    return (t % B) if seq_major else (t // seq_len)


def seq_aux_loss(logits: np.ndarray, idx: np.ndarray, seq_len: int, k: int, coeff: float,
                 score: str, seq_major: bool = False) -> float:
    """Handbook §3.3 "Load balancing", part "Scope" (seq_aux_loss): the
    Switch loss taken over each sequence on its own, with that sequence's
    counts, probabilities and length, then averaged over the B sequences:
      (1/B) sum_b coeff * E / (k * S^2) * sum_e c[b, e] * sum_{t in b} P[t, e]."""
    T, E = logits.shape
    B = T // seq_len
    seq = sequence_of_tokens(T, seq_len, seq_major)
    P = aux_probs(logits, score)
    total = 0.0
    for b in range(B):
        rows = np.nonzero(seq == b)[0]
        c = np.bincount(idx[rows].reshape(-1), minlength=E).astype(np.float64)
        total += coeff * E / (k * seq_len * seq_len) * float(np.sum(c * P[rows].sum(axis=0)))
    return total / B


def seq_aux_loss_backward(logits, idx, seq_len: int, k: int, coeff: float, score: str,
                          g: float = 1.0, seq_major: bool = False) -> np.ndarray:
    """d(g * seq_aux_loss)/d(logits), counts held constant: each sequence's
    tokens get the aux-loss gradient of their own sequence, scaled by 1/B."""
    T, E = logits.shape
    B = T // seq_len
    seq = sequence_of_tokens(T, seq_len, seq_major)
    out = np.zeros((T, E))
    for b in range(B):
        rows = np.nonzero(seq == b)[0]
        c = np.bincount(idx[rows].reshape(-1), minlength=E)
        out[rows] = aux_loss_backward(logits[rows], c, k, coeff, score, g / B, T_total=seq_len)
    return out


def accumulate_tokens_per_expert(acc: np.ndarray, counts: np.ndarray) -> np.ndarray:
    """Handbook §3.3 "Loss-free bias": the router keeps the token count of
    every expert in int64 and adds each micro-batch's counts to it."""
    return np.asarray(acc, dtype=np.int64) + np.asarray(counts, dtype=np.int64)


def expert_bias_update(tokens_per_expert: np.ndarray, bias: np.ndarray,
                       rate: float) -> np.ndarray:
    """Handbook §3.3 "Loss-free bias" (_update_router_expert_bias): every
    expert's bias moves by the update rate towards balance,
      bias += sign(total - count[e] * E) * rate,
    the comparison with the mean load made on the integers (count * E against
    the total), never on a floating-point mean."""
    c = [int(v) for v in np.asarray(tokens_per_expert).reshape(-1)]
    E = len(c)
    total = sum(c)
    direction = np.array([(total > v * E) - (total < v * E) for v in c], dtype=np.float64)
    return np.asarray(bias, dtype=np.float64) + direction * rate


# ----------------------------------------------------------------------------
# quantile balancing
# ----------------------------------------------------------------------------

def _kth_largest(values: np.ndarray, r: int) -> float:
    """The r-th largest entry (1-based) of a 1-D array, by a full sort."""
    return float(np.sort(values)[::-1][r - 1])


def quantile_route(logits: np.ndarray, beta: np.ndarray, k: int, score: str,
                   scaling: float = 1.0, solve: bool = True) -> Dict[str, np.ndarray]:
    """Handbook §3.3 "Load balancing", part "Quantile" (the quantile-balancing
    router): selection on the scores minus the per-expert quantile bias beta,
    top-(k+1) per token; the first k are the chosen experts and the (k+1)-th
    key is the token's threshold alpha. Each expert's local solution is the
    (col_target+1)-th largest of (score - alpha) over the micro-batch's
    tokens, col_target = T k / E (T k must be divisible by E).

    The router computes in fp32, so the rank decisions and the quantile are
    taken here on fp32 values: the scores rounded to fp32, then fp32
    subtractions (numpy float32 arithmetic rounds like the device). The
    mixing weights are those of the score function over the chosen experts:
    beta, like the expert bias, only selects.
    """
    T, E = logits.shape
    if not k < E:
        raise ValueError("quantile routing needs k < E (it ranks k + 1 experts)")
    s32 = scores(logits, score).astype(np.float32)
    v32 = s32 - beta.astype(np.float32)[None, :]
    order = np.argsort(-v32, axis=1, kind="stable")[:, :k + 1]
    idx = order[:, :k].astype(np.int64)
    alpha = v32[np.arange(T), order[:, k]]
    out = {"idx": idx, "alpha": alpha.astype(np.float64),
           "w": mixing_weights(logits, idx, score, scaling),
           "keys": v32.astype(np.float64), "gap": kth_gap(v32.astype(np.float64), k)}
    if solve:
        if (T * k) % E != 0:
            raise ValueError("quantile balancing needs T * k divisible by E")
        col_target = T * k // E
        d32 = s32 - alpha[:, None]
        out["beta_local"] = np.array([_kth_largest(d32[:, e], col_target + 1)
                                      for e in range(E)], dtype=np.float64)
    return out


def quantile_beta_update(beta: np.ndarray, accum: np.ndarray, count: int,
                         ema: float) -> np.ndarray:
    """Handbook §3.3 "Quantile": the micro-batches' solutions averaged
    (accum / max(count, 1)), mixed into the running beta by the EMA
    (ema * beta + (1 - ema) * average), then centred to zero mean."""
    local = np.asarray(accum, dtype=np.float64) / max(int(count), 1)
    nb = ema * np.asarray(beta, dtype=np.float64) + (1.0 - ema) * local
    return nb - nb.mean()


# ----------------------------------------------------------------------------
# whole layer, forward
# ----------------------------------------------------------------------------

def layer_forward(wl, inp: Dict[str, np.ndarray], idx=None) -> Dict[str, np.ndarray]:
    """S1..S7 for a workload `wl` (moe_inputs.Workload) on float64 inputs.

    `idx`: an optional given selection (see route)."""
    r = route(inp["x"], inp["w_router"], wl.k, wl.score, wl.scaling,
              inp.get("logit_bias"), inp.get("sel_bias"), idx=idx)
    act = act_of(wl)
    dsp = dispatch(r["idx"], wl.E)
    x_perm = permute_rows(inp["x"], dsp["src_tok"])
    ex = grouped_swiglu(x_perm, dsp["offsets"], inp["w1"], inp["w2"], act)
    out = dict(r)
    out.update(dsp)
    out["x_perm"] = x_perm
    out.update({"g": ex["g"], "u": ex["u"], "h": ex["h"], "out_perm": ex["out"]})
    y_s = None
    if inp.get("w1_s") is not None:
        # the shared expert is an MLP of the same configuration: same activation
        sh = swiglu_ffn(inp["x"], inp["w1_s"], inp["w2_s"], act)
        out.update({"g_s": sh["g"], "u_s": sh["u"], "h_s": sh["h"], "y_s": sh["out"]})
        y_s = sh["out"]
        if inp.get("w_gate_s") is not None:
            out["gate_s"] = shared_gate(inp["x"], inp["w_gate_s"])
            y_s = out["gate_s"][:, None] * y_s
    out["y"] = combine(ex["out"], dsp["row_of"], r["w"], y_s)
    out["aux"] = aux_loss(r["logits"], dsp["counts"], wl.k, wl.aux_coeff, wl.score)
    return out


# ----------------------------------------------------------------------------
# backward
# ----------------------------------------------------------------------------

def combine_backward(dy: np.ndarray, out_perm: np.ndarray, row_of: np.ndarray,
                     w: np.ndarray):
    """B6: d_out_perm[row_of[t,j]] = w[t,j] dy[t];  dw[t,j] = <dy[t], out_perm[row_of[t,j]]>."""
    T, k = row_of.shape
    d_out_perm = np.zeros_like(out_perm)
    dw = np.zeros((T, k))
    for j in range(k):
        rows = row_of[:, j]
        d_out_perm[rows] = w[:, j:j + 1] * dy
        dw[:, j] = np.sum(dy * out_perm[rows], axis=1)
    return d_out_perm, dw


def swiglu_ffn_backward(xs, w1, w2, g, u, h, d_out,
                        act: GluAct = SWIGLU, decide=None) -> Dict[str, np.ndarray]:
    """B5 + B4 for one expert: gradients of out = glu(g, u) @ w2.T, [g u] = xs @ w1.T.

    For SwiGLU d/dg silu(g) = sigmoid(g) * (1 + g * (1 - sigmoid(g))); the
    variants' derivatives are in glu_backward.
    """
    dh = d_out @ w2
    dW2 = d_out.T @ h
    dg, du = glu_backward(g, u, dh, act, decide)
    d_pre = np.concatenate([dg, du], axis=1)
    dxs = d_pre @ w1
    dW1 = d_pre.T @ xs
    return {"dh": dh, "d_pre": d_pre, "dxs": dxs, "dW1": dW1, "dW2": dW2}


def round_to(a: np.ndarray, act_dtype: str) -> np.ndarray:
    """a rounded to the layer's activation dtype (round to nearest even), back in float64."""
    import torch
    dt = torch.bfloat16 if act_dtype == "bf16" else torch.float32
    return torch.from_numpy(np.ascontiguousarray(a)).to(dt).double().numpy()


def clip_decisions(g, u, act: GluAct, act_dtype: str):
    """Where the SwiGLU clamp decides on the stored pre-activations: a bf16
    layer keeps gate|up in bf16 for the backward, so its clip decisions are
    taken on those values (the same precision on both sides of a check)."""
    if act.kind != "swiglu_clamp" or act_dtype != "bf16":
        return None
    return round_to(g, act_dtype), round_to(u, act_dtype)


def grouped_swiglu_backward(x_perm, offsets, w1, w2, g, u, h, d_out_perm, act: GluAct = SWIGLU,
                            act_dtype: str = "f32"):
    A, d = x_perm.shape
    E, twoF, _ = w1.shape
    d_pre = np.zeros((A, twoF))
    dx_perm = np.zeros((A, d))
    dW1 = np.zeros_like(w1)
    dW2 = np.zeros_like(w2)
    for e in range(E):
        r0, r1 = int(offsets[e]), int(offsets[e + 1])
        if r1 == r0:
            continue  # an expert with no rows has zero weight gradient
        res = swiglu_ffn_backward(x_perm[r0:r1], w1[e], w2[e], g[r0:r1], u[r0:r1],
                                  h[r0:r1], d_out_perm[r0:r1], act,
                                  clip_decisions(g[r0:r1], u[r0:r1], act, act_dtype))
        d_pre[r0:r1] = res["d_pre"]
        dx_perm[r0:r1] = res["dxs"]
        dW1[e] = res["dW1"]
        dW2[e] = res["dW2"]
    return {"d_pre": d_pre, "dx_perm": dx_perm, "dW1": dW1, "dW2": dW2}


def aux_loss_backward(logits, counts, k: int, coeff: float, score: str,
                      g_aux: float = 1.0, T_total: Optional[int] = None) -> np.ndarray:
    """B7: d(aux)/d(logits), counts held constant.

    dL/dP[t, e] = g * coeff * E * counts[e] / (k T^2). Softmax: d_logits =
    P * (dP - <P, dP>). Sigmoid reading (P = s / S): ds = (dP - <P, dP>) / S,
    d_logits = ds * s * (1 - s). `logits` may hold only some of the tokens;
    T_total is then the micro-batch's token count T.
    """
    n, E = logits.shape
    T = n if T_total is None else T_total
    dP = np.broadcast_to(g_aux * coeff * E * counts.astype(np.float64) / (k * T * T),
                         (n, E))
    if score in ("softmax", "softmax_pre"):
        P = softmax_rows(logits)
        return P * (dP - np.sum(P * dP, axis=1, keepdims=True))
    s = scores(logits, score)
    S = s.sum(axis=1, keepdims=True)
    P = s / S
    ds = (dP - np.sum(P * dP, axis=1, keepdims=True)) / S
    return ds * score_derivative(logits, score)


def scores_backward(logits, idx, dw, score: str, scaling: float) -> np.ndarray:
    """B2: d_logits from d(weights); zero for experts not chosen; no bias gradient.

    Softmax over the chosen logits: p = softmax(l_sel), w = c p,
      d l_sel = p * (c dw - <p, c dw>).
    Sigmoid / sqrt(softplus), k > 1: w = c s_sel / (S + eps), S = sum s_sel,
      d s_sel = c (dw - <dw, s_sel> / (S + eps)) / (S + eps), d l = d s * s'(l);
    k = 1: w = c s, d s = c dw.
    Pre-softmax: w_j = c P[idx_j] with P the softmax over all E, so every
    logit gets a gradient: d l_e = c P_e (g_e - sum_j P[idx_j] dw_j), where
    g_e = dw_j if e = idx_j and 0 otherwise.
    """
    T, E = logits.shape
    k = idx.shape[1]
    sel = np.take_along_axis(logits, idx, axis=1)
    if score == "softmax_pre":
        P = softmax_rows(logits)
        g = np.zeros((T, E))
        np.put_along_axis(g, idx, scaling * dw, axis=1)
        return P * (g - np.sum(np.take_along_axis(P, idx, axis=1) * scaling * dw, axis=1,
                               keepdims=True))
    if score == "softmax":
        p = softmax_rows(sel)
        gp = scaling * dw
        dsel = p * (gp - np.sum(p * gp, axis=1, keepdims=True))
    else:
        s = scores(sel, score)
        if k > 1:
            S = s.sum(axis=1, keepdims=True) + SIGMOID_RENORM_EPS
            ds = scaling * (dw - np.sum(dw * s, axis=1, keepdims=True) / S) / S
        else:
            ds = scaling * dw
        dsel = ds * score_derivative(sel, score)
    d_logits = np.zeros((T, E))
    np.put_along_axis(d_logits, idx, dsel, axis=1)
    return d_logits


def permute_backward(dx_perm: np.ndarray, row_of: np.ndarray) -> np.ndarray:
    """dx[t] = sum_j dx_perm[row_of[t, j]] (the transpose of the row copy)."""
    T, k = row_of.shape
    dx = np.zeros((T, dx_perm.shape[1]))
    for j in range(k):
        dx += dx_perm[row_of[:, j]]
    return dx


def layer_backward(wl, inp, fwd, dy: np.ndarray, g_aux: float = 1.0) -> Dict[str, np.ndarray]:
    """Gradients of  <dy, y> + g_aux * aux  w.r.t. x, the router and expert weights."""
    act = act_of(wl)
    d_out_perm, dw = combine_backward(dy, fwd["out_perm"], fwd["row_of"], fwd["w"])
    ex = grouped_swiglu_backward(fwd["x_perm"], fwd["offsets"], inp["w1"], inp["w2"],
                                 fwd["g"], fwd["u"], fwd["h"], d_out_perm, act, wl.act_dtype)
    d_logits = scores_backward(fwd["logits"], fwd["idx"], dw, wl.score, wl.scaling)
    d_logits = d_logits + aux_loss_backward(fwd["logits"], fwd["counts"], wl.k,
                                            wl.aux_coeff, wl.score, g_aux)
    dx = permute_backward(ex["dx_perm"], fwd["row_of"])
    dx = dx + d_logits @ inp["w_router"]
    out = {"d_out_perm": d_out_perm, "dw": dw, "d_pre": ex["d_pre"],
           "dx_perm": ex["dx_perm"], "dW1": ex["dW1"], "dW2": ex["dW2"],
           "d_logits": d_logits, "dW_r": d_logits.T @ inp["x"]}
    if inp.get("w1_s") is not None:
        dy_s = dy
        if inp.get("w_gate_s") is not None:
            gate = fwd["gate_s"]
            dy_s = gate[:, None] * dy
            d_gl = np.sum(dy * fwd["y_s"], axis=1) * gate * (1.0 - gate)
            out["d_gate_logit_s"] = d_gl
            out["dW_gate_s"] = d_gl @ inp["x"]
            dx = dx + d_gl[:, None] * inp["w_gate_s"][None, :]
        sh = swiglu_ffn_backward(inp["x"], inp["w1_s"], inp["w2_s"], fwd["g_s"],
                                 fwd["u_s"], fwd["h_s"], dy_s, act,
                                 clip_decisions(fwd["g_s"], fwd["u_s"], act, wl.act_dtype))
        out.update({"dW1_s": sh["dW1"], "dW2_s": sh["dW2"], "dx_s": sh["dxs"],
                    "d_pre_s": sh["d_pre"], "dy_s": dy_s})
        dx = dx + sh["dxs"]
    out["dx"] = dx
    return out


def layer_loss(wl, inp, dy: np.ndarray, g_aux: float = 1.0) -> float:
    """<dy, y> + g_aux * aux: the scalar whose gradient layer_backward returns."""
    f = layer_forward(wl, inp)
    return float(np.sum(dy * f["y"]) + g_aux * f["aux"])


# ----------------------------------------------------------------------------
# per-token and per-column evaluations, for checks at full size
# ----------------------------------------------------------------------------

def tokens_forward(wl, inp, tokens: Sequence[int], routing=None) -> Dict[str, np.ndarray]:
    """y (and the routing) of a few tokens, each computed on its own.

    The same definitions as layer_forward, applied to single rows: a token's
    output depends only on its own routing and the shared expert weights.
    `routing` (from route() on all tokens) may be given to reuse its idx/w.
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    x = inp["x"][tokens]
    if routing is None:
        r = route(x, inp["w_router"], wl.k, wl.score, wl.scaling,
                  inp.get("logit_bias"), inp.get("sel_bias"))
        idx, w = r["idx"], r["w"]
    else:
        idx, w = routing["idx"][tokens], routing["w"][tokens]
    act = act_of(wl)
    y = np.zeros((len(tokens), wl.d))
    for i in range(len(tokens)):
        for j in range(wl.k):
            res = swiglu_ffn(x[i:i + 1], inp["w1"][idx[i, j]], inp["w2"][idx[i, j]], act)
            y[i] += w[i, j] * res["out"][0]
    if inp.get("w1_s") is not None:
        y_s = swiglu_ffn(x, inp["w1_s"], inp["w2_s"], act)["out"]
        if inp.get("w_gate_s") is not None:
            y_s = shared_gate(x, inp["w_gate_s"])[:, None] * y_s
        y = y + y_s
    return {"idx": idx, "w": w, "y": y}


def tokens_backward(wl, inp, tokens: Sequence[int], routing, counts, dy_rows,
                    g_aux: float = 1.0) -> Dict[str, np.ndarray]:
    """dw, d_logits and dx of a few tokens, each computed on its own.

    Needs the routing of those tokens and the global counts (which enter the
    aux-loss gradient as constants).
    """
    tokens = np.asarray(tokens, dtype=np.int64)
    x = inp["x"][tokens]
    logits = routing["logits"][tokens]
    idx = routing["idx"][tokens]
    w = routing["w"][tokens]
    n = len(tokens)
    act = act_of(wl)
    dw = np.zeros((n, wl.k))
    dx = np.zeros((n, wl.d))
    for i in range(n):
        for j in range(wl.k):
            e = idx[i, j]
            f = swiglu_ffn(x[i:i + 1], inp["w1"][e], inp["w2"][e], act)
            dw[i, j] = float(np.sum(dy_rows[i] * f["out"][0]))
            b = swiglu_ffn_backward(x[i:i + 1], inp["w1"][e], inp["w2"][e], f["g"], f["u"],
                                    f["h"], w[i, j] * dy_rows[i:i + 1], act)
            dx[i] += b["dxs"][0]
    # the aux-loss gradient of a token needs its own logits, the global counts and T
    d_aux = aux_loss_backward(logits, counts, wl.k, wl.aux_coeff, wl.score, g_aux,
                              T_total=inp["x"].shape[0])
    d_logits = scores_backward(logits, idx, dw, wl.score, wl.scaling) + d_aux
    dx += d_logits @ inp["w_router"]
    if inp.get("w1_s") is not None:
        f = swiglu_ffn(x, inp["w1_s"], inp["w2_s"], act)
        dy_s = dy_rows
        if inp.get("w_gate_s") is not None:
            gate = shared_gate(x, inp["w_gate_s"])
            dy_s = gate[:, None] * dy_rows
            d_gl = np.sum(dy_rows * f["out"], axis=1) * gate * (1.0 - gate)
            dx += d_gl[:, None] * inp["w_gate_s"][None, :]
        b = swiglu_ffn_backward(x, inp["w1_s"], inp["w2_s"], f["g"], f["u"], f["h"], dy_s, act)
        dx += b["dxs"]
    return {"dw": dw, "d_logits": d_logits, "dx": dx}


def expert_grad_columns(x_rows, d_out_rows, w1_e, w2_e, cols: Sequence[int],
                        act: GluAct = SWIGLU) -> Dict[str, np.ndarray]:
    """Weight gradients of one expert restricted to FFN columns `cols`.

    The SwiGLU definitions separate per FFN column f: h[:, f] needs only gate
    row f and up row F+f of w1, and dW2[:, f], dW1[f, :], dW1[F+f, :] need only
    h[:, f] and column f of w2. So this is swiglu_ffn_backward on the weights
    sliced to those columns. Returns dW2_cols [d, n], dW1_gate [n, d],
    dW1_up [n, d].
    """
    cols = np.asarray(cols, dtype=np.int64)
    F = w2_e.shape[1]
    w1s = np.concatenate([w1_e[cols], w1_e[F + cols]], axis=0)
    w2s = w2_e[:, cols]
    f = swiglu_ffn(x_rows, w1s, w2s, act)
    b = swiglu_ffn_backward(x_rows, w1s, w2s, f["g"], f["u"], f["h"], d_out_rows, act)
    n = len(cols)
    return {"dW2_cols": b["dW2"], "dW1_gate": b["dW1"][:n], "dW1_up": b["dW1"][n:]}

