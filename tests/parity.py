"""Comparison helpers for the GPU-vs-oracle parity tests.

Bars (from the layer's parity contract):
  * expert indices and the permutation: bit-exact, except tokens whose k-th and
    (k+1)-th oracle keys differ by less than 1e-6 (near ties), which are
    reported and excluded;
  * floating point: max|gpu - ref| / max|ref| <= 1e-4 for quantities computed
    in fp32 from exact inputs, <= 2e-2 for anything downstream of bf16
    activations; the aux loss within 1e-5 relative.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import moe_oracle as O

NEAR_TIE = 1e-6
TOL_F32 = 1e-4
TOL_BF16 = 2e-2
TOL_AUX = 1e-5


def rel_err(gpu, ref) -> float:
    a = O.as_f64(gpu)
    r = np.asarray(ref, dtype=np.float64)
    assert a.shape == r.shape, (a.shape, r.shape)
    if a.size == 0:
        return 0.0
    den = float(np.max(np.abs(r)))
    num = float(np.max(np.abs(a - r)))
    if den == 0.0:
        return num
    return num / den


def assert_close(name, gpu, ref, tol):
    e = rel_err(gpu, ref)
    assert e <= tol, f"{name}: max|d|/max|ref| = {e:.3e} > {tol:.1e}"
    return e


def act_tol(wl):
    return TOL_F32 if wl.act_dtype == "f32" else TOL_BF16


def routing_checks(wl, b, f, report):
    """Indices bit-exact on decided tokens; permutation segments equal after
    removing the near-tie tokens; counts consistent with the permutation."""
    T, k, E = wl.T, wl.k, wl.E
    excl = f["gap"] < NEAR_TIE
    report["near_tie_tokens"] = int(excl.sum())
    g_idx = b["idx"].cpu().numpy().astype(np.int64)
    ok = ~excl
    mism = np.nonzero(np.any(g_idx[ok] != f["idx"][ok], axis=1))[0]
    assert mism.size == 0, f"top-k differs on {mism.size} decided tokens, e.g. {np.nonzero(ok)[0][mism[:5]]}"
    # every token's k experts are distinct and in range
    assert np.all((g_idx >= 0) & (g_idx < E))
    assert all(len(set(r)) == k for r in g_idx.tolist())
    g_counts = b["counts"].cpu().numpy().astype(np.int64)
    g_off = b["offsets"].cpu().numpy().astype(np.int64)
    g_row = b["row_of"].cpu().numpy().astype(np.int64)
    g_src = b["src_tok"].cpu().numpy().astype(np.int64)
    assert g_off[0] == 0 and g_off[-1] == T * k
    assert np.array_equal(np.diff(g_off), g_counts)
    # gpu permutation is a bijection consistent with its own idx
    assert np.array_equal(np.sort(g_row.ravel()), np.arange(T * k))
    assert np.array_equal(g_src[g_row], np.repeat(np.arange(T)[:, None], k, axis=1))
    for e in range(E):
        gseg = g_src[g_off[e]:g_off[e + 1]]
        oseg = f["src_tok"][f["offsets"][e]:f["offsets"][e + 1]]
        gseg = gseg[~excl[gseg]]
        oseg = oseg[~excl[oseg]]
        assert np.array_equal(gseg, oseg), f"expert {e}: permutation differs"
    if report["near_tie_tokens"] == 0:
        assert np.array_equal(g_counts, f["counts"])
        assert np.array_equal(g_off, f["offsets"])
        assert np.array_equal(g_row, f["row_of"])
        assert np.array_equal(g_src, f["src_tok"])
    return ok


def gpu_choice_on_near_ties(wl, b, f):
    """The selection to re-run the oracle on: the oracle's own on decided
    tokens, the GPU's on near-tie tokens, after checking that the GPU's choice
    there is one of the valid ones: k distinct experts, each with a key within
    the near-tie band of the oracle's k-th key, and no expert left out whose
    key beats a chosen one by more than the band."""
    keys = f["keys"]
    excl = f["gap"] < NEAR_TIE
    g_idx = b["idx"].cpu().numpy().astype(np.int64)
    idx = f["idx"].copy()
    k = wl.k
    for t in np.nonzero(excl)[0]:
        chosen = g_idx[t]
        assert len(set(chosen.tolist())) == k, f"token {t}: repeated expert"
        kth = np.sort(keys[t])[::-1][k - 1]
        ck = keys[t, chosen]
        assert np.all(ck >= kth - NEAR_TIE), f"token {t}: a chosen key lies below the band"
        left = np.setdiff1d(np.arange(wl.E), chosen)
        if left.size:
            assert keys[t, left].max() <= ck.min() + NEAR_TIE, f"token {t}: a better expert left out"
        # the chosen are sorted by descending key, up to the band
        assert np.all(np.diff(ck) <= NEAR_TIE), f"token {t}: selection not sorted"
        idx[t] = chosen
    return idx


def record(case, **kw):
    """One line of the run's parity summary (printed at the end of the session)."""
    REPORTS.append((case, kw))


REPORTS = []


def matched_rows(b, f, ok):
    """(gpu rows, oracle rows) of the assignments of the decided tokens."""
    g_row = b["row_of"].cpu().numpy().astype(np.int64)
    return g_row[ok].ravel(), f["row_of"][ok].ravel()


def to_np(t: torch.Tensor) -> np.ndarray:
    return O.as_f64(t)
