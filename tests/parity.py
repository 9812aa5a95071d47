"""Parity harness: runs the CUDA path and the fp64 oracle on the same seeded
inputs and compares them with the stated tolerances.

Tolerances:
  * topk_idx bit-exact, except near-tie tokens (a gap < 1e-6 between the
    sorted probabilities at or before slot k), which are counted;
  * y: max|y - y*| / rms(y*) <= 1e-4 (fp32), 2e-2 (bf16); for a near-tie
    token whose GPU selection differs, y* is recomputed with the GPU's
    selection (both answers are correct);
  * topk_w (alpha) within 1e-5 absolute of the oracle's, on tokens whose
    selection agrees;
  * aux_loss within 1e-5 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
from swiglu_mlp_top_gb300.inputs import make_inputs, to_f64

import os

Y_TOL = {"f32": 1e-4, "bf16": 2e-2}
ALPHA_TOL = 1e-5
AUX_TOL = 1e-5
TIE_GAP = 1e-6


def rel_err(y, ref):
    ref = np.asarray(ref, dtype=np.float64)
    y = np.asarray(y, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    return float(np.abs(y - ref).max() / rms) if ref.size else 0.0


def to_dev(inp, dev="cuda"):
    out = {}
    for n, v in inp.items():
        if v is None:
            out[n] = None
        elif isinstance(v, torch.Tensor):
            out[n] = v.to(dev)
        else:
            out[n] = [w.to(dev) for w in v]
    return out


def moe_inputs(T, H, I, E, dtype, seed=0, bias=None):
    return make_inputs(T, H, I, dtype, E=E, seed=seed, logit_bias=bias)


#: One entry per routing comparison of the session: the test, its token count,
#: the near-tie tokens (excluded from the bit-exact index check), how many of
#: those the GPU decided differently, and the largest errors.  The terminal
#: summary of the test run prints it (tests/conftest.py).
ROUTE_REPORT = []


def _current_test():
    return os.environ.get("PYTEST_CURRENT_TEST", "?").split(" ")[0]


def check_route(gpu_idx, gpu_w, gpu_aux, ref, k):
    """Compare routing outputs; returns (near-tie mask, mismatch mask).

    Every call is recorded in ROUTE_REPORT, and the assertion messages carry
    the near-tie count, so a failing or passing run shows how many tokens
    were excluded from the bit-exact check."""
    gpu_idx = np.asarray(gpu_idx)
    tie = oracle.near_tie_tokens(ref["probs"], k, TIE_GAP)
    diff = (gpu_idx != ref["topk_idx"]).any(axis=-1)
    bad = diff & ~tie
    n_tie, n_flip = int(tie.sum()), int((diff & tie).sum())
    agree = ~diff
    w_err = float(np.abs(np.asarray(gpu_w)[agree] - ref["topk_w"][agree]).max()) if agree.any() else 0.0
    aux_err = abs(float(gpu_aux) - ref["aux_loss"])
    entry = {"test": _current_test(), "tokens": int(gpu_idx.shape[0]), "near_ties": n_tie,
             "near_tie_flips": n_flip, "idx_mismatch_non_tie": int(bad.sum()),
             "topk_w_err": w_err, "aux_err": aux_err}
    ROUTE_REPORT.append(entry)
    tag = f"[{n_tie} near-tie tokens, {n_flip} decided differently]"
    assert not bad.any(), (f"topk_idx differs on {int(bad.sum())} non-tie tokens, "
                           f"e.g. {np.nonzero(bad)[0][:5]} {tag}")
    assert w_err <= ALPHA_TOL, f"topk_w err {w_err} {tag}"
    assert aux_err <= AUX_TOL, (float(gpu_aux), ref["aux_loss"], tag)
    return tie, diff


def ref_y_rows(inp64, ref, gpu_idx, rows, k):
    """Oracle y for `rows`, using the GPU's selection on rows where it differs
    (near-ties) — alpha recomputed from the oracle's probabilities."""
    gpu_idx = np.asarray(gpu_idx)
    sel = ref["topk_idx"][rows].copy()
    diff = (gpu_idx[rows] != sel).any(axis=-1)
    sel[diff] = gpu_idx[rows][diff]
    p = ref["probs"][rows]
    val = np.take_along_axis(p, sel.astype(np.int64), axis=-1)
    alpha = oracle.renormalise(val)
    return oracle.combine(inp64["x"][rows], inp64["Wg"], inp64["Wu"], inp64["Wd"], sel, alpha)


def inputs64(inp):
    return {n: to_f64(v) for n, v in inp.items()}
