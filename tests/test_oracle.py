"""Pins for the fp64 oracle against values the pages print and against
mathematics that fixes the result independently of the oracle's own code.

Each test names the passage (page title + section) or the identity it uses.
"""
import itertools
import json
import math
import os

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rng(seed=0):
    return np.random.default_rng(seed)


# --------------------------------------------------------------------------
# SiLU
# --------------------------------------------------------------------------
def test_silu_printed_values():
    """Demo example 2: SiLU(0) = 0; minimum near -1.278 with value -0.278."""
    g = golden("silu_values.json")
    assert O.silu(0.0) == g["silu_at_zero"]
    # locate the minimum of the oracle's SiLU by golden-section search
    a, b = -3.0, 0.0
    phi = (math.sqrt(5) - 1) / 2
    for _ in range(200):
        c, d = b - phi * (b - a), a + phi * (b - a)
        if O.silu(c) < O.silu(d):
            b = d
        else:
            a = c
    xmin = 0.5 * (a + b)
    tol = 0.5 * 10 ** -g["printed_decimals"]
    assert abs(xmin - g["argmin_approx"]) <= tol
    assert abs(float(O.silu(xmin)) - g["min_approx"]) <= tol
    # closed form at the minimum: d/dx x*s(x) = s(x)(1 + x(1 - s(x))) = 0
    # -> x(1 - s(x)) = -1 -> SiLU(x*) = x* * s(x*) = x* + 1.  Solve the
    # stationarity condition by bisection (s from its definition, not the oracle).
    s = lambda v: 1.0 / (1.0 + math.exp(-v))
    lo, hi = -2.0, -1.0                      # x(1-s(x)) + 1 changes sign here
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        if mid * (1 - s(mid)) + 1 > 0:     # f(-2) < 0 < f(-1)
            hi = mid
        else:
            lo = mid
    xstar = 0.5 * (lo + hi)
    assert abs(xstar - xmin) < 1e-6
    assert abs(float(O.silu(xstar)) - (xstar + 1.0)) < 1e-14
    assert O.silu(xstar - 1e-4) > O.silu(xstar) < O.silu(xstar + 1e-4)


def test_silu_asymptotes_and_sign():
    z = np.array([30.0, 50.0, -30.0, -50.0, 1.0, -1.0])
    s = O.silu(z)
    assert abs(s[0] - 30.0) < 1e-9 and abs(s[1] - 50.0) < 1e-12
    assert -1e-11 < s[2] < 0 and -1e-20 < s[3] < 0
    # SiLU(1) = e/(1+e); SiLU(-1) = -1/(1+e)
    assert abs(s[4] - math.e / (1 + math.e)) < 1e-15
    assert abs(s[5] + 1.0 / (1 + math.e)) < 1e-15
    # no overflow for very negative arguments
    assert O.silu(-1000.0) == 0.0


# --------------------------------------------------------------------------
# Dense SwiGLU FFN
# --------------------------------------------------------------------------
def test_swiglu_hand_case():
    """Lesson 13 §0/§1.2 equations, evaluated by hand (H=2, I=3)."""
    g = golden("swiglu_hand_case.json")
    y = O.swiglu_ffn(np.array([g["x"]]), np.array(g["Wg"]), np.array(g["Wu"]),
                     np.array(g["Wd"]))
    e = math.e
    expect = [eval(s, {"e": e}) for s in g["y_closed_form"]]
    assert y.shape == (1, 2)
    np.testing.assert_allclose(y[0], expect, rtol=0, atol=1e-15)


def test_swiglu_zero_gate_or_value_gives_zero():
    r = rng(1)
    x = r.normal(size=(5, 6))
    Wg, Wu, Wd = r.normal(size=(7, 6)), r.normal(size=(7, 6)), r.normal(size=(6, 7))
    assert np.all(O.swiglu_ffn(x, np.zeros_like(Wg), Wu, Wd) == 0)   # SiLU(0) = 0
    assert np.all(O.swiglu_ffn(x, Wg, np.zeros_like(Wu), Wd) == 0)


def test_swiglu_linear_in_down_and_up():
    r = rng(2)
    x = r.normal(size=(4, 6))
    Wg, Wu = r.normal(size=(9, 6)), r.normal(size=(9, 6))
    D1, D2 = r.normal(size=(6, 9)), r.normal(size=(6, 9))
    y = O.swiglu_ffn(x, Wg, Wu, D1 + 3.0 * D2)
    np.testing.assert_allclose(y, O.swiglu_ffn(x, Wg, Wu, D1) + 3.0 * O.swiglu_ffn(x, Wg, Wu, D2),
                               atol=1e-11)
    U2 = r.normal(size=(9, 6))
    y = O.swiglu_ffn(x, Wg, Wu - 2.0 * U2, D1)
    np.testing.assert_allclose(y, O.swiglu_ffn(x, Wg, Wu, D1) - 2.0 * O.swiglu_ffn(x, Wg, U2, D1),
                               atol=1e-11)


def test_swiglu_token_permutation_equivariance():
    """The FFN acts on each position independently (lesson 13 §1.1)."""
    r = rng(3)
    x = r.normal(size=(11, 5))
    W = (r.normal(size=(8, 5)), r.normal(size=(8, 5)), r.normal(size=(5, 8)))
    perm = r.permutation(11)
    np.testing.assert_allclose(O.swiglu_ffn(x[perm], *W), O.swiglu_ffn(x, *W)[perm], atol=1e-13)


def test_swiglu_large_gate_is_bilinear():
    """For g >> 0, SiLU(g) -> g, so y -> Wd((Wg x) * (Wu x)) (elementwise)."""
    x = np.array([[1.0, 2.0]])
    Wg = np.array([[40.0, 0.0], [0.0, 30.0], [20.0, 20.0]])   # g = [40, 60, 60]
    Wu = np.array([[1.0, -1.0], [0.5, 0.0], [0.0, 2.0]])      # u = [-1, 0.5, 4]
    Wd = np.array([[1.0, 2.0, 3.0], [-1.0, 0.0, 1.0]])
    h = np.array([40.0 * -1.0, 60.0 * 0.5, 60.0 * 4.0])
    np.testing.assert_allclose(O.swiglu_ffn(x, Wg, Wu, Wd)[0], Wd @ h, rtol=1e-14)


# --------------------------------------------------------------------------
# Router, top-k, renormalisation
# --------------------------------------------------------------------------
def _logits_for_probs(p, H=6):
    """x = e_0, Wr[:, 0] = log p  ->  r = log p  ->  softmax(r) = p exactly (up to rounding)."""
    E = len(p)
    x = np.zeros((1, H))
    x[0, 0] = 1.0
    Wr = np.zeros((E, H))
    Wr[:, 0] = np.log(p)
    return x, Wr


@pytest.mark.parametrize("via", ["weights", "bias", "noise"])
def test_routing_worked_example(via):
    """Lesson 13 §1.5: p = [0.05, 0.10, 0.80, 0.05]."""
    g = golden("routing_worked_example.json")
    p = np.array(g["p"])
    if via == "weights":
        x, Wr = _logits_for_probs(p)
        bias = None
    elif via == "bias":
        x, Wr, bias = np.ones((1, 3)), np.zeros((4, 3)), np.log(p)
    noise = None
    if via == "noise":                         # the logits arrive as router noise
        x, Wr, bias, noise = np.ones((1, 3)), np.zeros((4, 3)), None, np.log(p)[None, :]
    probs = O.softmax(O.router_logits(x, Wr, bias, noise))
    np.testing.assert_allclose(probs[0], p, rtol=1e-14)
    for key, k in (("top1", 1), ("top2", 2)):
        r = O.moe_route(x, Wr, k, 0.0, bias, noise)
        assert r["topk_idx"][0].tolist() == g[key]["idx"]
        np.testing.assert_allclose(r["topk_w"][0], g[key]["alpha"], rtol=1e-14)


def test_softmax_properties():
    r = rng(4)
    logits = r.normal(size=(7, 5)) * 3
    p = O.softmax(logits)
    np.testing.assert_allclose(p.sum(-1), 1.0, atol=1e-15)
    np.testing.assert_allclose(O.softmax(logits + 123.0), p, atol=1e-15)
    # two experts: p_0 = sigmoid(r_0 - r_1)
    two = O.softmax(np.array([[0.7, -0.4]]))
    assert abs(two[0, 0] - 1.0 / (1.0 + math.exp(-1.1))) < 1e-15
    assert np.all(O.softmax(np.zeros((2, 6))) == 1.0 / 6)
    # large logits do not overflow
    assert np.all(np.isfinite(O.softmax(np.array([[1000.0, 0.0, -1000.0]]))))


def _bruteforce_topk(p_row, k):
    """The unique k-subset whose members all precede every non-member in the
    order (descending p, then ascending index); slots ordered the same way."""
    E = len(p_row)
    before = lambda a, b: (p_row[a] > p_row[b]) or (p_row[a] == p_row[b] and a < b)
    hits = [S for S in itertools.combinations(range(E), k)
            if all(before(a, b) for a in S for b in range(E) if b not in S)]
    assert len(hits) == 1
    S = list(hits[0])
    # order the slots by insertion sort with the same comparison
    out = []
    for a in S:
        i = 0
        while i < len(out) and before(out[i], a):
            i += 1
        out.insert(i, a)
    return out


@pytest.mark.parametrize("seed", range(6))
def test_topk_vs_bruteforce(seed):
    r = rng(10 + seed)
    E = int(r.integers(1, 7))
    p = O.softmax(r.normal(size=(9, E)))
    # plant exact ties in some rows
    if E >= 3:
        p[0, 1] = p[0, 2]
        p[1, :] = p[1, 0]
    for k in range(1, E + 1):
        idx, val = O.topk(p, k)
        for t in range(p.shape[0]):
            assert idx[t].tolist() == _bruteforce_topk(p[t], k)
            assert val[t].tolist() == [p[t, e] for e in idx[t]]
        # the selected values are the k largest, in descending order
        np.testing.assert_array_equal(val, -np.sort(-p, axis=-1)[:, :k])


def test_topk_rejects_bad_k():
    with pytest.raises(ValueError):
        O.topk(np.ones((2, 3)), 0)
    with pytest.raises(ValueError):
        O.topk(np.ones((2, 3)), 4)


@pytest.mark.parametrize("E,k", [(4, 1), (4, 2), (8, 2), (8, 3), (5, 5)])
def test_tie_break_uniform_router(E, k):
    """Wr = 0 -> every p = 1/E exactly -> experts 0..k-1, alpha = 1/k."""
    x = rng(5).normal(size=(6, 7))
    r = O.moe_route(x, np.zeros((E, 7)), k, 0.01)
    assert np.all(r["probs"] == 1.0 / E)
    assert np.all(r["topk_idx"] == np.arange(k)[None, :])
    np.testing.assert_allclose(r["topk_w"], 1.0 / k, rtol=1e-15)


def test_alpha_sums_to_one_and_k1_is_one():
    """Demo example 6: renormalised top-k weights sum to 1 (atol 1e-5 there)."""
    r = rng(6)
    x, Wr = r.normal(size=(50, 8)), r.normal(size=(6, 8))
    for k in (1, 2, 3, 6):
        a = O.moe_route(x, Wr, k, 0.0)["topk_w"]
        np.testing.assert_allclose(a.sum(-1), 1.0, atol=1e-15)
        assert np.all(a > 0)
        assert np.all(np.diff(a, axis=-1) <= 0)         # descending like p
    assert np.all(O.moe_route(x, Wr, 1, 0.0)["topk_w"] == 1.0)


# --------------------------------------------------------------------------
# aux loss
# --------------------------------------------------------------------------
def test_aux_extremes_table():
    """Chapter 4 §4.4 table: balanced -> 0.25 (x E = 1.0); collapsed -> 0.7 (x E = 2.8)."""
    g = golden("aux_loss_tables.json")
    for row in g["extremes"]:
        E = len(row["load"])
        s = O.aux_loss_from_stats(row["load"], row["prob"], 1, 1.0)
        assert abs(s - row["sum_f_P"]) < 1e-15
        assert abs(O.aux_loss_from_stats(row["load"], row["prob"], E, 1.0) - row["times_E"]) < 1e-14


def test_load_example():
    """Chapter 4 §4.4 step 1: 30 of 100 tokens on expert 0 -> load 0.3."""
    g = golden("aux_loss_tables.json")["load_example"]
    idx = np.array([0] * g["count_expert0"] + [1] * (g["T"] - g["count_expert0"]))[:, None]
    load, counts = O.expert_load(idx, g["E"])
    assert counts[0] == g["count_expert0"]
    assert load[0] == g["load_expert0"]


@pytest.mark.parametrize("E,k", [(4, 1), (8, 2), (6, 3)])
def test_aux_uniform_router_is_k_coef(E, k):
    """Wr = 0: load = 1 on experts 0..k-1, prob = 1/E  ->  aux = E*coef*k/E = k*coef."""
    x = rng(7).normal(size=(12, 5))
    coef = 0.01
    r = O.moe_route(x, np.zeros((E, 5)), k, coef)
    assert abs(r["aux_loss"] - k * coef) < 1e-17


@pytest.mark.parametrize("E", [2, 4, 8])
def test_aux_uniform_top1_load_is_coef(E):
    """Exactly uniform top-1 counts (count_e = T/E) give aux = coef whatever
    the probabilities: E*coef*sum_e (1/E) P_e = coef * sum_e P_e = coef."""
    H = E + 3
    T = 5 * E
    r = rng(8)
    Wr = np.zeros((E, H))
    Wr[:, :E] = 4.0 * np.eye(E)
    Wr[:, E:] = r.normal(size=(E, 3)) * 0.1          # perturb the probabilities
    x = np.zeros((T, H))
    for t in range(T):
        x[t, t % E] = 1.0
        x[t, E:] = r.normal(size=3)
    coef = 0.01
    out = O.moe_route(x, Wr, 1, coef)
    assert np.bincount(out["topk_idx"][:, 0], minlength=E).tolist() == [T // E] * E
    assert abs(out["aux_loss"] - coef) < 1e-15


def test_aux_coef_zero_is_zero():
    r = rng(9)
    out = O.moe_route(r.normal(size=(10, 4)), r.normal(size=(3, 4)), 2, 0.0)
    assert out["aux_loss"] == 0.0


def test_aux_loss_wrapper_extremes_table():
    """aux_loss(topk_idx, p, coef) on selections and probabilities built to
    give chapter 4 §4.4's two rows (E = 4, top-1, coef = 1): balanced load and
    mean probability 1/4 -> 1.0; every token on expert 0 with mean
    probabilities (0.7, 0.1, 0.1, 0.1) -> 2.8."""
    g = golden("aux_loss_tables.json")
    bal, col = g["extremes"]
    T = 8
    idx = (np.arange(T) % 4)[:, None]                         # 2 tokens per expert
    p = np.full((T, 4), 0.25)
    assert abs(O.aux_loss(idx, p, 1.0) - bal["times_E"]) < 1e-14
    idx = np.zeros((T, 1), dtype=np.int64)                     # collapsed on expert 0
    p = np.tile(np.array(col["prob"]), (T, 1))
    p[:4] += np.array([0.1, -0.1, 0.0, 0.0])                   # rows differ, the mean does not
    p[4:] -= np.array([0.1, -0.1, 0.0, 0.0])
    assert abs(O.aux_loss(idx, p, 1.0) - col["times_E"]) < 1e-14


def test_aux_loss_wrapper_counts_every_slot_and_every_expert():
    """k = 2 with a uniform router: load_e = count_e / T summed over both slots
    (sum_e load_e = k), prob_e = 1/E, so aux = E*coef*k/E = k*coef (lesson 13
    §1.6 / step 6 summed [k, E] one-hot mean).  The highest expert is never
    selected: E must come from the probabilities, not from the indices."""
    E, k, T, coef = 6, 2, 10, 0.01
    idx = np.tile(np.arange(k), (T, 1))                        # experts 0, 1 only
    p = np.full((T, E), 1.0 / E)
    assert abs(O.aux_loss(idx, p, coef) - k * coef) < 1e-17
    # agrees with the routing path's own value on a random router
    r = rng(10)
    x, Wr = r.normal(size=(T, 7)), r.normal(size=(E, 7))
    out = O.moe_route(x, Wr, k, coef)
    assert abs(O.aux_loss(out["topk_idx"], out["probs"], coef) - out["aux_loss"]) < 1e-17


# --------------------------------------------------------------------------
# MoE layer: special cases that reduce to known forms
# --------------------------------------------------------------------------
def _experts(r, E, H, I, scale=0.3):
    return ([r.normal(size=(I, H)) * scale for _ in range(E)],
            [r.normal(size=(I, H)) * scale for _ in range(E)],
            [r.normal(size=(H, I)) * scale for _ in range(E)])


def test_k_equals_E_is_dense_softmax_mixture():
    """k = E: alpha = p, so y_t = sum_e p_{t,e} FFN_e(x_t); load_e = 1 -> aux = E*coef."""
    r = rng(11)
    T, H, I, E = 7, 5, 6, 4
    x, Wr = r.normal(size=(T, H)), r.normal(size=(E, H))
    Wg, Wu, Wd = _experts(r, E, H, I)
    out = O.moe_forward(x, Wr, Wg, Wu, Wd, E, 0.02)
    p = out["probs"]
    mix = sum(p[:, e:e + 1] * O.swiglu_ffn(x, Wg[e], Wu[e], Wd[e]) for e in range(E))
    np.testing.assert_allclose(out["y"], mix, atol=1e-13)
    assert abs(out["aux_loss"] - E * 0.02) < 1e-15


def test_single_expert_is_dense_ffn():
    """E = 1: alpha = 1, y = FFN(x), aux = coef."""
    r = rng(12)
    x = r.normal(size=(6, 5))
    Wg, Wu, Wd = _experts(r, 1, 5, 7)
    out = O.moe_forward(x, r.normal(size=(1, 5)), Wg, Wu, Wd, 1, 0.05)
    np.testing.assert_allclose(out["y"], O.swiglu_ffn(x, Wg[0], Wu[0], Wd[0]), rtol=1e-12, atol=1e-15)
    assert abs(out["aux_loss"] - 0.05) < 1e-16


@pytest.mark.parametrize("k", [1, 2, 3])
def test_identical_experts_give_dense(k):
    """All experts equal: y = sum_S alpha * FFN(x) = FFN(x) since sum alpha = 1."""
    r = rng(13)
    x = r.normal(size=(9, 5))
    Wg, Wu, Wd = _experts(r, 1, 5, 6)
    E = 4
    out = O.moe_forward(x, r.normal(size=(E, 5)), Wg * E, Wu * E, Wd * E, k, 0.0)
    np.testing.assert_allclose(out["y"], O.swiglu_ffn(x, Wg[0], Wu[0], Wd[0]), atol=1e-13)


def test_expert_routing_selects_the_right_expert():
    """A token routed (top-1) to expert e gets exactly FFN_e(x_t)."""
    r = rng(14)
    T, H, I, E = 8, 6, 5, 4
    Wr = np.zeros((E, H))
    Wr[:, :E] = 10.0 * np.eye(E)
    x = r.normal(size=(T, H)) * 0.1
    route = [3, 0, 2, 2, 1, 3, 0, 1]
    for t, e in enumerate(route):
        x[t, e] = 1.0
    Wg, Wu, Wd = _experts(r, E, H, I)
    out = O.moe_forward(x, Wr, Wg, Wu, Wd, 1, 0.0)
    assert out["topk_idx"][:, 0].tolist() == route
    for t, e in enumerate(route):
        np.testing.assert_allclose(out["y"][t], O.swiglu_ffn(x[t:t + 1], Wg[e], Wu[e], Wd[e])[0],
                                   rtol=1e-12, atol=1e-15)


def _bruteforce_moe(x, Wr, Wg, Wu, Wd, k, coef, bias=None):
    """Per-token scalar loops in Python floats (fp64)."""
    T, H = len(x), len(x[0])
    E, I = len(Wr), len(Wg[0])
    y = [[0.0] * H for _ in range(T)]
    idx_all, a_all = [], []
    count = [0] * E
    psum = [0.0] * E
    for t in range(T):
        logit = [sum(Wr[e][j] * x[t][j] for j in range(H)) + (bias[e] if bias is not None else 0.0)
                 for e in range(E)]
        m = max(logit)
        ex = [math.exp(v - m) for v in logit]
        z = sum(ex)
        p = [v / z for v in ex]
        S = _bruteforce_topk(p, k)
        denom = sum(p[e] for e in S) + 1e-20
        alpha = [p[e] / denom for e in S]
        idx_all.append(S)
        a_all.append(alpha)
        for e in range(E):
            psum[e] += p[e]
        for e, a in zip(S, alpha):
            count[e] += 1
            hvec = []
            for i in range(I):
                g = sum(Wg[e][i][j] * x[t][j] for j in range(H))
                u = sum(Wu[e][i][j] * x[t][j] for j in range(H))
                hvec.append(g / (1.0 + math.exp(-g)) * u)
            for o in range(H):
                y[t][o] += a * sum(Wd[e][o][i] * hvec[i] for i in range(I))
    aux = E * coef * sum((count[e] / T) * (psum[e] / T) for e in range(E))
    return np.array(y), np.array(idx_all), np.array(a_all), aux


@pytest.mark.parametrize("seed,E,k,with_bias", [(0, 3, 1, False), (1, 3, 2, False),
                                                (2, 5, 2, True), (3, 4, 3, False)])
def test_moe_bruteforce_tiny(seed, E, k, with_bias):
    r = rng(20 + seed)
    T, H, I = 6, 4, 5
    x, Wr = r.normal(size=(T, H)), r.normal(size=(E, H))
    Wg, Wu, Wd = _experts(r, E, H, I, scale=0.5)
    bias = r.normal(size=E) if with_bias else None
    out = O.moe_forward(x, Wr, Wg, Wu, Wd, k, 0.03, bias)
    y, idx, a, aux = _bruteforce_moe(x.tolist(), Wr.tolist(), [w.tolist() for w in Wg],
                                     [w.tolist() for w in Wu], [w.tolist() for w in Wd],
                                     k, 0.03, None if bias is None else bias.tolist())
    np.testing.assert_array_equal(out["topk_idx"], idx)
    np.testing.assert_allclose(out["topk_w"], a, atol=1e-15)
    np.testing.assert_allclose(out["y"], y, atol=1e-13)
    assert abs(out["aux_loss"] - aux) < 1e-15


def test_moe_token_permutation_equivariance():
    r = rng(30)
    T, H, I, E = 10, 4, 6, 5
    x, Wr = r.normal(size=(T, H)), r.normal(size=(E, H))
    Wg, Wu, Wd = _experts(r, E, H, I)
    perm = r.permutation(T)
    a = O.moe_forward(x, Wr, Wg, Wu, Wd, 2, 0.01)
    b = O.moe_forward(x[perm], Wr, Wg, Wu, Wd, 2, 0.01)
    np.testing.assert_allclose(b["y"], a["y"][perm], atol=1e-13)
    np.testing.assert_array_equal(b["topk_idx"], a["topk_idx"][perm])
    assert abs(a["aux_loss"] - b["aux_loss"]) < 1e-16


def test_near_tie_detection():
    p = np.array([[0.5, 0.3, 0.2],
                  [0.4, 0.4 - 5e-7, 0.2 + 5e-7],      # slot-order tie at j = 1
                  [0.6, 0.2, 0.2 - 1e-9 + 1e-9],       # exact tie at the k/k+1 boundary
                  [0.6, 0.3, 0.1]])
    m1 = O.near_tie_tokens(p, 1)
    m2 = O.near_tie_tokens(p, 2)
    assert m1.tolist() == [False, True, False, False]
    assert m2.tolist() == [False, True, True, False]
    assert O.near_tie_tokens(p, 3).tolist() == m2.tolist()


def test_config_intermediate_size():
    """Chapter 4 §4.1: I = ceil(768 * pi / 64) * 64 = 2432."""
    from swiglu_mlp_top_gb300.inputs import intermediate_size
    g = golden("minimind_config.json")
    assert intermediate_size(g["hidden_size"]) == g["intermediate_size"]


# --------------------------------------------------------------------------
# Router variants (p-chao.com note 08 §10 table: router noise, z-loss)
# --------------------------------------------------------------------------
def _lse_bruteforce(row):
    """log of the plain sum of exponentials (no maximum taken out), summed
    exactly with math.fsum: fine for the small logits it is used on."""
    return math.log(math.fsum(math.exp(v) for v in row))


def test_logsumexp_closed_forms():
    # two experts: log(e^a + e^b); all-equal logits c: c + log E
    for a, b in ((0.3, -1.2), (2.0, 2.0), (-5.0, 1.0)):
        assert abs(O.logsumexp(np.array([[a, b]]))[0] - math.log(math.exp(a) + math.exp(b))) < 1e-15
    for E, c in ((1, 0.7), (4, 0.0), (8, -3.0)):
        assert abs(O.logsumexp(np.full((1, E), c))[0] - (c + math.log(E))) < 1e-14
    # a dominant logit: lse = max + log(1 + e^{-1000}) = 1000 exactly in fp64
    # (a plain exp of the logits would overflow)
    assert O.logsumexp(np.array([[1000.0, 0.0]]))[0] == 1000.0


def test_logsumexp_bruteforce():
    r = rng(11).normal(size=(9, 6)) * 2
    for t in range(r.shape[0]):
        assert abs(O.logsumexp(r[t:t + 1])[0] - _lse_bruteforce(r[t].tolist())) < 1e-13


def test_z_loss_closed_forms():
    """Uniform router (Wr = 0): lse = log E for every token, so
    L_z = z_coef (log E)^2; one expert: lse = r, L_z = z_coef mean r^2;
    z_coef = 0 gives 0."""
    x = rng(12).normal(size=(10, 5))
    for E in (2, 4, 8):
        out = O.moe_route(x, np.zeros((E, 5)), 1, 0.0, z_coef=1e-3)
        assert abs(out["z_loss"] - 1e-3 * math.log(E) ** 2) < 1e-17
    Wr = rng(13).normal(size=(1, 5))
    r = x @ Wr.T
    assert abs(O.z_loss(r, 0.5) - 0.5 * float(np.mean(r[:, 0] ** 2))) < 1e-14
    assert O.moe_route(x, rng(14).normal(size=(4, 5)), 2, 0.01)["z_loss"] == 0.0


def test_z_loss_bruteforce():
    r = rng(15).normal(size=(7, 5))
    ref = 0.02 * math.fsum(_lse_bruteforce(r[t].tolist()) ** 2 for t in range(7)) / 7
    assert abs(O.z_loss(r, 0.02) - ref) < 1e-15


def test_noise_equal_rows_is_a_logit_bias():
    """Noise that is the same vector b for every token routes exactly as
    logit_bias = b (two independent code paths of the oracle)."""
    r = rng(16)
    x, Wr = r.normal(size=(20, 6)), r.normal(size=(5, 6)) * 0.5
    b = r.normal(size=5)
    a = O.moe_route(x, Wr, 2, 0.01, logit_bias=b, z_coef=1e-2)
    n = O.moe_route(x, Wr, 2, 0.01, logit_noise=np.tile(b, (20, 1)), z_coef=1e-2)
    for key in ("topk_idx", "topk_w", "probs", "lse"):
        np.testing.assert_allclose(a[key], n[key], rtol=0, atol=1e-15)
    assert abs(a["aux_loss"] - n["aux_loss"]) < 1e-17 and abs(a["z_loss"] - n["z_loss"]) < 1e-16


def test_per_token_constant_noise_moves_only_the_partition_function():
    """Softmax is shift invariant: noise c_t on every expert of token t leaves
    p, the selection, alpha and aux unchanged and moves lse_t by c_t."""
    r = rng(17)
    x, Wr = r.normal(size=(12, 4)), r.normal(size=(6, 4))
    c = r.normal(size=12)
    a = O.moe_route(x, Wr, 3, 0.01, z_coef=1.0)
    n = O.moe_route(x, Wr, 3, 0.01, logit_noise=np.repeat(c[:, None], 6, axis=1), z_coef=1.0)
    np.testing.assert_allclose(n["probs"], a["probs"], rtol=1e-13)
    assert np.array_equal(n["topk_idx"], a["topk_idx"])
    np.testing.assert_allclose(n["lse"], a["lse"] + c, rtol=0, atol=1e-13)
    assert abs(n["z_loss"] - float(np.mean((a["lse"] + c) ** 2))) < 1e-13


def test_noise_changes_the_choice():
    """A noise large enough on one expert takes top-1 for every token."""
    r = rng(18)
    x, Wr = r.normal(size=(8, 4)), r.normal(size=(5, 4)) * 0.1
    noise = np.zeros((8, 5))
    noise[:, 3] = 50.0
    out = O.moe_route(x, Wr, 1, 0.0, logit_noise=noise)
    assert (out["topk_idx"][:, 0] == 3).all()


# --------------------------------------------------------------------------
# Backward pass: finite differences of the oracle's own forward (itself
# pinned above) and the special cases the pages fix
# --------------------------------------------------------------------------
def _fd_grad(f, a, eps=1e-5):
    """Central differences of the scalar f() with respect to every element of a."""
    g = np.zeros_like(a)
    it = np.nditer(a, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = a[i]
        a[i] = old + eps
        fp = f()
        a[i] = old - eps
        fm = f()
        a[i] = old
        g[i] = (fp - fm) / (2 * eps)
    return g


def test_swiglu_backward_finite_differences():
    r = rng(30)
    x, dy = r.normal(size=(3, 4)), r.normal(size=(3, 4))
    Wg, Wu, Wd = r.normal(size=(5, 4)), r.normal(size=(5, 4)), r.normal(size=(4, 5))
    loss = lambda: float(np.sum(dy * O.swiglu_ffn(x, Wg, Wu, Wd)))
    dx, dWg, dWu, dWd = O.swiglu_ffn_backward(x, Wg, Wu, Wd, dy)
    for got, a in ((dx, x), (dWg, Wg), (dWu, Wu), (dWd, Wd)):
        np.testing.assert_allclose(got, _fd_grad(loss, a), rtol=0, atol=1e-7)


def _moe_case(seed, T=6, H=5, I=4, E=4):
    r = rng(seed)
    return (r.normal(size=(T, H)), r.normal(size=(E, H)) * 0.7,
            [r.normal(size=(I, H)) for _ in range(E)], [r.normal(size=(I, H)) for _ in range(E)],
            [r.normal(size=(H, I)) for _ in range(E)], r.normal(size=(T, H)))


@pytest.mark.parametrize("k,with_noise", [(1, False), (2, False), (2, True), (3, True)])
def test_moe_backward_finite_differences(k, with_noise):
    """dL/d(every input) for L = <dy, y> + d_aux aux + d_z z: the router's
    gradient through alpha, P_e and lse, the experts' through alpha dy."""
    coef, zc, d_aux, d_z = 0.05, 0.02, 1.3, 0.7
    # finite differences are valid only away from a change of selection:
    # take the first draw with no top-k gap below 1e-3
    for seed in range(31, 81):
        x, Wr, Wg, Wu, Wd, dy = _moe_case(seed + 100 * k)
        T, E = x.shape[0], Wr.shape[0]
        bias = rng(seed).normal(size=E) * 0.3
        noise = rng(seed + 1).normal(size=(T, E)) * 0.5 if with_noise else None
        p = O.moe_route(x, Wr, k, coef, bias, noise)["probs"]
        if not O.near_tie_tokens(p, k, gap=1e-3).any():
            break

    def loss():
        f = O.moe_forward(x, Wr, Wg, Wu, Wd, k, coef, bias, noise, zc)
        return float(np.sum(dy * f["y"])) + d_aux * f["aux_loss"] + d_z * f["z_loss"]

    assert not O.near_tie_tokens(p, k, gap=1e-3).any()
    g = O.moe_backward(x, Wr, Wg, Wu, Wd, k, coef, dy, d_aux, bias, noise, zc, d_z)
    np.testing.assert_allclose(g["dx"], _fd_grad(loss, x), rtol=0, atol=1e-7)
    np.testing.assert_allclose(g["dWr"], _fd_grad(loss, Wr), rtol=0, atol=1e-7)
    np.testing.assert_allclose(g["d_bias"], _fd_grad(loss, bias), rtol=0, atol=1e-7)
    for e in range(E):
        np.testing.assert_allclose(g["dWg"][e], _fd_grad(loss, Wg[e]), rtol=0, atol=1e-7)
        np.testing.assert_allclose(g["dWu"][e], _fd_grad(loss, Wu[e]), rtol=0, atol=1e-7)
        np.testing.assert_allclose(g["dWd"][e], _fd_grad(loss, Wd[e]), rtol=0, atol=1e-7)


def test_moe_backward_top1_router_learns_only_from_aux():
    """Top-1 with renormalisation: alpha = p / p = 1 is constant, so <dy, y>
    sends the router no gradient (note 08 §7: the router learns through
    topk_weight; here that weight is 1) - only aux and z-loss reach it."""
    x, Wr, Wg, Wu, Wd, dy = _moe_case(50)
    g = O.moe_backward(x, Wr, Wg, Wu, Wd, 1, 0.0, dy, z_coef=0.0)
    assert np.abs(g["dWr"]).max() < 1e-12 and np.abs(g["d_bias"]).max() < 1e-12
    g = O.moe_backward(x, Wr, Wg, Wu, Wd, 1, 0.05, dy, z_coef=0.0)
    assert np.abs(g["dWr"]).max() > 1e-4


def test_moe_backward_unselected_expert_gets_no_gradient():
    x, Wr, Wg, Wu, Wd, dy = _moe_case(51)
    noise = np.zeros((x.shape[0], 4))
    noise[:, 2] = -50.0                       # expert 2 is never selected
    g = O.moe_backward(x, Wr, Wg, Wu, Wd, 2, 0.01, dy, logit_noise=noise)
    assert np.all(g["dWg"][2] == 0) and np.all(g["dWu"][2] == 0) and np.all(g["dWd"][2] == 0)
    assert np.abs(g["dWg"][0]).max() > 0


def test_moe_backward_single_expert_is_dense_backward():
    """E = 1, k = 1: alpha = 1, y = FFN(x), so the expert's gradients and dx
    are the dense FFN's; with coef = z = 0 the router gets nothing."""
    x, Wr, Wg, Wu, Wd, dy = _moe_case(52, E=1)
    g = O.moe_backward(x, Wr, Wg, Wu, Wd, 1, 0.0, dy)
    dx, dWg, dWu, dWd = O.swiglu_ffn_backward(x, Wg[0], Wu[0], Wd[0], dy)
    np.testing.assert_allclose(g["dx"], dx, rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dWg"][0], dWg, rtol=0, atol=1e-13)
    np.testing.assert_allclose(g["dWd"][0], dWd, rtol=0, atol=1e-13)
    assert np.abs(g["dWr"]).max() < 1e-12


def test_moe_backward_all_experts_identical_and_k_equal_E():
    """k = E with identical experts: y = sum_e p_e FFN(x) = FFN(x) does not
    depend on the router, so with coef = z = 0 dWr = 0 and dx is the dense
    FFN's dx; the weight gradient of each expert is p_e times the dense one."""
    x, Wr, Wg, Wu, Wd, dy = _moe_case(53)
    E = 4
    Wg, Wu, Wd = [Wg[0]] * E, [Wu[0]] * E, [Wd[0]] * E
    g = O.moe_backward(x, Wr, Wg, Wu, Wd, E, 0.0, dy)
    dx, dWg, _, _ = O.swiglu_ffn_backward(x, Wg[0], Wu[0], Wd[0], dy)
    np.testing.assert_allclose(g["dx"], dx, rtol=0, atol=1e-12)
    assert np.abs(g["dWr"]).max() < 1e-12
    np.testing.assert_allclose(sum(g["dWg"]), dWg, rtol=0, atol=1e-12)


# --------------------------------------------------------------------------
# Block fusion (lesson 13 §3 step 2): RMSNorm and the residual
# --------------------------------------------------------------------------
def test_rms_norm_hand_case():
    """[3, 4]: mean square 12.5, so x / sqrt(12.5) = [0.848528.., 1.131370..];
    times w = [2, -1]."""
    y = O.rms_norm(np.array([[3.0, 4.0]]), np.array([2.0, -1.0]), 0.0)
    np.testing.assert_allclose(y[0], [2 * 3 / math.sqrt(12.5), -4 / math.sqrt(12.5)], rtol=1e-15)


def test_rms_norm_properties():
    r = rng(60)
    x = r.normal(size=(7, 16)) * 3
    ones = np.ones(16)
    y = O.rms_norm(x, ones, 0.0)
    np.testing.assert_allclose(np.sqrt(np.mean(y ** 2, axis=1)), 1.0, rtol=1e-14)   # unit rms
    np.testing.assert_allclose(O.rms_norm(5.0 * x, ones, 0.0), y, rtol=1e-14)      # scale invariant
    # eps: a constant row c gives c / sqrt(c^2 + eps)
    c = 0.01
    assert abs(O.rms_norm(np.full((1, 4), c), ones[:4], 1e-4)[0, 0] - c / math.sqrt(c * c + 1e-4)) < 1e-16
    w = r.normal(size=16)
    np.testing.assert_allclose(O.rms_norm(x, w, 1e-5), O.rms_norm(x, ones, 1e-5) * w, rtol=1e-14)


def test_block_residual_and_zero_mlp():
    """A zero down projection makes the block the identity; otherwise block -
    x is the FFN of the normalised input (dense and MoE)."""
    r = rng(61)
    x = r.normal(size=(9, 8))
    w = r.normal(size=8)
    Wg, Wu, Wd = r.normal(size=(6, 8)), r.normal(size=(6, 8)), r.normal(size=(8, 6))
    np.testing.assert_array_equal(O.swiglu_block(x, w, 1e-5, Wg, Wu, np.zeros_like(Wd)), x)
    np.testing.assert_allclose(O.swiglu_block(x, w, 1e-5, Wg, Wu, Wd) - x,
                               O.swiglu_ffn(O.rms_norm(x, w, 1e-5), Wg, Wu, Wd), atol=1e-13)
    Wr = r.normal(size=(3, 8))
    G = [r.normal(size=(6, 8)) for _ in range(3)]
    U = [r.normal(size=(6, 8)) for _ in range(3)]
    D = [r.normal(size=(8, 6)) for _ in range(3)]
    b = O.moe_block(x, w, 1e-5, Wr, G, U, D, 2, 0.01)
    m = O.moe_forward(O.rms_norm(x, w, 1e-5), Wr, G, U, D, 2, 0.01)
    assert np.array_equal(b["topk_idx"], m["topk_idx"])   # routing on the normalised input
    np.testing.assert_allclose(b["y"] - x, m["y"], atol=1e-13)
    assert b["aux_loss"] == m["aux_loss"]
    zero = O.moe_block(x, w, 1e-5, Wr, G, U, [np.zeros((8, 6))] * 3, 2, 0.01)
    np.testing.assert_array_equal(zero["y"], x)
