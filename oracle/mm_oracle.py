"""fp64 CPU oracle for the SwiGLU FFN and the top-k MoE forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may call it.  It shares no code with the CUDA library.

Every function is the plain definition written out in float64 numpy, in the
order and notation of the pages it follows.  A matrix product (``@``) and a
sort (``np.lexsort``) are the only library primitives used; nothing is
blocked, fused or reordered.

Sources (cited by tag below):
  [L13]   MiniMind course, lesson 13 "FFN 与 MoE" (course/13_ffn_and_moe.md)
  [CH4]   minimind3.com, chapter 4 "前馈网络 MLP & MoE"
  [DEMO]  minimind3.com, example "前馈网络 MLP & MoE：示例代码" (04-mlp-moe-demo.py)

Notation (as on the pages): T tokens (the pages' N = B*S), H hidden size,
I intermediate size, E experts, k experts per token.  Weights follow the
nn.Linear layout [out, in]: Wg, Wu: [I, H]; Wd: [H, I]; Wr: [E, H].

Readings taken where the pages are silent or inconsistent (each one is
listed with its reason in the design notes of the repository):
  * top-k order: descending probability; equal probabilities -> the lower
    expert index first ([L13] step 4 uses torch.topk(sorted=False), which
    leaves both unspecified).
  * aux loss for k > 1: load_e = count_e / T, i.e. the [k, E] "load" of
    [L13] step 6 / [CH4] §4.4 summed over the k slots (the value the module
    returns), not the per-slot mean of the demo's printed breakdown.
  * aux loss is always computed; coef = 0 gives 0 (the eval branch).
  * The "+1e-20" of the renormalisation is kept.
Parity is pinned for every function here (tests/test_oracle.py); no
function is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

F64 = np.float64

#: Added to the denominator of the top-k renormalisation ([L13] step 5;
#: [CH4] §4.3 step 2).
RENORM_EPS = 1e-20


def _f64(a) -> np.ndarray:
    return np.asarray(a, dtype=F64)


# --------------------------------------------------------------------------
# Dense SwiGLU FFN
# --------------------------------------------------------------------------
def silu(z):
    """SiLU(z) = z * sigmoid(z) = z / (1 + exp(-z))  ([CH4] §4.2 "原理说明")."""
    z = _f64(z)
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def swiglu_ffn(x, Wg, Wu, Wd):
    """Dense SwiGLU feed-forward, [L13] §0 / §1.2 equations:

        u = W_up x,  g = W_gate x,  h = SiLU(g) ⊙ u,  y = W_down h

    x: [T, H]; Wg, Wu: [I, H]; Wd: [H, I]  ->  y: [T, H]  (all float64).
    """
    x, Wg, Wu, Wd = _f64(x), _f64(Wg), _f64(Wu), _f64(Wd)
    u = x @ Wu.T            # [T, I]
    g = x @ Wg.T            # [T, I]
    h = silu(g) * u         # [T, I]
    return h @ Wd.T         # [T, H]


# --------------------------------------------------------------------------
# Router: logits, softmax, top-k, renormalisation
# --------------------------------------------------------------------------
def router_logits(x, Wr, logit_bias=None, logit_noise=None):
    """r = W_router x  ([L13] §1.5; [CH4] §4.3 "gate" = nn.Linear(H, E, bias=False)).

    ``logit_bias`` ([E] or None) is added to every token's logits; None gives
    the pages' bias-free router exactly.  ``logit_noise`` ([T, E] or None) is
    the router noise of NOTE08 §10's table ("add noise to the router to
    encourage exploration"), read as an additive perturbation of each
    token's logits; its random draws are an input.
    """
    r = _f64(x) @ _f64(Wr).T                      # [T, E]
    if logit_bias is not None:
        r = r + _f64(logit_bias)[None, :]
    if logit_noise is not None:
        r = r + _f64(logit_noise)
    return r


def logsumexp(r):
    """lse_t = log sum_e exp(r_{t,e}), with the row maximum taken out first
    (lse = m + log sum_e exp(r_e - m), the same value)."""
    r = _f64(r)
    m = r.max(axis=-1)
    return m + np.log(np.exp(r - m[:, None]).sum(axis=-1))


def z_loss(r, z_coef):
    """Router z-loss: L_z = z_coef * (1/T) * sum_t (lse_t)^2.

    NOTE08 §10's table names z-loss as the mechanism that keeps the router
    logits from growing too large and gives no formula; this is the
    standard definition (the mean squared log-partition function of the
    router's softmax), the plainest reading.
    """
    lse = logsumexp(r)
    return F64(z_coef) * float(np.mean(lse ** 2))


def softmax(r):
    """p_e = exp(r_e) / sum_j exp(r_j) over the expert axis ([L13] §1.5).

    The row maximum is subtracted first; the quotient is unchanged.
    """
    r = _f64(r)
    z = np.exp(r - r.max(axis=-1, keepdims=True))
    return z / z.sum(axis=-1, keepdims=True)


def topk(p, k):
    """S = TopK(p, k) per token ([L13] §1.5 and step 4).

    Returns (idx [T, k] int64, val [T, k] float64) with each row ordered by
    descending probability, equal probabilities broken towards the lower
    expert index.
    """
    p = _f64(p)
    T, E = p.shape
    if not 1 <= k <= E:
        raise ValueError(f"need 1 <= k <= E, got k={k}, E={E}")
    ids = np.broadcast_to(np.arange(E), (T, E))
    # np.lexsort sorts by the LAST key first: primary -p, secondary index.
    order = np.lexsort((ids, -p), axis=-1)
    idx = order[:, :k].astype(np.int64)
    val = np.take_along_axis(p, idx, axis=-1)
    return idx, val


def renormalise(val):
    """alpha_e = p_e / (sum_{j in S} p_j + 1e-20)  ([L13] step 5; [CH4] §4.3 step 2)."""
    val = _f64(val)
    return val / (val.sum(axis=-1, keepdims=True) + RENORM_EPS)


# --------------------------------------------------------------------------
# Load-balancing auxiliary loss
# --------------------------------------------------------------------------
def expert_load(topk_idx, E):
    """load_e = (1/T) * #{(t, s): topk_idx[t, s] == e}  ([L13] §1.6; [CH4] §4.4 step 1).

    For k = 1 this is the fraction of tokens routed to e; for k > 1 it is the
    [k, E] one-hot mean of the pages summed over the k slots.
    """
    topk_idx = np.asarray(topk_idx)
    T = topk_idx.shape[0]
    counts = np.zeros(E, dtype=np.int64)
    for e in topk_idx.reshape(-1):
        counts[int(e)] += 1
    return counts.astype(F64) / F64(T), counts


def mean_prob(p):
    """prob_e = (1/T) * sum_t p_{t,e}  ([L13] §1.6; [CH4] §4.4 step 2)."""
    return _f64(p).mean(axis=0)


def aux_loss_from_stats(load, prob, E, coef):
    """L_aux = E * coef * sum_e load_e * prob_e  ([L13] §1.6 equation; [CH4] §4.4 step 3)."""
    return F64(E) * F64(coef) * float(np.sum(_f64(load) * _f64(prob)))


def aux_loss(topk_idx, p, coef):
    """L_aux from the selections and the probabilities directly ([L13] §1.6;
    [CH4] §4.4): E is the number of probability columns, load_e counts every
    slot (the [k, E] one-hot mean summed over k)."""
    p = _f64(p)
    E = p.shape[1]
    load, _ = expert_load(topk_idx, E)
    return aux_loss_from_stats(load, mean_prob(p), E, coef)


# --------------------------------------------------------------------------
# MoE layer
# --------------------------------------------------------------------------
def combine(x, Wg, Wu, Wd, topk_idx, alpha):
    """y_t = sum_s alpha_{t,s} * Expert_{idx[t,s]}(x_t)  ([L13] §0 MoE equation, step 5).

    The pages' dispatch: for each expert e, gather the tokens that chose it,
    run the expert on them, scale by their weight and add into y at those
    tokens (index_add_).  Wg/Wu/Wd are sequences of E per-expert matrices.
    """
    x = _f64(x)
    topk_idx = np.asarray(topk_idx)
    alpha = _f64(alpha)
    T, H = x.shape
    y = np.zeros((T, H), dtype=F64)
    for e in range(len(Wg)):
        mask = topk_idx == e                         # [T, k]
        if not mask.any():
            continue
        tok = np.nonzero(mask.any(axis=-1))[0]       # tokens that chose e
        w = alpha[mask]                              # their weights, token order
        out = swiglu_ffn(x[tok], Wg[e], Wu[e], Wd[e])
        y[tok] += out * w[:, None]
    return y


def moe_forward(x, Wr, Wg, Wu, Wd, k, coef, logit_bias=None, logit_noise=None, z_coef=0.0):
    """The MoE layer forward ([L13] step 4-6; [CH4] §4.3-4.4).

    Returns a dict with y [T, H], topk_idx [T, k], topk_w (alpha) [T, k],
    aux_loss (float), probs p [T, E], the per-expert counts [E], the
    logsumexp of each token's logits lse [T] and the router z-loss.
    """
    out = moe_route(x, Wr, k, coef, logit_bias, logit_noise, z_coef)
    out["y"] = combine(x, Wg, Wu, Wd, out["topk_idx"], out["topk_w"])
    return out


def moe_route(x, Wr, k, coef, logit_bias=None, logit_noise=None, z_coef=0.0):
    """Router half of :func:`moe_forward` (no experts): idx, alpha, aux, probs,
    counts, lse, z_loss."""
    x = _f64(x)
    r = router_logits(x, Wr, logit_bias, logit_noise)
    p = softmax(r)
    E = p.shape[1]
    idx, val = topk(p, k)
    alpha = renormalise(val)
    load, counts = expert_load(idx, E)
    aux = aux_loss_from_stats(load, mean_prob(p), E, coef)
    return {"topk_idx": idx, "topk_w": alpha, "aux_loss": aux, "probs": p,
            "counts": counts, "lse": logsumexp(r), "z_loss": z_loss(r, z_coef)}


def near_tie_tokens(p, k, gap=1e-6):
    """Tokens whose top-k choice or slot order is decided by a probability gap
    below ``gap``: sort the row descending, q_1 >= ... >= q_E; the token is a
    near-tie if q_j - q_{j+1} < gap for some j <= k (j + 1 <= E).
    Returns a boolean mask [T].
    """
    q = -np.sort(-_f64(p), axis=-1)
    E = q.shape[1]
    jmax = min(k, E - 1)
    if jmax <= 0:
        return np.zeros(q.shape[0], dtype=bool)
    gaps = q[:, :jmax] - q[:, 1:jmax + 1]
    return (gaps < gap).any(axis=-1)


# --------------------------------------------------------------------------
# Backward pass (training: L_train = L_lm + L_aux, lesson 13 step 8)
# --------------------------------------------------------------------------
def swiglu_ffn_backward(x, Wg, Wu, Wd, dy):
    """Gradients of the dense SwiGLU FFN for an upstream gradient dy = dL/dy
    (the chain rule through [L13] §0 / §1.2's equations):

        g = Wg x, u = Wu x, s = sigmoid(g), h = g s u, y = Wd h
        dWd = dy^T h,  dh = dy Wd
        du = dh * SiLU(g),  dg = dh * u * SiLU'(g),  SiLU'(g) = s (1 + g (1 - s))
        dx = dg Wg + du Wu,  dWg = dg^T x,  dWu = du^T x

    Returns (dx [T, H], dWg [I, H], dWu [I, H], dWd [H, I]).
    """
    x, Wg, Wu, Wd, dy = _f64(x), _f64(Wg), _f64(Wu), _f64(Wd), _f64(dy)
    g = x @ Wg.T
    u = x @ Wu.T
    sg = 1.0 / (1.0 + np.exp(-g))
    h = g * sg * u
    dWd = dy.T @ h
    dh = dy @ Wd
    du = dh * (g * sg)
    dg = dh * u * (sg * (1.0 + g * (1.0 - sg)))
    dx = dg @ Wg + du @ Wu
    return dx, dg.T @ x, du.T @ x, dWd


def moe_backward(x, Wr, Wg, Wu, Wd, k, coef, dy, d_aux=1.0, logit_bias=None,
                 logit_noise=None, z_coef=0.0, d_z=1.0, topk_idx=None):
    """Gradients of L = <dy, y> + d_aux * aux_loss + d_z * z_loss for the MoE
    layer (the scalar upstream gradients d_aux, d_z are 1 for L_lm + L_aux).

    Routing is recomputed as in :func:`moe_forward`; the selection S is a
    discrete choice with no gradient, so (p-chao.com note 08 §7) the router
    receives gradient only through the selected weights alpha, and the
    experts a token did not select receive none from it.  In aux, the load
    f_e is a count with no gradient and the mean probability P_e carries it
    ([CH4] §4.4: f_i is not differentiable, P_i is).  Steps:

      o_{t,s} = Expert_{S_s}(x_t);   y_t = sum_s alpha_{t,s} o_{t,s}
      dalpha_{t,s} = <dy_t, o_{t,s}>;  expert backward with upstream alpha dy_t
      alpha_s = p_s / Z, Z = sum_S p + 1e-20:
          dp_{S_s} += dalpha_s / Z - (sum_j dalpha_j p_{S_j}) / Z^2
      aux = E coef sum_e (count_e / T)(sum_t p_{t,e} / T):
          dp_{t,e} += d_aux * E * coef * count_e / T^2
      softmax: dr_{t,e} = p_{t,e} (dp_{t,e} - sum_j p_{t,j} dp_{t,j})
      z-loss = z_coef / T * sum_t lse_t^2:  dr_{t,e} += d_z * 2 z_coef lse_t p_{t,e} / T
      dWr = dr^T x;  dx += dr Wr;  d_bias = sum_t dr_t (the logit bias as a parameter)

    ``topk_idx`` (optional) replaces the selection: on a near-tie token both
    selections are correct forwards, and a backward is compared on the one
    the forward took.

    Returns a dict: dx [T, H], dWr [E, H], dWg / dWu / dWd (lists of E),
    d_bias [E], dalpha [T, k], dlogits [T, E].
    """
    x, Wr, dy = _f64(x), _f64(Wr), _f64(dy)
    T, H = x.shape
    E = len(Wg)
    r = router_logits(x, Wr, logit_bias, logit_noise)
    p = softmax(r)
    idx, val = topk(p, k)
    if topk_idx is not None:
        idx = np.asarray(topk_idx).astype(np.int64)
        val = np.take_along_axis(p, idx, axis=-1)
    alpha = renormalise(val)
    _, counts = expert_load(idx, E)
    dx = np.zeros((T, H))
    dWg = [np.zeros_like(_f64(w)) for w in Wg]
    dWu = [np.zeros_like(_f64(w)) for w in Wu]
    dWd = [np.zeros_like(_f64(w)) for w in Wd]
    dalpha = np.zeros((T, k))
    for e in range(E):
        for s in range(k):
            tok = np.nonzero(idx[:, s] == e)[0]
            if tok.size == 0:
                continue
            o = swiglu_ffn(x[tok], Wg[e], Wu[e], Wd[e])
            dalpha[tok, s] = np.sum(dy[tok] * o, axis=1)
            up = dy[tok] * alpha[tok, s][:, None]
            gx, gg, gu, gd = swiglu_ffn_backward(x[tok], Wg[e], Wu[e], Wd[e], up)
            dx[tok] += gx
            dWg[e] += gg
            dWu[e] += gu
            dWd[e] += gd
    dp = np.zeros((T, E))
    Z = val.sum(axis=1) + RENORM_EPS
    c = np.sum(dalpha * val, axis=1)
    for s in range(k):
        dp[np.arange(T), idx[:, s]] += dalpha[:, s] / Z - c / Z ** 2
    dp += F64(d_aux) * F64(E) * F64(coef) * counts[None, :].astype(F64) / F64(T) ** 2
    dr = p * (dp - np.sum(p * dp, axis=1, keepdims=True))
    lse = logsumexp(r)
    dr += F64(d_z) * 2.0 * F64(z_coef) * lse[:, None] * p / F64(T)
    dx += dr @ Wr
    return {"dx": dx, "dWr": dr.T @ x, "dWg": dWg, "dWu": dWu, "dWd": dWd,
            "d_bias": dr.sum(axis=0), "dalpha": dalpha, "dlogits": dr}


# --------------------------------------------------------------------------
# Block fusion: hidden = hidden + mlp(post_attention_layernorm(hidden))
# --------------------------------------------------------------------------
def rms_norm(x, w, eps):
    """RMSNorm of each row: x / sqrt(mean_h x_h^2 + eps) * w.

    The pages name the block's post_attention_layernorm an RMSNorm ([L13]
    §3 step 2 and the block diagram of §7) without its formula; this is the
    standard definition, with eps an argument.
    """
    x, w = _f64(x), _f64(w)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + F64(eps)) * w[None, :]


def swiglu_block(x, norm_w, eps, Wg, Wu, Wd):
    """x + FFN(RMSNorm(x)): the dense FFN in its MiniMind block ([L13] §3 step 2)."""
    return _f64(x) + swiglu_ffn(rms_norm(x, norm_w, eps), Wg, Wu, Wd)


def moe_block(x, norm_w, eps, Wr, Wg, Wu, Wd, k, coef, logit_bias=None, logit_noise=None,
              z_coef=0.0):
    """x + MoE(RMSNorm(x)) ([L13] §3 step 2 with use_moe): the routing outputs
    are those of the MoE layer on the normalised input."""
    out = moe_forward(rms_norm(x, norm_w, eps), Wr, Wg, Wu, Wd, k, coef, logit_bias,
                      logit_noise, z_coef)
    out["y"] = _f64(x) + out["y"]
    return out
