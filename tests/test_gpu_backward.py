"""GPU parity of the backward pass (bf16, tensor cores) against the fp64
oracle's backward: the dense SwiGLU FFN and the MoE layer (router gradient
through alpha, aux and z-loss; per-expert weight gradients; dx).

Bar (no tolerance is stated for gradients; this one is derived from the
arithmetic): every element within 2e-2 * (rms(g*) + |g*|).  Each gradient
element is a sum of products whose operands passed through at most one
fp16 rounding (dh, 2^-11 relative) and one bf16 rounding (dG / dU or
alpha h: ~2^-8 relative), so its error is bounded by that times the sum
of |terms|.  For a gradient over one or a
few tokens (an outer product such as dG^T x for one token) that sum is
|g*| itself, and the heavy tail of dG = dh u SiLU'(g) puts max|g*| at over
10 rms: an RMS-only measure would flag elements that are within 2^-8
relative.  Where a gradient sums over many tokens no outer product
dominates, and the forward's own measure, max|g - g*| / rms(g*) <= 2e-2,
is asserted as well (T >= 1000 per call).
Experts that no token selected must get exact zeros.  The MoE backward runs
on the routing its own forward produced (topk_idx, topk_w, probabilities,
logsumexp), as a training step would; the oracle takes the GPU's selection
on near-tie tokens (both are correct forwards).
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_top_gb300 as mm
from swiglu_mlp_top_gb300.inputs import make_inputs, make_router_noise, to_f64

from parity import check_route, inputs64, moe_inputs, to_dev

pytestmark = pytest.mark.gpu

G_TOL = 2e-2


def grad_err(g, ref):
    """(max |g - g*| / (rms(g*) + |g*|), max |g - g*| / rms(g*))."""
    g = np.asarray(g, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    rms = np.sqrt(np.mean(ref ** 2))
    d = np.abs(g - ref)
    return float((d / (rms + np.abs(ref))).max()), float(d.max() / rms)


def assert_grad(name, got, want, rms_bar):
    mixed, rms_rel = grad_err(got, want)
    assert mixed <= G_TOL, f"{name}: {mixed} (max err / rms: {rms_rel})"
    if rms_bar:
        assert rms_rel <= G_TOL, f"{name}: max err / rms {rms_rel}"
    return rms_rel


def _dy(T, H, seed):
    gen = torch.Generator().manual_seed(seed)
    return torch.randn(T, H, generator=gen).to(torch.bfloat16)


@pytest.mark.parametrize("T,H,I", [(1, 256, 384), (300, 256, 384), (1000, 768, 2432),
                                   (257, 128, 192), (4096, 768, 2432)])
def test_dense_backward(T, H, I):
    inp = make_inputs(T, H, I, "bf16", seed=400 + T)
    dy = _dy(T, H, 500 + T)
    g = to_dev(inp)
    dx, dWg, dWu, dWd = mm.swiglu_ffn_backward(g["x"], g["Wg"], g["Wu"], g["Wd"], dy.cuda())
    torch.cuda.synchronize()
    ref = oracle.swiglu_ffn_backward(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")], to_f64(dy))
    for name, got, want in zip(("dx", "dWg", "dWu", "dWd"), (dx, dWg, dWu, dWd), ref):
        assert_grad(name, got.double().cpu().numpy(), want, rms_bar=T >= 1000)


@pytest.mark.parametrize("scale,expect", [(1.0, 0), (1e6, 6)])
def test_fp16_dh_overflow_is_reported(scale, expect):
    """The backward keeps dh = dy Wd in fp16.  With dy scaled by 1e6 (Wd
    N(0, 0.02), H = 256: |dh| ~ 3e5) dh is beyond fp16's 65504, and the call
    must report MM_ERR_RANGE through mm_check_status; unscaled, nothing.
    The status clears once read."""
    T, H, I = 64, 256, 384
    inp = make_inputs(T, H, I, "bf16", seed=41)
    dy = (_dy(T, H, 42).float() * scale).to(torch.bfloat16)
    g = to_dev(inp)
    lib = mm._lib.load()
    ws = mm.new_workspace(lib.mm_swiglu_ffn_backward_workspace_bytes(T, H, I, 1))
    mm.swiglu_ffn_backward(g["x"], g["Wg"], g["Wu"], g["Wd"], dy.cuda(), workspace=ws)
    assert mm.check_status(ws) == expect
    assert mm.check_status(ws) == 0


def _moe_step(inp, k, coef, z_coef, noise, dy, path="tensor"):
    g = to_dev(inp)
    stats = {}
    y, idx, w, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, coef,
                                    logit_bias=g.get("logit_bias"), path=path,
                                    logit_noise=None if noise is None else noise.cuda(),
                                    z_coef=z_coef, stats=stats)
    grads = mm.moe_backward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, coef, idx, w,
                            stats["probs"], dy.cuda(), d_aux=1.0, lse=stats["lse"],
                            z_coef=z_coef, d_z=1.0, bias_grad=True)
    torch.cuda.synchronize()
    return idx, w, aux, grads


def _check_moe(inp, k, coef=0.01, z_coef=1e-3, noise_std=0.0, seed=0):
    T, H = inp["x"].shape
    E = len(inp["Wg"])
    noise = make_router_noise(T, E, noise_std, seed=seed) if noise_std else None
    dy = _dy(T, H, 600 + seed)
    idx, w, aux, grads = _moe_step(inp, k, coef, z_coef, noise, dy)
    i64 = inputs64(inp)
    nz = None if noise is None else to_f64(noise)
    route = oracle.moe_route(i64["x"], i64["Wr"], k, coef, i64.get("logit_bias"), nz, z_coef)
    check_route(idx.cpu().numpy(), w.cpu().numpy(), float(aux), route, k)
    ref = oracle.moe_backward(i64["x"], i64["Wr"], i64["Wg"], i64["Wu"], i64["Wd"], k, coef,
                              to_f64(dy), 1.0, i64.get("logit_bias"), nz, z_coef, 1.0,
                              topk_idx=idx.cpu().numpy())
    big = T >= 1000
    errs = {"dx": assert_grad("dx", grads["dx"].double().cpu().numpy(), ref["dx"], big),
            "dWr": assert_grad("dWr", grads["dWr"].cpu().numpy(), ref["dWr"], big),
            "d_bias": assert_grad("d_bias", grads["d_bias"].cpu().numpy(), ref["d_bias"], big)}
    counts = np.bincount(idx.cpu().numpy().reshape(-1), minlength=E)
    for name in ("dWg", "dWu", "dWd"):
        for e in range(E):
            got = grads[name][e].cpu().numpy()
            want = ref[name][e]
            if counts[e] == 0:
                assert not np.any(got), f"{name}[{e}]: an unselected expert got a gradient"
                continue
            errs[f"{name}[{e}]"] = assert_grad(f"{name}[{e}]", got, want, counts[e] >= 1000)
    return errs


@pytest.mark.parametrize("T,H,I,E,k,bias", [
    (777, 256, 320, 8, 2, (1.5, 0.5, 0, 0, 0, 0, 0, 0)),
    (513, 128, 192, 6, 3, None),
    (1000, 256, 384, 4, 1, None),
    (300, 256, 192, 64, 8, None),
    (600, 256, 256, 8, 2, (0.0, 0.0, 0.0, 8.0, 0.0, -8.0, -8.0, -8.0)),   # experts 5-7 unused
    (5, 256, 256, 4, 2, None),
])
def test_moe_backward(T, H, I, E, k, bias):
    _check_moe(moe_inputs(T, H, I, E, "bf16", seed=700 + T, bias=bias), k, seed=T)


@pytest.mark.parametrize("z_coef,noise_std,coef", [(0.0, 0.0, 0.0), (1e-2, 0.5, 0.02)])
def test_moe_backward_router_variants(z_coef, noise_std, coef):
    """Without aux / z the router learns only through alpha; with router
    noise and z-loss the noise and lse enter through the saved statistics."""
    inp = moe_inputs(900, 256, 256, 8, "bf16", seed=801)
    _check_moe(inp, 2, coef=coef, z_coef=z_coef, noise_std=noise_std, seed=11)


def test_moe_backward_deterministic():
    inp = moe_inputs(700, 256, 320, 8, "bf16", seed=802)
    dy = _dy(700, 256, 33)
    a = _moe_step(inp, 2, 0.01, 1e-3, None, dy)[3]
    b = _moe_step(inp, 2, 0.01, 1e-3, None, dy)[3]
    for name in ("dx", "dWr", "d_bias"):
        assert torch.equal(a[name], b[name]), name
    for name in ("dWg", "dWu", "dWd"):
        assert all(torch.equal(u, v) for u, v in zip(a[name], b[name])), name


def test_moe_backward_full_size_top2():
    """The top-2 skewed workload at full size (T = 16384, H = 768, I = 2432,
    E = 8): every gradient against the oracle."""
    from swiglu_mlp_top_gb300.inputs import WORKLOADS, make_workload_inputs
    w = WORKLOADS["moe_e8k2_t16384_skew"]
    errs = _check_moe(make_workload_inputs(w), w.k, coef=w.coef, seed=5)
    assert max(errs.values()) <= G_TOL, errs
