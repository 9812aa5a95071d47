"""GPU parity of the router variants (router noise, z-loss) and the saved
router statistics (probabilities, logsumexp) against the fp64 oracle, on
every kernel family that routes: the tensor-core prefill router, the
CUDA-core router (fp32, and bf16 shapes the tensor-core one does not take),
the two weight-streaming kernels (including the speculative form that
routes while every expert streams), and the router-only entry point.

Bars: the routing bars of the other parity tests (indices bit-exact except
near-ties, alpha within 1e-5, aux within 1e-5); z-loss within 1e-5
absolute, the aux bar (both are scalar losses of the same size class);
probabilities and lse within 1e-5 absolute; y as the other tests.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_top_gb300 as mm
from swiglu_mlp_top_gb300.inputs import make_router_noise, to_f64

from parity import Y_TOL, check_route, inputs64, moe_inputs, ref_y_rows, rel_err, to_dev

pytestmark = pytest.mark.gpu

Z_TOL = 1e-5
STAT_TOL = 1e-5
Z_COEF = 1e-3


def _check(inp, k, dtype, path, noise_std, route_only=False):
    T, E = inp["x"].shape[0], len(inp["Wg"])
    noise = make_router_noise(T, E, noise_std, seed=T + E) if noise_std else None
    g = to_dev(inp)
    stats = {}
    if route_only:
        idx, w, aux, _ = mm.moe_route(g["x"], g["Wr"], k, 0.01, logit_bias=g.get("logit_bias"),
                                      logit_noise=None if noise is None else noise.cuda(),
                                      z_coef=Z_COEF, stats=stats)
        y = None
    else:
        y, idx, w, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, 0.01,
                                        logit_bias=g.get("logit_bias"), path=path,
                                        logit_noise=None if noise is None else noise.cuda(),
                                        z_coef=Z_COEF, stats=stats)
    torch.cuda.synchronize()
    i64 = inputs64(inp)
    ref = oracle.moe_route(i64["x"], i64["Wr"], k, 0.01, i64.get("logit_bias"),
                           None if noise is None else to_f64(noise), Z_COEF)
    idx = idx.cpu().numpy()
    tie, diff = check_route(idx, w.cpu().numpy(), float(aux), ref, k)
    assert abs(float(stats["z_loss"]) - ref["z_loss"]) <= Z_TOL, (float(stats["z_loss"]), ref["z_loss"])
    assert np.abs(stats["probs"].cpu().numpy() - ref["probs"]).max() <= STAT_TOL
    assert np.abs(stats["lse"].cpu().numpy() - ref["lse"]).max() <= STAT_TOL
    if y is not None:
        yd = y.double().cpu().numpy()
        yref = oracle.combine(i64["x"], i64["Wg"], i64["Wu"], i64["Wd"], ref["topk_idx"],
                              ref["topk_w"])
        if diff.any():
            rows = np.nonzero(diff)[0]
            yref[rows] = ref_y_rows(i64, ref, idx, rows, k)
        assert rel_err(yd, yref) <= Y_TOL[dtype]
    return ref


@pytest.mark.parametrize("T,H,I,E,k,dtype,path,bias", [
    (777, 256, 320, 8, 2, "bf16", "tensor", (1.5, 0.5, 0, 0, 0, 0, 0, 0)),   # tensor-core router
    (300, 256, 192, 64, 8, "bf16", "tensor", None),                         # 64 experts, top-8
    (300, 128, 192, 8, 2, "f32", "auto", None),                             # CUDA-core router, fp32
    (3, 768, 2432, 8, 2, "bf16", "stream", None),                           # CUDA-core streaming
    (40, 768, 2432, 8, 2, "bf16", "stream_tc", (1.5, 0.5, 0, 0, 0, 0, 0, 0)),
    (16, 768, 2432, 8, 2, "bf16", "auto", None),                            # speculative streaming
    (64, 768, 2432, 8, 2, "bf16", "auto", None),
])
@pytest.mark.parametrize("noise_std", [0.0, 0.5])
def test_router_variants_match_the_oracle(T, H, I, E, k, dtype, path, bias, noise_std):
    inp = moe_inputs(T, H, I, E, dtype, seed=200 + T, bias=bias)
    _check(inp, k, dtype, path, noise_std)


@pytest.mark.parametrize("T,H,E,k", [(5000, 768, 8, 2), (700, 200, 6, 3)])
def test_route_only_with_router_variants(T, H, E, k):
    """The second shape (H = 200, not a multiple of 64) takes the CUDA-core
    router for bf16."""
    inp = moe_inputs(T, H, 64, E, "bf16", seed=210 + T)
    _check(inp, k, "bf16", "auto", 0.3, route_only=True)


def test_large_noise_overrides_the_router():
    """Noise of +50 on expert 5 for every token: every token's first choice is
    expert 5 on the GPU too."""
    T, E = 400, 8
    inp = moe_inputs(T, 256, 256, E, "bf16", seed=220)
    g = to_dev(inp)
    noise = torch.zeros(T, E)
    noise[:, 5] = 50.0
    _, idx, _, _ = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01,
                                  path="tensor", logit_noise=noise.cuda())
    assert (idx[:, 0] == 5).all()


def test_options_of_zero_are_the_plain_forward():
    """An options struct with no variant gives the plain forward bit for bit;
    asking only for the statistics changes no output."""
    inp = moe_inputs(500, 256, 320, 8, "bf16", seed=221)
    g = to_dev(inp)
    a = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01)
    stats = {}
    b = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01, stats=stats)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    assert float(stats["z_loss"]) == 0.0
