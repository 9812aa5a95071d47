"""The router and the permute in one kernel (x read once, one grid-wide
barrier) against the two-kernel router + dispatch on the same inputs: every
output the same bit for bit (y, topk_idx, topk_w, aux; router statistics,
z-loss; the block's norm and residual), since the fused kernel takes the same
per-token decisions and writes the same per-router-block partials.  The
two-kernel path is itself checked against the fp64 oracle by the other
parity tests; one case here checks the fused path against the oracle too.

Shapes cover several fused blocks and a ragged last one (T = 129: a block of
one token; T = 65: one block spanning one and a bit router blocks), top-1 to
top-4, E = 16 (the widest it takes), H = 192 / 256 / 512 / 768 (3, 4, 8 and
12 k-blocks) and the full top-2 workload.  The kernel takes blocks of 64
tokens while one per SM covers T and 128 beyond: T = 64 x SMs (the largest
grid of 64-token blocks, every SM holding one) and one token more (the first
call on 128-token blocks, with a block of one token) are both checked.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_top_gb300 as mm
from swiglu_mlp_top_gb300.inputs import make_router_noise

from parity import Y_TOL, check_route, inputs64, moe_inputs, ref_y_rows, rel_err, to_dev

pytestmark = pytest.mark.gpu

SKEW = (1.5, 0.5, 0, 0, 0, 0, 0, 0)


def _both(g, k, coef, **kw):
    outs = []
    for sep in (False, True):
        stats = {} if "z_coef" in kw else None
        r = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, coef,
                           logit_bias=g.get("logit_bias"), path="tensor", stats=stats,
                           separate_routing=sep, **kw)
        torch.cuda.synchronize()
        outs.append((r, stats))
    return outs


def _assert_same(outs):
    (a, sa), (b, sb) = outs
    for u, v in zip(a, b):
        assert torch.equal(u, v)
    if sa is not None:
        for n in sa:
            assert torch.equal(sa[n], sb[n]), n


@pytest.mark.parametrize("T,H,I,E,k,bias", [
    (129, 256, 192, 8, 2, SKEW),
    (65, 768, 320, 8, 2, None),
    (777, 192, 256, 4, 1, None),
    (1000, 512, 256, 16, 4, None),
    (2048, 768, 2432, 8, 3, SKEW),
    (8192, 768, 2432, 4, 1, None),
])
def test_fused_routing_equals_two_kernels(T, H, I, E, k, bias):
    inp = moe_inputs(T, H, I, E, "bf16", seed=300 + T, bias=bias)
    g = to_dev(inp)
    _assert_same(_both(g, k, 0.01))


@pytest.mark.parametrize("extra", [0, 1])
def test_fused_routing_at_the_block_size_switch(extra):
    n_sms = torch.cuda.get_device_properties(0).multi_processor_count
    T = 64 * n_sms + extra
    inp = moe_inputs(T, 768, 256, 8, "bf16", seed=330 + extra, bias=SKEW)
    g = to_dev(inp)
    _assert_same(_both(g, 2, 0.01))


def test_fused_routing_full_size_top2():
    inp = moe_inputs(16384, 768, 2432, 8, "bf16", seed=0, bias=SKEW)
    g = to_dev(inp)
    _assert_same(_both(g, 2, 0.01))


def test_fused_routing_with_router_variants():
    T, E = 3000, 8
    inp = moe_inputs(T, 768, 512, E, "bf16", seed=310, bias=SKEW)
    g = to_dev(inp)
    noise = make_router_noise(T, E, 0.5, seed=311).cuda()
    _assert_same(_both(g, 2, 0.01, logit_noise=noise, z_coef=1e-3))


def test_fused_routing_with_block_norm_and_residual():
    T, H, E = 2500, 768, 8
    inp = moe_inputs(T, H, 512, E, "bf16", seed=320)
    g = to_dev(inp)
    gen = torch.Generator().manual_seed(321)
    w = (1.0 + 0.1 * torch.randn(H, generator=gen)).to(torch.bfloat16).cuda()
    _assert_same(_both(g, 2, 0.01, norm_weight=w, residual=True))


def test_fused_routing_matches_the_oracle():
    """The fused path on its own against the fp64 oracle (routing bars and y)."""
    T, H, I, E, k = 1500, 768, 320, 8, 2
    inp = moe_inputs(T, H, I, E, "bf16", seed=330, bias=SKEW)
    g = to_dev(inp)
    y, idx, w, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, 0.01,
                                    logit_bias=g["logit_bias"], path="tensor")
    torch.cuda.synchronize()
    i64 = inputs64(inp)
    ref = oracle.moe_route(i64["x"], i64["Wr"], k, 0.01, i64["logit_bias"])
    idx = idx.cpu().numpy()
    tie, diff = check_route(idx, w.cpu().numpy(), float(aux), ref, k)
    yref = oracle.combine(i64["x"], i64["Wg"], i64["Wu"], i64["Wd"], ref["topk_idx"], ref["topk_w"])
    if diff.any():
        rows = np.nonzero(diff)[0]
        yref[rows] = ref_y_rows(i64, ref, idx, rows, k)
    assert rel_err(y.double().cpu().numpy(), yref) <= Y_TOL["bf16"]
