"""GPU parity of the MiniMind block fusion (lesson 13 §3 step 2:
hidden + mlp(post_attention_layernorm(hidden))) against the oracle's
rms_norm / swiglu_block / moe_block: the RMSNorm prologue (router at full
precision, experts on the normalised rows) and the residual added in the
down GEMM's epilogue before y's one rounding.

Bars: the forward's (y within 2e-2 of rms(y*) for bf16, 1e-4 for fp32;
routing bit-exact except near-ties; aux within 1e-5).  y* includes x, so
the measure is normalised by the block output's rms.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_top_gb300 as mm
from swiglu_mlp_top_gb300.inputs import make_inputs, to_f64

from parity import Y_TOL, check_route, inputs64, moe_inputs, rel_err, to_dev

pytestmark = pytest.mark.gpu

EPS = 1e-5


def _norm_w(H, dtype, seed):
    gen = torch.Generator().manual_seed(seed)
    w = 1.0 + 0.1 * torch.randn(H, generator=gen)
    return w.to(torch.bfloat16 if dtype == "bf16" else torch.float32)


@pytest.mark.parametrize("T,H,I,dtype", [(300, 256, 384, "bf16"), (1000, 768, 2432, "bf16"),
                                         (4096, 768, 2432, "bf16"), (70, 64, 256, "f32"),
                                         (1, 256, 384, "bf16")])
def test_dense_block(T, H, I, dtype):
    inp = make_inputs(T, H, I, dtype, seed=900 + T)
    w = _norm_w(H, dtype, T)
    g = to_dev(inp)
    y = mm.swiglu_block(g["x"], w.cuda(), g["Wg"], g["Wu"], g["Wd"], norm_eps=EPS)
    torch.cuda.synchronize()
    ref = oracle.swiglu_block(to_f64(inp["x"]), to_f64(w), EPS,
                              *[to_f64(inp[n]) for n in ("Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL[dtype]


def _moe_block_check(inp, k, dtype, path, norm=True, residual=True):
    T, H = inp["x"].shape
    w = _norm_w(H, dtype, T + 1)
    g = to_dev(inp)
    y, idx, tw, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, 0.01,
                                     logit_bias=g.get("logit_bias"), path=path,
                                     norm_weight=w.cuda() if norm else None, norm_eps=EPS,
                                     residual=residual)
    torch.cuda.synchronize()
    i64 = inputs64(inp)
    xin = oracle.rms_norm(i64["x"], to_f64(w), EPS) if norm else i64["x"]
    ref = oracle.moe_forward(xin, i64["Wr"], i64["Wg"], i64["Wu"], i64["Wd"], k, 0.01,
                             i64.get("logit_bias"))
    idx = idx.cpu().numpy()
    tie, diff = check_route(idx, tw.cpu().numpy(), float(aux), ref, k)
    yref = ref["y"].copy()
    if diff.any():
        rows = np.nonzero(diff)[0]
        sel = idx[rows].astype(np.int64)
        alpha = oracle.renormalise(np.take_along_axis(ref["probs"][rows], sel, axis=-1))
        yref[rows] = oracle.combine(xin[rows], i64["Wg"], i64["Wu"], i64["Wd"], sel, alpha)
    if residual:
        yref = yref + i64["x"]
    assert rel_err(y.double().cpu().numpy(), yref) <= Y_TOL[dtype]


@pytest.mark.parametrize("T,H,I,E,k,dtype,path,bias", [
    (777, 256, 320, 8, 2, "bf16", "auto", (1.5, 0.5, 0, 0, 0, 0, 0, 0)),   # tensor-core router
    (1000, 256, 384, 4, 1, "bf16", "tensor", None),
    (513, 128, 192, 6, 3, "bf16", "tensor", None),
    (300, 256, 192, 64, 8, "bf16", "tensor", None),                       # CUDA-core router (2E > 64)
    (300, 128, 192, 8, 2, "f32", "auto", None),                           # fp32, CUDA cores
    (400, 256, 256, 8, 2, "bf16", "simt", None),
    (3, 768, 2432, 8, 2, "bf16", "auto", None),                           # decode-sized: GEMM path
])
def test_moe_block(T, H, I, E, k, dtype, path, bias):
    _moe_block_check(moe_inputs(T, H, I, E, dtype, seed=950 + T, bias=bias), k, dtype, path)


@pytest.mark.parametrize("norm,residual", [(True, False), (False, True)])
def test_moe_block_parts(norm, residual):
    _moe_block_check(moe_inputs(600, 256, 320, 8, "bf16", seed=990), 2, "bf16", "tensor",
                     norm=norm, residual=residual)


def test_moe_block_full_size_top2():
    from swiglu_mlp_top_gb300.inputs import WORKLOADS, make_workload_inputs
    w = WORKLOADS["moe_e8k2_t16384_skew"]
    _moe_block_check(make_workload_inputs(w), w.k, "bf16", "auto")


def test_block_rejects_streaming_paths_and_aliasing():
    inp = moe_inputs(8, 768, 2432, 8, "bf16", seed=991)
    g = to_dev(inp)
    w = _norm_w(768, "bf16", 3).cuda()
    with pytest.raises(RuntimeError, match="MM_ERR_UNSUPPORTED"):
        mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01, path="stream_tc",
                       norm_weight=w)
    with pytest.raises(RuntimeError, match="MM_ERR_INVALID_ARG"):
        mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01, residual=True,
                       out=g["x"])
