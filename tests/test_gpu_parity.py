"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle,
element by element, on seeded inputs.  Small cases span several tiles and a
ragged tail; the full-size workloads are checked on every routing output and
every row of y.
"""
import numpy as np
import pytest
import torch

import oracle
import swiglu_mlp_top_gb300 as mm
from swiglu_mlp_top_gb300.inputs import WORKLOADS, make_inputs, make_workload_inputs, to_f64

from parity import (Y_TOL, check_route, inputs64, moe_inputs, ref_y_rows, rel_err, to_dev)

pytestmark = pytest.mark.gpu


def run_moe(inp, k, coef, path="auto"):
    g = to_dev(inp)
    y, idx, w, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, coef,
                                    logit_bias=g.get("logit_bias"), path=path)
    torch.cuda.synchronize()
    return (y.double().cpu().numpy(), idx.cpu().numpy(), w.cpu().numpy(), float(aux))


def full_moe_check(inp, k, coef, dtype, path="auto"):
    y, idx, w, aux = run_moe(inp, k, coef, path)
    i64 = inputs64(inp)
    ref = oracle.moe_forward(i64["x"], i64["Wr"], i64["Wg"], i64["Wu"], i64["Wd"], k, coef,
                             i64.get("logit_bias"))
    tie, diff = check_route(idx, w, aux, ref, k)
    yref = ref["y"].copy()
    if diff.any():
        rows = np.nonzero(diff)[0]
        yref[rows] = ref_y_rows(i64, ref, idx, rows, k)
    err = rel_err(y, yref)
    assert np.isfinite(y).all(), "non-finite y"
    assert err <= Y_TOL[dtype], f"y rel err {err} [{int(tie.sum())} near-tie tokens]"
    return err, int(tie.sum())


# ------------------------------------------------------------------ fp32 (SIMT)
def test_tiny_moe_f32_config():
    """B=2, S=16, H=64, I=256, E=4, k=1, coef 0.01, fp32."""
    w = WORKLOADS["tiny_moe_f32"]
    inp = make_workload_inputs(w)
    full_moe_check(inp, w.k, w.coef, "f32")


@pytest.mark.parametrize("T,H,I,E,k", [(77, 64, 96, 5, 2), (45, 32, 64, 6, 3), (33, 64, 128, 4, 4)])
def test_moe_f32_ragged(T, H, I, E, k):
    full_moe_check(moe_inputs(T, H, I, E, "f32", seed=3), k, 0.01, "f32")


def test_dense_f32():
    inp = make_inputs(70, 64, 256, "f32", seed=4)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"])
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["f32"]


# ------------------------------------------------------------------ bf16 tensor cores
@pytest.mark.parametrize("T", [1, 100, 300, 1000])
def test_dense_bf16_tensor(T):
    inp = make_inputs(T, 256, 384, "bf16", seed=T)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="tensor")
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("T,H,I", [(3500, 1536, 512), (3400, 1408, 320)])
def test_dense_bf16_tensor_wide_down_tiles(T, H, I):
    """Shapes whose down GEMM takes 384-wide tiles (256-wide ones would need a
    second wave): two N = 192 MMAs per k-step into one accumulator; the
    second case ends in a tile with 256 valid columns."""
    inp = make_inputs(T, H, I, "bf16", seed=T + 17)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="tensor")
    torch.cuda.synchronize()
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


def test_moe_top1_wide_down_tiles():
    """Top-1 over 4 experts at T = 6000, H = 768: 384-wide down tiles with
    the rows scattered back to their tokens."""
    full_moe_check(moe_inputs(6000, 768, 384, 4, "bf16", seed=19), 1, 0.01, "bf16", path="tensor")


@pytest.mark.parametrize("T,H,I,E,k,bias", [
    (1000, 256, 384, 4, 1, None),
    (777, 256, 320, 8, 2, (1.5, 0.5, 0, 0, 0, 0, 0, 0)),
    (513, 128, 192, 6, 3, None),
    (260, 192, 256, 4, 4, None),
    (130, 64, 128, 1, 1, None),
    (1, 256, 384, 8, 2, None),
])
def test_moe_bf16_tensor(T, H, I, E, k, bias):
    full_moe_check(moe_inputs(T, H, I, E, "bf16", seed=7, bias=bias), k, 0.01, "bf16", path="tensor")


@pytest.mark.parametrize("T,path", [(300, "tensor"), (300, "simt"), (16, "auto"), (40, "stream_tc"),
                                    (3, "stream")])
def test_moe_max_experts_and_topk(T, path):
    """The build's limits: 64 experts, top-8 (k * E = 512 groups on the
    tensor path), with every path that takes the shape."""
    full_moe_check(moe_inputs(T, 256, 192, 64, "bf16", seed=150 + T), 8, 0.01, "bf16", path=path)


@pytest.mark.parametrize("T,path", [(2000, "tensor"), (300, "simt"), (40, "stream_tc"), (3, "stream")])
def test_moe_all_tokens_to_one_expert(T, path):
    """Degenerate routing: a logit bias of +8 on expert 3 makes it every
    token's first choice and -8 on experts 5-7 keeps them unselected, so the
    slot-0 group of expert 3 holds all T rows and eleven of the sixteen
    (slot, expert) groups are empty."""
    bias = (0.0, 0.0, 0.0, 8.0, 0.0, -8.0, -8.0, -8.0)
    inp = moe_inputs(T, 256, 320, 8, "bf16", seed=170 + T, bias=bias)
    full_moe_check(inp, 2, 0.01, "bf16", path=path)
    _, idx, _, _ = run_moe(inp, 2, 0.01, path)
    idx = np.asarray(idx)
    assert (idx[:, 0] == 3).all()
    assert not np.isin(idx, (5, 6, 7)).any()


@pytest.mark.parametrize("T,E,k", [(300, 4, 1), (257, 8, 2)])
def test_moe_bf16_simt_second_path(T, E, k):
    full_moe_check(moe_inputs(T, 128, 192, E, "bf16", seed=9), k, 0.01, "bf16", path="simt")


def test_tensor_and_simt_paths_agree_on_routing():
    inp = moe_inputs(400, 256, 256, 8, "bf16", seed=11)
    a = run_moe(inp, 2, 0.01, "tensor")
    b = run_moe(inp, 2, 0.01, "simt")
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[2], b[2]) and a[3] == b[3]
    assert rel_err(a[0], b[0]) < 2e-2


def test_uniform_router_tie_break_on_gpu():
    """Wr = 0 -> p = 1/E for every token -> experts 0..k-1, alpha = 1/k, aux = k*coef."""
    inp = moe_inputs(200, 128, 128, 8, "bf16", seed=12)
    inp["Wr"] = torch.zeros_like(inp["Wr"])
    y, idx, w, aux = run_moe(inp, 3, 0.01, "tensor")
    assert np.all(idx == np.arange(3)[None, :])
    assert np.allclose(w, 1.0 / 3, atol=1e-7)
    assert abs(aux - 0.03) < 1e-6


def test_moe_deterministic():
    inp = moe_inputs(900, 256, 256, 8, "bf16", seed=13)
    a = run_moe(inp, 2, 0.01)
    b = run_moe(inp, 2, 0.01)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1]) and a[3] == b[3]


def test_route_only_entry_point():
    inp = moe_inputs(5000, 768, 64, 8, "bf16", seed=14, bias=(1.5, 0.5, 0, 0, 0, 0, 0, 0))
    g = to_dev(inp)
    idx, w, aux, counts = mm.moe_route(g["x"], g["Wr"], 2, 0.01, logit_bias=g["logit_bias"])
    torch.cuda.synchronize()
    i64 = inputs64(inp)
    ref = oracle.moe_route(i64["x"], i64["Wr"], 2, 0.01, i64["logit_bias"])
    tie, diff = check_route(idx.cpu().numpy(), w.cpu().numpy(), float(aux), ref, 2)
    if not diff.any():
        assert counts.cpu().numpy().tolist() == ref["counts"].tolist()


def test_dense_empty_input():
    x = torch.empty(0, 256, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(384, 256, dtype=torch.bfloat16, device="cuda")
    Wd = torch.zeros(256, 384, dtype=torch.bfloat16, device="cuda")
    y = mm.swiglu_ffn(x, W, W, Wd)
    assert y.shape == (0, 256)


# ------------------------------------------------------------------ decode streaming path
@pytest.mark.parametrize("T", [1, 3, 8])
def test_dense_stream_path(T):
    inp = make_inputs(T, 768, 2432, "bf16", seed=40 + T)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="stream")
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("T,E,k,bias", [(1, 8, 2, None), (4, 8, 2, (1.5, 0.5, 0, 0, 0, 0, 0, 0)),
                                        (8, 4, 1, None), (5, 6, 3, None)])
def test_moe_stream_path(T, E, k, bias):
    full_moe_check(moe_inputs(T, 768, 2432, E, "bf16", seed=50 + T, bias=bias), k, 0.01, "bf16",
                   path="stream")


def test_stream_path_is_bf16_only():
    inp = make_inputs(5, 64, 256, "f32", seed=61)
    g = to_dev(inp)
    with pytest.raises(RuntimeError, match="MM_ERR_UNSUPPORTED"):
        mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="stream")


# ------------------------------------------------------------------ decode on the tensor cores
@pytest.mark.parametrize("T", [1, 5, 16, 17, 40, 64, 100, 128])
def test_dense_stream_tc_path(T):
    inp = make_inputs(T, 768, 2432, "bf16", seed=80 + T)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="stream_tc")
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("T,H,I", [(7, 256, 384), (33, 384, 320), (64, 128, 64), (64, 1024, 256),
                                   (20, 2048, 192), (17, 1792, 8192)])
def test_dense_stream_tc_small_shapes(T, H, I):
    """Several output m-blocks, a ragged last block of I (320 = 2.5 x 128),
    the smallest admissible shape, split gate/up ranges, and (the last) the
    down product per I-block with one (G, U) TMEM buffer."""
    inp = make_inputs(T, H, I, "bf16", seed=90 + T)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="stream_tc")
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("T,E,k,bias", [(1, 8, 2, None), (4, 8, 2, (1.5, 0.5, 0, 0, 0, 0, 0, 0)),
                                        (16, 8, 2, None), (33, 4, 1, None),
                                        (64, 8, 2, (1.5, 0.5, 0, 0, 0, 0, 0, 0)), (9, 6, 3, None),
                                        (20, 1, 1, None), (12, 16, 4, None), (64, 16, 4, None),
                                        (16, 8, 2, (8.0, 8.0, 0, 0, 0, 0, 0, 0))])
def test_moe_stream_tc_path(T, E, k, bias):
    """The last case routes every token to experts 0 and 1: the experts
    streamed before the routing is known but never selected add nothing."""
    full_moe_check(moe_inputs(T, 768, 2432, E, "bf16", seed=100 + T, bias=bias), k, 0.01, "bf16",
                   path="stream_tc")


@pytest.mark.parametrize("T,H,I,E,k", [(64, 1024, 256, 4, 2), (48, 1152, 256, 4, 2),
                                       (16, 256, 192, 32, 4)])
def test_moe_stream_tc_shapes(T, H, I, E, k):
    """The first two: y^T does not fit in TMEM beside the gate/up accumulators,
    so h goes through global memory between the two products.  The last: the
    down product runs per (expert, I-block) unit, with a half-empty last
    I-block (192 = 1.5 x 128)."""
    full_moe_check(moe_inputs(T, H, I, E, "bf16", seed=130 + T), k, 0.01, "bf16", path="stream_tc")


def test_moe_stream_tc_deterministic():
    inp = moe_inputs(40, 768, 2432, 8, "bf16", seed=121)
    a = run_moe(inp, 2, 0.01, path="stream_tc")
    b = run_moe(inp, 2, 0.01, path="stream_tc")
    assert all(np.array_equal(u, v) for u, v in zip(a[:3], b[:3])) and a[3] == b[3]


def test_stream_tc_shape_limits():
    """H must be a multiple of 128 and I of 64; the dense FFN streams up to 128
    tokens, the MoE layer up to 64; beyond that the path is refused."""
    inp = make_inputs(5, 192, 256, "bf16", seed=122)
    g = to_dev(inp)
    with pytest.raises(RuntimeError, match="MM_ERR_UNSUPPORTED"):
        mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="stream_tc")
    inp = make_inputs(129, 256, 256, "bf16", seed=123)
    g = to_dev(inp)
    with pytest.raises(RuntimeError, match="MM_ERR_UNSUPPORTED"):
        mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], path="stream_tc")
    with pytest.raises(RuntimeError, match="MM_ERR_UNSUPPORTED"):
        run_moe(moe_inputs(65, 256, 256, 4, "bf16", seed=124), 2, 0.01, path="stream_tc")


@pytest.mark.parametrize("T", [1, 4, 16, 64])
def test_decode_workloads(T):
    """The decode-shaped workloads at full size, in the launch configuration the
    benchmark uses (path chosen automatically)."""
    w = WORKLOADS[f"decode_moe_e8k2_t{T}"]
    full_moe_check(make_workload_inputs(w), w.k, w.coef, "bf16")
    w = WORKLOADS[f"decode_dense_t{T}"]
    inp = make_workload_inputs(w)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"])
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("E,k", [(64, 8), (8, 2), (32, 4)])
def test_moe_back_to_back_calls(E, k):
    """Calls issued back to back on the tensor path, on fresh zeroed
    workspaces and then on one reused workspace with new inputs (so new
    routing) each call: every result matches the oracle.  The grouped GEMMs
    launch before the dispatch kernel has written the group offsets
    (programmatic dependent launch), so this catches a kernel that reads
    them before waiting for it."""
    T, H, I = 300, 256, 192
    ws = mm.new_workspace(mm.moe_workspace_bytes(T, H, I, E, k, torch.bfloat16))
    for call in range(6):
        inp = moe_inputs(T, H, I, E, "bf16", seed=300 + 10 * E + call)
        g = to_dev(inp)
        y, idx, w, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, 0.01,
                                        path="tensor", workspace=ws if call >= 3 else None)
        torch.cuda.synchronize()
        i64 = inputs64(inp)
        ref = oracle.moe_forward(i64["x"], i64["Wr"], i64["Wg"], i64["Wu"], i64["Wd"], k, 0.01)
        tie, diff = check_route(idx.cpu().numpy(), w.cpu().numpy(), float(aux), ref, k)
        yref = ref["y"].copy()
        if diff.any():
            rows = np.nonzero(diff)[0]
            yref[rows] = ref_y_rows(i64, ref, idx.cpu().numpy(), rows, k)
        err = rel_err(y.double().cpu().numpy(), yref)
        assert err <= Y_TOL["bf16"], f"call {call}: y rel err {err}"


# ------------------------------------------------------------------ full-size workloads
@pytest.mark.parametrize("name", ["dense_t4096", "dense_t100"])
def test_dense_full_size(name):
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    g = to_dev(inp)
    y = mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"])
    torch.cuda.synchronize()
    ref = oracle.swiglu_ffn(*[to_f64(inp[n]) for n in ("x", "Wg", "Wu", "Wd")])
    assert rel_err(y.double().cpu().numpy(), ref) <= Y_TOL["bf16"]


@pytest.mark.parametrize("name", ["moe_e4k1_t8192", "moe_e8k2_t16384_skew"])
def test_moe_full_size(name):
    """The two prefill MoE workloads at full size, path chosen automatically:
    every routing output and every row of y against the oracle (the near-tie
    count is in the assertion messages and the run's summary)."""
    w = WORKLOADS[name]
    inp = make_workload_inputs(w)
    err, n_tie = full_moe_check(inp, w.k, w.coef, "bf16")
    assert err <= Y_TOL["bf16"]


# ------------------------------------------------------------------ CUDA graphs
@pytest.mark.parametrize("T", [4, 40, 600])
def test_moe_forward_graph_capture_replays_identically(T):
    """The forward allocates nothing and issues only stream work once warmed up,
    so it can be captured in a CUDA graph; replays reproduce the eager result."""
    inp = moe_inputs(T, 768, 2432, 8, "bf16", seed=70)
    g = to_dev(inp)
    dt = torch.bfloat16
    ws = mm.new_workspace(mm.moe_workspace_bytes(T, 768, 2432, 8, 2, dt))
    y = torch.empty(T, 768, dtype=dt, device="cuda")
    idx = torch.empty(T, 2, dtype=torch.int32, device="cuda")
    w = torch.empty(T, 2, dtype=torch.float32, device="cuda")
    aux = torch.empty((), dtype=torch.float32, device="cuda")

    def call():
        mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01, out=y, topk_idx=idx,
                       topk_w=w, aux_loss=aux, workspace=ws)

    call()
    torch.cuda.synchronize()
    eager = (y.clone(), idx.clone(), w.clone(), aux.clone())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    y.zero_()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(y, eager[0]) and torch.equal(idx, eager[1])
    assert torch.equal(w, eager[2]) and torch.equal(aux, eager[3])


# ------------------------------------------------------------------ fp16 range of h
@pytest.mark.parametrize("scale,expect", [(1.0, 0), (2000.0, 6)])
def test_fp16_h_overflow_is_reported(scale, expect):
    """The bf16 prefill path keeps h = SiLU(g) * u in fp16.  With x scaled by
    2000 (weights N(0, 0.02), H = 256) g and u are ~ 600, so |h| reaches
    ~ 3e5, beyond fp16's 65504: the call must report MM_ERR_RANGE through
    mm_check_status instead of leaving a silent inf in y.  Unscaled inputs
    report nothing; the status clears once read."""
    inp = make_inputs(300, 256, 384, "bf16", seed=31)
    x = (inp["x"].float() * scale).to(torch.bfloat16)
    g = to_dev(inp)
    ws = mm.new_workspace(mm.ffn_workspace_bytes(300, 256, 384, torch.bfloat16))
    mm.swiglu_ffn(x.cuda(), g["Wg"], g["Wu"], g["Wd"], workspace=ws, path="tensor")
    assert mm.check_status(ws) == expect
    assert mm.check_status(ws) == 0


def test_fp16_h_overflow_is_reported_by_the_moe_forward():
    inp = moe_inputs(400, 256, 320, 4, "bf16", seed=32)
    inp["x"] = (inp["x"].float() * 2000.0).to(torch.bfloat16)
    g = to_dev(inp)
    ws = mm.new_workspace(mm.moe_workspace_bytes(400, 256, 320, 4, 2, torch.bfloat16))
    mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01, workspace=ws,
                   path="tensor")
    assert mm.check_status(ws) == 6


# ------------------------------------------------------------------ watchdog
def test_watchdog_reports_timeout_and_recovers():
    ws = mm.new_workspace(256)
    assert mm.check_status(ws) == 0
    mm.watchdog_selftest(ws, 2000)          # 2 ms wait that nothing ends
    assert mm.check_status(ws) == 5          # MM_ERR_TIMEOUT
    assert mm.check_status(ws) == 0          # cleared
    # the context is still usable
    inp = make_inputs(64, 128, 128, "bf16", seed=2)
    g = to_dev(inp)
    mm.swiglu_ffn(g["x"], g["Wg"], g["Wu"], g["Wd"], workspace=None)
    torch.cuda.synchronize()


# ------------------------------------------------------------------ permute-free gate/up
@pytest.mark.parametrize("T,H,I,E,k,bias", [
    (1000, 256, 384, 4, 1, None),
    (777, 256, 320, 8, 2, (1.5, 0.5, 0, 0, 0, 0, 0, 0)),
    (300, 256, 192, 64, 8, None),
    (1, 256, 384, 8, 2, None),
    (2000, 256, 320, 8, 2, (0.0, 0.0, 0.0, 8.0, 0.0, -8.0, -8.0, -8.0)),
])
def test_moe_gather_path_matches_copy_path(T, H, I, E, k, bias):
    """The gate/up GEMM gathering x rows by token index (TMA gather4, no
    permuted copy) reads the same rows as the copy path: the same MMAs on
    the same values, so every output is bit-identical."""
    inp = moe_inputs(T, H, I, E, "bf16", seed=1100 + T, bias=bias)
    a = run_moe(inp, k, 0.01, "tensor")
    b = run_moe(inp, k, 0.01, "tensor_gather")
    assert all(np.array_equal(u, v) for u, v in zip(a[:3], b[:3])) and a[3] == b[3]


@pytest.mark.parametrize("name", ["moe_e4k1_t8192", "moe_e8k2_t16384_skew"])
def test_moe_gather_path_full_size(name):
    w = WORKLOADS[name]
    full_moe_check(make_workload_inputs(w), w.k, w.coef, "bf16", path="tensor_gather")


def test_moe_gather_path_runs_in_its_smaller_workspace():
    """Without the permuted copy of x the gathering path needs T*k*H*2 bytes
    less workspace; the copy path refuses that smaller workspace."""
    from swiglu_mlp_top_gb300 import _lib as L
    T, H, I, E, k = 1500, 256, 320, 8, 2
    lib = L.load()
    small = lib.mm_moe_workspace_bytes_for_path(T, H, I, E, k, L.MM_DTYPE_BF16, L.MM_PATH_TENSOR_GATHER)
    full = lib.mm_moe_workspace_bytes_for_path(T, H, I, E, k, L.MM_DTYPE_BF16, L.MM_PATH_TENSOR)
    assert full - small >= T * k * H * 2
    inp = moe_inputs(T, H, I, E, "bf16", seed=1200)
    g = to_dev(inp)
    ws = mm.new_workspace(small)
    y, idx, w, aux = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, 0.01,
                                    workspace=ws, path="tensor_gather")
    torch.cuda.synchronize()
    ref = run_moe(inp, k, 0.01, "tensor")
    assert np.array_equal(y.double().cpu().numpy(), ref[0])
    with pytest.raises(RuntimeError, match="MM_ERR_WORKSPACE"):
        mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], k, 0.01, workspace=ws,
                       path="tensor")


# ------------------------------------------------------------------ prepared down weights
def test_prepared_down_weights_give_the_same_outputs():
    """The fp16 copy of Wd made once (mm_prepare_down_weights) is the copy the
    tensor-core path makes inside every call: the outputs agree bit for bit
    (MoE top-2 and the dense FFN), and the forward no longer converts."""
    inp = moe_inputs(1500, 256, 320, 8, "bf16", seed=1300, bias=(1.5, 0.5, 0, 0, 0, 0, 0, 0))
    g = to_dev(inp)
    wd16 = [mm.prepare_down_weights(w) for w in g["Wd"]]
    a = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01,
                       logit_bias=g["logit_bias"], path="tensor")
    b = mm.moe_forward(g["x"], g["Wr"], g["Wg"], g["Wu"], g["Wd"], 2, 0.01,
                       logit_bias=g["logit_bias"], path="tensor", wd_f16=wd16)
    torch.cuda.synchronize()
    assert all(torch.equal(u, v) for u, v in zip(a, b))
    d = make_inputs(700, 256, 384, "bf16", seed=1301)
    gd = to_dev(d)
    y0 = mm.swiglu_ffn(gd["x"], gd["Wg"], gd["Wu"], gd["Wd"], path="tensor")
    y1 = mm.swiglu_ffn(gd["x"], gd["Wg"], gd["Wu"], gd["Wd"], path="tensor",
                       wd_f16=mm.prepare_down_weights(gd["Wd"]))
    torch.cuda.synchronize()
    assert torch.equal(y0, y1)
    assert torch.equal(wd16[0], g["Wd"][0].to(torch.float16))     # exact conversion


def test_prepare_down_weights_reports_the_fp16_range():
    ws = mm.new_workspace(256)
    Wd = torch.zeros(64, 64, dtype=torch.bfloat16, device="cuda")
    Wd[3, 5] = 70000.0
    mm.prepare_down_weights(Wd, status_workspace=ws)
    assert mm.check_status(ws) == 6
    Wd[3, 5] = 60000.0
    mm.prepare_down_weights(Wd, status_workspace=ws)
    assert mm.check_status(ws) == 0
