import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Near-tie report of the routing comparisons this session ran."""
    try:
        from parity import ROUTE_REPORT
    except Exception:  # pragma: no cover
        return
    if not ROUTE_REPORT:
        return
    tr = terminalreporter
    tr.section("routing parity: near-tie tokens (gap < 1e-6) per comparison")
    tot_tok = sum(r["tokens"] for r in ROUTE_REPORT)
    tot_tie = sum(r["near_ties"] for r in ROUTE_REPORT)
    tot_flip = sum(r["near_tie_flips"] for r in ROUTE_REPORT)
    for r in ROUTE_REPORT:
        if r["near_ties"] or r["tokens"] >= 4096:
            tr.write_line(f"{r['test']}: {r['tokens']} tokens, {r['near_ties']} near-ties, "
                          f"{r['near_tie_flips']} flipped, {r['idx_mismatch_non_tie']} non-tie "
                          f"mismatches, max |dalpha| {r['topk_w_err']:.2e}, |daux| {r['aux_err']:.2e}")
    tr.write_line(f"total: {len(ROUTE_REPORT)} comparisons, {tot_tok} tokens, {tot_tie} near-tie "
                  f"tokens, {tot_flip} decided differently, "
                  f"{sum(r['idx_mismatch_non_tie'] for r in ROUTE_REPORT)} non-tie mismatches")
