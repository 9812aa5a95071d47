"""mm_swiglu_ffn_noalloc: the dense FFN for callers that cannot allocate
device memory, running on the library's fixed device scratch.

It must give the same output as mm_swiglu_ffn with a caller-owned
workspace, on two calls in a row, so the scratch is reused correctly.
This file is collected last so that a run stopping at its first failure has
already run every other test.  It passes on its own in a fresh process and
after the other tests.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from swiglu_mlp_top_gb300 import _lib as L
from swiglu_mlp_top_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

Y_TOL_BF16 = 2e-2     # the bf16 tolerance of the parity tests (max |dy| / rms)


def _call_noalloc(lib, g, y, T, H, I):
    stream = torch.cuda.current_stream().cuda_stream
    return lib.mm_swiglu_ffn_noalloc(g["x"].data_ptr(), g["Wg"].data_ptr(), g["Wu"].data_ptr(),
                                     g["Wd"].data_ptr(), y.data_ptr(), T, H, I,
                                     L.MM_DTYPE_BF16, stream)


def _call_workspace(lib, g, y, T, H, I):
    need = lib.mm_swiglu_ffn_workspace_bytes(T, H, I, L.MM_DTYPE_BF16)
    ws = torch.zeros(need, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    rc = lib.mm_swiglu_ffn(g["x"].data_ptr(), g["Wg"].data_ptr(), g["Wu"].data_ptr(),
                           g["Wd"].data_ptr(), y.data_ptr(), T, H, I, L.MM_DTYPE_BF16,
                           ws.data_ptr(), need, stream)
    torch.cuda.synchronize()
    return rc


def _rel(a, b):
    a = a.double().cpu().numpy()
    b = b.double().cpu().numpy()
    return float(np.abs(a - b).max() / np.sqrt((b ** 2).mean()))


def test_noalloc_matches_workspace_entry_point_twice():
    import __graft_entry__
    __graft_entry__.build()
    lib = L.load()
    H, I = 768, 2432
    for seed, T in ((21, 300), (22, 1000)):            # two calls in a row, new inputs each
        inp = make_inputs(T, H, I, "bf16", seed=seed)
        g = {n: v.cuda() for n, v in inp.items()}
        y_ref = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        assert _call_workspace(lib, g, y_ref, T, H, I) == L.MM_OK
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(lib, g, y, T, H, I) == L.MM_OK
        torch.cuda.synchronize()
        assert torch.isfinite(y.float()).all()
        assert _rel(y, y_ref) <= Y_TOL_BF16


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import __graft_entry__
    __graft_entry__.build()
    lib = L.load()
    H, I = 768, 2432
    T = 4096                                            # needs ~23.7 MB > 16 MiB
    assert lib.mm_swiglu_ffn_workspace_bytes(T, H, I, L.MM_DTYPE_BF16) > L.MM_NOALLOC_SCRATCH_BYTES
    x = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    W = torch.zeros(I, H, dtype=torch.bfloat16, device="cuda")
    Wd = torch.zeros(H, I, dtype=torch.bfloat16, device="cuda")
    y = torch.zeros(T, H, dtype=torch.bfloat16, device="cuda")
    g = {"x": x, "Wg": W, "Wu": W, "Wd": Wd}
    assert _call_noalloc(lib, g, y, T, H, I) == L.MM_ERR_UNSUPPORTED
