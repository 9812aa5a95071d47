"""mm_swiglu_ffn_noalloc: the dense FFN for callers that cannot allocate
device memory, running on the library's fixed device scratch.

It must give the same output as mm_swiglu_ffn with a caller-owned
workspace, bit for bit, on two calls in a row, so the scratch is reused
correctly, for every kernel family the automatic path picks.
This file is collected last so that a run stopping at its first failure has
already run every other test.  It passes on its own in a fresh process and
after the other tests.
"""
import pytest
import torch

from swiglu_mlp_top_gb300 import _lib as L
from swiglu_mlp_top_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


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


# Token counts that take each kernel family the automatic path picks: the
# CUDA-core streaming kernel (1, 4 tokens), the tensor-core streaming kernel
# with the tokens as the M operand (64, 100), and the tensor-core GEMMs (300,
# 1000).  The streaming kernels keep grid-barrier counters in the scratch
# header, so each case runs twice in a row on the same array.
@pytest.mark.parametrize("T", [1, 4, 64, 100, 300, 1000])
def test_noalloc_matches_workspace_entry_point_twice(T):
    import __graft_entry__
    __graft_entry__.build()
    lib = L.load()
    H, I = 768, 2432
    for call in range(2):                                # two calls in a row, new inputs each
        inp = make_inputs(T, H, I, "bf16", seed=20 + 2 * T + call)
        g = {n: v.cuda() for n, v in inp.items()}
        y_ref = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        assert _call_workspace(lib, g, y_ref, T, H, I) == L.MM_OK
        y = torch.full((T, H), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _call_noalloc(lib, g, y, T, H, I) == L.MM_OK
        torch.cuda.synchronize()
        # the same kernels on the same inputs: every kernel is deterministic,
        # so the two results agree bit for bit
        assert torch.equal(y, y_ref), f"T={T} call {call}: noalloc result differs"


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
