"""The C-ABI library: it loads, exports every symbol include/mm.h declares,
and rejects bad arguments synchronously (no compute call, no GPU needed)."""
import ctypes as C
import os
import re

import pytest

from swiglu_mlp_top_gb300 import _lib as L

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "mm.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(mm_[a-z0-9_]+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__ as g
    g.build()
    return L.load()


def test_header_declares_expected_entry_points():
    fns = header_functions()
    for name in ("mm_swiglu_ffn", "mm_moe_forward", "mm_moe_workspace_bytes", "mm_check_status",
                 "mm_status_string"):
        assert name in fns


def test_every_declared_symbol_is_exported(lib):
    fns = header_functions()
    raw = C.CDLL(L.LIB_PATH)
    for name in fns:
        assert hasattr(raw, name), name
    # the binding covers exactly the header
    assert set(L.SIGNATURES) == set(fns)


def test_status_strings(lib):
    assert lib.mm_status_string(0) == b"MM_OK"
    assert lib.mm_status_string(5) == b"MM_ERR_TIMEOUT"
    assert lib.mm_status_string(6) == b"MM_ERR_RANGE"
    assert lib.mm_version() >= 100


def test_workspace_sizes(lib):
    bf16 = L.MM_DTYPE_BF16
    T, H, I, E, k = 16384, 768, 2432, 8, 2
    ws = lib.mm_moe_workspace_bytes(T, H, I, E, k, bf16)
    # at least the permuted activations and h: T*k*(H + I) bf16 values
    assert ws >= T * k * (H + I) * 2
    assert lib.mm_moe_workspace_bytes(T, H, I, E, 9, bf16) == 0         # k > E
    assert lib.mm_moe_workspace_bytes(T, H, I, 65, 2, bf16) == 0        # E > max
    assert lib.mm_swiglu_ffn_workspace_bytes(4096, H, I, bf16) >= 4096 * I * 2
    assert lib.mm_swiglu_ffn_workspace_bytes(0, H, I, bf16) == 256 + H * I * 2   # fp16 Wd copy
    assert lib.mm_moe_route_workspace_bytes(0, 8, 2) == 0
    assert lib.mm_moe_workspace_bytes(T, H, I, 16, 9, bf16) == 0        # k > MM_MAX_TOPK


def test_bad_arguments_rejected_before_any_launch(lib):
    fake = C.c_void_p(1 << 20)      # never dereferenced: validation fails first
    bf16 = L.MM_DTYPE_BF16
    rc = lib.mm_swiglu_ffn(fake, fake, fake, fake, fake, 10, 768, 2432, 7, fake, 1 << 30, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # bad dtype
    rc = lib.mm_swiglu_ffn(None, fake, fake, fake, fake, 10, 768, 2432, bf16, fake, 1 << 30, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # null x
    rc = lib.mm_swiglu_ffn(C.c_void_p((1 << 20) + 2), fake, fake, fake, fake, 10, 768, 2432, bf16,
                           fake, 1 << 30, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # misaligned x
    rc = lib.mm_swiglu_ffn(fake, fake, fake, fake, fake, 10, 768, 2432, bf16, fake, 10, None)
    assert rc == L.MM_ERR_WORKSPACE                         # workspace too small
    rc = lib.mm_swiglu_ffn_ex(fake, fake, fake, fake, fake, 10, 100, 2432, bf16, fake, 1 << 30,
                              None, L.MM_PATH_TENSOR)
    assert rc == L.MM_ERR_UNSUPPORTED                       # H not a multiple of 64
    rc = lib.mm_swiglu_ffn(fake, fake, fake, fake, fake, 0, 768, 2432, bf16, None, 0, None)
    assert rc == L.MM_OK                                    # empty input: nothing to do
    ptrs, keep = L.ptr_array([1 << 20] * 4)
    args = dict(T=10, H=768, I=2432, E=4, k=5)
    rc = lib.mm_moe_forward(fake, fake, ptrs, ptrs, ptrs, args["T"], args["H"], args["I"],
                            args["E"], args["k"], 0.01, bf16, None, fake, fake, fake, fake, fake,
                            1 << 34, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # k > E
    rc = lib.mm_moe_forward(fake, fake, ptrs, ptrs, ptrs, 0, 768, 2432, 4, 1, 0.01, bf16, None,
                            fake, fake, fake, fake, fake, 1 << 34, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # T = 0
    rc = lib.mm_moe_forward(fake, fake, ptrs, ptrs, ptrs, 10, 768, 2432, 4, 1, 0.01, bf16, None,
                            fake, fake, fake, fake, fake, 100, None)
    assert rc == L.MM_ERR_WORKSPACE
    rc = lib.mm_watchdog_selftest(fake, 256, 0, None)
    assert rc == L.MM_ERR_INVALID_ARG
    del keep


def test_backward_workspace_layout(lib):
    """The backward workspaces hold dh and the per-assignment dx rows in fp16
    (2 bytes each) beside the bf16 operands: dense T*I*(2 dh + 4 dG|dU + 2 h)
    bytes plus the 256-byte header; MoE R*(6H + 8I) bytes for the padded rows
    R = T*k + 63*E (x, dy, dx rows: 2H each; dh, alpha*h: 2I; dG|dU: 4I) plus
    small per-block partials."""
    bf16 = L.MM_DTYPE_BF16
    T, H, I = 4096, 768, 2432
    assert lib.mm_swiglu_ffn_backward_workspace_bytes(T, H, I, bf16) == 256 + T * I * 8
    T, E, k = 16384, 8, 2
    R = T * k + 63 * E
    ws = lib.mm_moe_backward_workspace_bytes(T, H, I, E, k, bf16)
    core = R * (6 * H + 8 * I)
    assert core <= ws <= core + 16 * 2 ** 20
    assert lib.mm_moe_backward_workspace_bytes(T, H, I, E, k, L.MM_DTYPE_F32) == 0
    assert lib.mm_moe_backward_workspace_bytes(T, H, I, E, 9, bf16) == 0          # k > E


def test_backward_bad_arguments_rejected_before_any_launch(lib):
    fake = C.c_void_p(1 << 20)      # never dereferenced: validation fails first
    bf16, f32 = L.MM_DTYPE_BF16, L.MM_DTYPE_F32
    wsb = 1 << 34
    rc = lib.mm_swiglu_ffn_backward(fake, fake, fake, fake, fake, 10, 768, 2432, f32, fake, fake,
                                    fake, fake, fake, wsb, None)
    assert rc == L.MM_ERR_UNSUPPORTED                       # bf16 only
    rc = lib.mm_swiglu_ffn_backward(fake, fake, fake, fake, fake, 10, 100, 2432, bf16, fake, fake,
                                    fake, fake, fake, wsb, None)
    assert rc == L.MM_ERR_UNSUPPORTED                       # H not a multiple of 64
    rc = lib.mm_swiglu_ffn_backward(fake, fake, fake, fake, fake, 10, 768, 2432, bf16, None, fake,
                                    fake, fake, fake, wsb, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # null dx
    rc = lib.mm_swiglu_ffn_backward(fake, fake, fake, fake, fake, 10, 768, 2432, bf16, fake, fake,
                                    fake, fake, fake, 100, None)
    assert rc == L.MM_ERR_WORKSPACE                         # workspace too small
    ptrs, keep = L.ptr_array([1 << 20] * 4)
    common = (fake, fake, ptrs, ptrs, ptrs)
    rc = lib.mm_moe_backward(*common, 10, 768, 2432, 4, 5, 0.01, bf16, fake, fake, fake, fake,
                             fake, 1.0, 0.0, 0.0, fake, fake, ptrs, ptrs, ptrs, None, fake, wsb, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # k > E
    rc = lib.mm_moe_backward(*common, 10, 768, 2432, 4, 2, 0.01, bf16, fake, fake, fake, None,
                             fake, 1.0, 1e-3, 1.0, fake, fake, ptrs, ptrs, ptrs, None, fake, wsb, None)
    assert rc == L.MM_ERR_INVALID_ARG                       # z-loss asked for without lse
    rc = lib.mm_moe_backward(*common, 10, 768, 2432, 4, 2, 0.01, bf16, fake, fake, fake, fake,
                             fake, 1.0, 0.0, 0.0, fake, fake, ptrs, ptrs, ptrs, None, fake, 100, None)
    assert rc == L.MM_ERR_WORKSPACE                         # workspace too small
    del keep
