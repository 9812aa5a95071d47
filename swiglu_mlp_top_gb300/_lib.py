"""ctypes binding of the C ABI declared in include/mm.h (libmm.so, built in-tree).

Loading fails loudly when the library is missing: there is no fallback.
"""
from __future__ import annotations

import ctypes as C
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libmm.so")

(MM_OK, MM_ERR_INVALID_ARG, MM_ERR_UNSUPPORTED, MM_ERR_WORKSPACE, MM_ERR_CUDA, MM_ERR_TIMEOUT,
 MM_ERR_RANGE) = range(7)
MM_DTYPE_F32, MM_DTYPE_BF16 = 0, 1
(MM_PATH_AUTO, MM_PATH_TENSOR, MM_PATH_STREAM, MM_PATH_SIMT, MM_PATH_STREAM_TC,
 MM_PATH_TENSOR_GATHER) = 0, 1, 2, 3, 4, 5
MM_MAX_EXPERTS = 64
MM_MAX_TOPK = 8
MM_NOALLOC_SCRATCH_BYTES = 16 << 20

_vp, _i32, _i64, _f32, _sz = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t
_pp = C.POINTER(C.c_void_p)


class MoeOptions(C.Structure):
    """mm_moe_options (include/mm.h), field for field."""
    _fields_ = [("path", C.c_int), ("logit_noise", C.c_void_p), ("z_coef", C.c_float),
                ("z_loss", C.c_void_p), ("router_probs", C.c_void_p),
                ("router_lse", C.c_void_p), ("norm_weight", C.c_void_p),
                ("norm_eps", C.c_float), ("residual", C.c_int), ("wd_f16", C.c_void_p),
                ("separate_routing", C.c_int)]


_opt = C.POINTER(MoeOptions)

# name -> (restype, argtypes); mirrors include/mm.h
SIGNATURES = {
    "mm_status_string": (C.c_char_p, [_i32]),
    "mm_version": (_i32, []),
    "mm_last_error": (C.c_char_p, []),
    "mm_swiglu_ffn_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32]),
    "mm_swiglu_ffn": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp, _sz, _vp]),
    "mm_swiglu_ffn_ex": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp, _sz, _vp,
                                _i32]),
    "mm_swiglu_ffn_noalloc": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp]),
    "mm_prepare_down_weights": (_i32, [_vp, _vp, _i32, _i32, _vp, _vp]),
    "mm_swiglu_ffn_prepared": (_i32, [_vp, _vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp,
                                      _sz, _vp, _i32]),
    "mm_moe_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32]),
    "mm_moe_workspace_bytes_for_path": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32, _i32]),
    "mm_moe_forward": (_i32, [_vp, _vp, _pp, _pp, _pp, _i64, _i32, _i32, _i32, _i32, _f32, _i32,
                              _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp]),
    "mm_moe_forward_ex": (_i32, [_vp, _vp, _pp, _pp, _pp, _i64, _i32, _i32, _i32, _i32, _f32,
                                 _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _i32]),
    "mm_moe_forward_opts": (_i32, [_vp, _vp, _pp, _pp, _pp, _i64, _i32, _i32, _i32, _i32, _f32,
                                   _i32, _vp, _vp, _vp, _vp, _vp, _vp, _sz, _vp, _opt]),
    "mm_moe_route_workspace_bytes": (_sz, [_i64, _i32, _i32]),
    "mm_moe_route_opts": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _vp,
                                 _vp, _vp, _sz, _vp, _opt]),
    "mm_moe_route": (_i32, [_vp, _vp, _i64, _i32, _i32, _i32, _f32, _i32, _vp, _vp, _vp, _vp,
                            _vp, _vp, _sz, _vp]),
    "mm_swiglu_ffn_block_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32]),
    "mm_swiglu_ffn_block": (_i32, [_vp, _vp, _f32, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32,
                                   _vp, _sz, _vp]),
    "mm_swiglu_ffn_backward_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32]),
    "mm_swiglu_ffn_backward": (_i32, [_vp, _vp, _vp, _vp, _vp, _i64, _i32, _i32, _i32, _vp, _vp,
                                      _vp, _vp, _vp, _sz, _vp]),
    "mm_moe_backward_workspace_bytes": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32]),
    "mm_moe_backward": (_i32, [_vp, _vp, _pp, _pp, _pp, _i64, _i32, _i32, _i32, _i32, _f32, _i32,
                               _vp, _vp, _vp, _vp, _vp, _f32, _f32, _f32, _vp, _vp, _pp, _pp, _pp,
                               _vp, _vp, _sz, _vp]),
    "mm_check_status": (_i32, [_vp, _vp]),
    "mm_watchdog_selftest": (_i32, [_vp, _sz, C.c_uint32, _vp]),
    "mm_launch_count": (C.c_uint64, []),
    "mm_profile_start": (_i32, [_i32, _i32]),
    "mm_profile_stop": (_i32, [C.POINTER(C.c_double), C.POINTER(C.c_int)]),
}
MM_KERNEL_ROUTER, MM_KERNEL_DISPATCH, MM_KERNEL_GATEUP, MM_KERNEL_DOWN, MM_KERNEL_DECODE = 1, 3, 4, 5, 7
MM_KERNEL_BWD_DGRAD, MM_KERNEL_BWD_SWIGLU, MM_KERNEL_BWD_WGRAD, MM_KERNEL_BWD_ROUTER = 8, 9, 10, 11

_lib = None


class MMError(RuntimeError):
    def __init__(self, code: int, what: str):
        lib = load()
        name = lib.mm_status_string(code).decode()
        detail = lib.mm_last_error().decode() if code == MM_ERR_CUDA else ""
        super().__init__(f"{what}: {name}" + (f" ({detail})" if detail else ""))
        self.code = code


def load():
    """Load libmm.so once and attach the signatures of include/mm.h."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(
            f"{LIB_PATH} is missing: build it first (python -c 'import __graft_entry__ as g; g.build()')")
    lib = C.CDLL(LIB_PATH)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(code: int, what: str) -> None:
    if code != MM_OK:
        raise MMError(code, what)


def ptr_array(ptrs):
    arr = (C.c_void_p * max(1, len(ptrs)))(*[C.c_void_p(p) for p in ptrs])
    return C.cast(arr, _pp), arr   # keep `arr` alive while the call runs
