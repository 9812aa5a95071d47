"""GB300 (sm_103a) SwiGLU FFN and top-k MoE forward behind a C ABI (libmm.so).

Public API: swiglu_ffn, moe_forward, moe_route, check_status (see api.py);
the C entry points are declared in include/mm.h.
"""
from .api import (  # noqa: F401
    swiglu_ffn_backward, moe_backward, swiglu_block, prepare_down_weights,
    swiglu_ffn, swiglu_ffn_noalloc, moe_forward, moe_route, check_status, watchdog_selftest,
    ffn_workspace_bytes, moe_workspace_bytes, new_workspace,
)
