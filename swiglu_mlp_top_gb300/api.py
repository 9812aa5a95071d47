"""Python face of the C ABI: argument marshalling only.

torch supplies device memory and the current CUDA stream; every step of the
computation runs in the CUDA kernels of libmm.so.  Nothing here computes.
"""
from __future__ import annotations

import ctypes as C
from typing import Optional, Sequence

import torch

from . import _lib as L

_DTYPES = {torch.bfloat16: L.MM_DTYPE_BF16, torch.float32: L.MM_DTYPE_F32}
_PATHS = {"auto": L.MM_PATH_AUTO, "tensor": L.MM_PATH_TENSOR, "stream": L.MM_PATH_STREAM,
          "simt": L.MM_PATH_SIMT, "stream_tc": L.MM_PATH_STREAM_TC,
          "tensor_gather": L.MM_PATH_TENSOR_GATHER}


def _dev(t: torch.Tensor, name: str, dtype=None) -> int:
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _stream(stream) -> int:
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _dtype_code(x: torch.Tensor) -> int:
    if x.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {x.dtype}")
    return _DTYPES[x.dtype]


def ffn_workspace_bytes(T: int, H: int, I: int, dtype: torch.dtype) -> int:
    return int(L.load().mm_swiglu_ffn_workspace_bytes(T, H, I, _DTYPES[dtype]))


def moe_workspace_bytes(T: int, H: int, I: int, E: int, k: int, dtype: torch.dtype) -> int:
    return int(L.load().mm_moe_workspace_bytes(T, H, I, E, k, _DTYPES[dtype]))


def new_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Caller-owned scratch; the first 256 bytes hold the watchdog word and
    must start at zero."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def prepare_down_weights(Wd: torch.Tensor, *, status_workspace: Optional[torch.Tensor] = None,
                         stream=None) -> torch.Tensor:
    """The fp16 copy of a bf16 down-projection matrix for the tensor-core
    prefill path (mm_prepare_down_weights); values beyond the fp16 range are
    reported through check_status(status_workspace)."""
    H, I = Wd.shape
    out = torch.empty(H, I, dtype=torch.float16, device=Wd.device)
    rc = L.load().mm_prepare_down_weights(
        _dev(Wd, "Wd", torch.bfloat16), out.data_ptr(), H, I,
        None if status_workspace is None else _dev(status_workspace, "status_workspace"),
        _stream(stream))
    L.check(rc, "mm_prepare_down_weights")
    return out


def swiglu_ffn(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, *,
               out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
               path: str = "auto", stream=None,
               wd_f16: Optional[torch.Tensor] = None) -> torch.Tensor:
    """y = Wd (SiLU(Wg x) ⊙ Wu x) for x [T, H] (mm_swiglu_ffn; with wd_f16,
    the prepared fp16 down weights, mm_swiglu_ffn_prepared)."""
    lib = L.load()
    T, H = x.shape
    I = Wg.shape[0]
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    need = lib.mm_swiglu_ffn_workspace_bytes(T, H, I, dt)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    if wd_f16 is None:
        rc = lib.mm_swiglu_ffn_ex(
            _dev(x, "x"), _dev(Wg, "Wg", x.dtype), _dev(Wu, "Wu", x.dtype), _dev(Wd, "Wd", x.dtype),
            _dev(out, "out", x.dtype), T, H, I, dt, _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream), _PATHS[path])
    else:
        rc = lib.mm_swiglu_ffn_prepared(
            _dev(x, "x"), _dev(Wg, "Wg", x.dtype), _dev(Wu, "Wu", x.dtype), _dev(Wd, "Wd", x.dtype),
            _dev(wd_f16, "wd_f16", torch.float16), _dev(out, "out", x.dtype), T, H, I, dt,
            _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _stream(stream), _PATHS[path])
    L.check(rc, "mm_swiglu_ffn")
    return out


def swiglu_block(x: torch.Tensor, norm_weight: torch.Tensor, Wg: torch.Tensor,
                 Wu: torch.Tensor, Wd: torch.Tensor, *, norm_eps: float = 1e-5,
                 out: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    """y = x + FFN(RMSNorm(x)) (mm_swiglu_ffn_block): the dense FFN in its block."""
    lib = L.load()
    T, H = x.shape
    I = Wg.shape[0]
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    need = lib.mm_swiglu_ffn_block_workspace_bytes(T, H, I, dt)
    if workspace is None:
        workspace = new_workspace(need, x.device)
    rc = lib.mm_swiglu_ffn_block(
        _dev(x, "x"), _dev(norm_weight, "norm_weight", x.dtype), float(norm_eps),
        _dev(Wg, "Wg", x.dtype), _dev(Wu, "Wu", x.dtype), _dev(Wd, "Wd", x.dtype),
        _dev(out, "out", x.dtype), T, H, I, dt, _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    L.check(rc, "mm_swiglu_ffn_block")
    return out


def swiglu_ffn_noalloc(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor, *,
                       out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """mm_swiglu_ffn_noalloc: the dense FFN using the library's fixed device
    scratch instead of a workspace (for callers that cannot allocate)."""
    lib = L.load()
    T, H = x.shape
    I = Wg.shape[0]
    dt = _dtype_code(x)
    if out is None:
        out = torch.empty_like(x)
    rc = lib.mm_swiglu_ffn_noalloc(
        _dev(x, "x"), _dev(Wg, "Wg", x.dtype), _dev(Wu, "Wu", x.dtype), _dev(Wd, "Wd", x.dtype),
        _dev(out, "out", x.dtype), T, H, I, dt, _stream(stream))
    L.check(rc, "mm_swiglu_ffn_noalloc")
    return out


def _router_options(T: int, E: int, dev, path: str, logit_noise, z_coef, stats,
                    norm_weight=None, norm_eps=1e-5, residual=False, dtype=None, wd_f16=None):
    """mm_moe_options for the router variants, the block prologue / epilogue
    and prepared down weights; fills `stats` (a dict) with the output tensors
    it asks for: z_loss [], probs [T, E], lse [T] (fp32).  Returns (options,
    objects to keep alive during the call)."""
    o = L.MoeOptions()
    o.path = _PATHS[path]
    keep = None
    if wd_f16 is not None:
        pw, keep = L.ptr_array([_dev(w, "wd_f16", torch.float16) for w in wd_f16])
        o.wd_f16 = C.cast(pw, C.c_void_p)
    if norm_weight is not None:
        o.norm_weight = _dev(norm_weight, "norm_weight", dtype)
        o.norm_eps = float(norm_eps)
    o.residual = 1 if residual else 0
    if logit_noise is not None:
        if tuple(logit_noise.shape) != (T, E):
            raise ValueError(f"logit_noise must be [{T}, {E}]")
        o.logit_noise = _dev(logit_noise, "logit_noise", torch.float32)
    o.z_coef = float(z_coef or 0.0)
    if stats is not None:
        shapes = {"z_loss": (), "probs": (T, E), "lse": (T,)}
        for name, shape in shapes.items():
            if stats.get(name) is None:
                stats[name] = torch.empty(shape, dtype=torch.float32, device=dev)
        o.z_loss = _dev(stats["z_loss"], "z_loss", torch.float32)
        o.router_probs = _dev(stats["probs"], "probs", torch.float32)
        o.router_lse = _dev(stats["lse"], "lse", torch.float32)
    return o, keep


def moe_forward(x: torch.Tensor, Wr: torch.Tensor, Wg: Sequence[torch.Tensor],
                Wu: Sequence[torch.Tensor], Wd: Sequence[torch.Tensor], k: int, coef: float, *,
                logit_bias: Optional[torch.Tensor] = None, out: Optional[torch.Tensor] = None,
                topk_idx: Optional[torch.Tensor] = None, topk_w: Optional[torch.Tensor] = None,
                aux_loss: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                path: str = "auto", stream=None, logit_noise: Optional[torch.Tensor] = None,
                z_coef: float = 0.0, stats: Optional[dict] = None,
                norm_weight: Optional[torch.Tensor] = None, norm_eps: float = 1e-5,
                residual: bool = False, wd_f16: Optional[Sequence[torch.Tensor]] = None,
                separate_routing: bool = False):
    """Top-k MoE forward (mm_moe_forward; mm_moe_forward_opts when router
    noise, z-loss, router statistics, the block's norm / residual, prepared
    down weights or separate routing kernels are asked for).

    Returns (y [T,H], topk_idx [T,k] int32, topk_w [T,k] fp32, aux_loss [] fp32).
    With a dict `stats`, it also receives z_loss [] (z_coef * mean_t lse_t^2),
    probs [T, E] and lse [T] (fp32 device tensors).  With norm_weight the
    layer runs on RMSNorm(x); with residual, y = x + MoE(...).  wd_f16: the
    experts' prepared fp16 down weights (prepare_down_weights).
    separate_routing: the router and the permute as two kernels instead of
    one (same results; see mm_moe_options.separate_routing).
    """
    lib = L.load()
    T, H = x.shape
    E = len(Wg)
    I = Wg[0].shape[0]
    dt = _dtype_code(x)
    dev = x.device
    out = torch.empty_like(x) if out is None else out
    topk_idx = torch.empty(T, k, dtype=torch.int32, device=dev) if topk_idx is None else topk_idx
    topk_w = torch.empty(T, k, dtype=torch.float32, device=dev) if topk_w is None else topk_w
    aux_loss = torch.empty((), dtype=torch.float32, device=dev) if aux_loss is None else aux_loss
    need = lib.mm_moe_workspace_bytes(T, H, I, E, k, dt)
    if workspace is None:
        workspace = new_workspace(need, dev)
    pg, ag = L.ptr_array([_dev(w, "Wg", x.dtype) for w in Wg])
    pu, au = L.ptr_array([_dev(w, "Wu", x.dtype) for w in Wu])
    pd, ad = L.ptr_array([_dev(w, "Wd", x.dtype) for w in Wd])
    bias_ptr = None if logit_bias is None else _dev(logit_bias, "logit_bias", torch.float32)
    args = (_dev(x, "x"), _dev(Wr, "Wr", x.dtype), pg, pu, pd, T, H, I, E, k, float(coef), dt,
            bias_ptr, _dev(out, "out", x.dtype), _dev(topk_idx, "topk_idx", torch.int32),
            _dev(topk_w, "topk_w", torch.float32), _dev(aux_loss, "aux_loss", torch.float32),
            _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
            _stream(stream))
    if (logit_noise is None and not z_coef and stats is None and norm_weight is None
            and not residual and wd_f16 is None and not separate_routing):
        rc = lib.mm_moe_forward_ex(*args, _PATHS[path])
    else:
        o, keep = _router_options(T, E, dev, path, logit_noise, z_coef, stats, norm_weight,
                                  norm_eps, residual, x.dtype, wd_f16)
        o.separate_routing = 1 if separate_routing else 0
        rc = lib.mm_moe_forward_opts(*args, C.byref(o))
        del keep
    del ag, au, ad
    L.check(rc, "mm_moe_forward")
    return out, topk_idx, topk_w, aux_loss


def moe_route(x: torch.Tensor, Wr: torch.Tensor, k: int, coef: float, *,
              logit_bias: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
              stream=None, logit_noise: Optional[torch.Tensor] = None, z_coef: float = 0.0,
              stats: Optional[dict] = None):
    """Router only (mm_moe_route / mm_moe_route_opts): (topk_idx, topk_w,
    aux_loss, expert_counts); router variants and `stats` as moe_forward."""
    lib = L.load()
    T, H = x.shape
    E = Wr.shape[0]
    dt = _dtype_code(x)
    dev = x.device
    idx = torch.empty(T, k, dtype=torch.int32, device=dev)
    w = torch.empty(T, k, dtype=torch.float32, device=dev)
    aux = torch.empty((), dtype=torch.float32, device=dev)
    counts = torch.empty(E, dtype=torch.int32, device=dev)
    need = lib.mm_moe_route_workspace_bytes(T, E, k)
    if workspace is None:
        workspace = new_workspace(need, dev)
    bias_ptr = None if logit_bias is None else _dev(logit_bias, "logit_bias", torch.float32)
    args = (_dev(x, "x"), _dev(Wr, "Wr", x.dtype), T, H, E, k, float(coef), dt,
            bias_ptr, idx.data_ptr(), w.data_ptr(), aux.data_ptr(),
            counts.data_ptr(), _dev(workspace, "workspace"),
            workspace.numel() * workspace.element_size(), _stream(stream))
    if logit_noise is None and not z_coef and stats is None:
        rc = lib.mm_moe_route(*args)
    else:
        o, _ = _router_options(T, E, dev, "auto", logit_noise, z_coef, stats)
        rc = lib.mm_moe_route_opts(*args, C.byref(o))
    L.check(rc, "mm_moe_route")
    return idx, w, aux, counts


def swiglu_ffn_backward(x: torch.Tensor, Wg: torch.Tensor, Wu: torch.Tensor, Wd: torch.Tensor,
                        dy: torch.Tensor, *, workspace: Optional[torch.Tensor] = None,
                        stream=None):
    """Backward of the dense FFN (mm_swiglu_ffn_backward, bf16): returns
    (dx [T, H] bf16, dWg [I, H], dWu [I, H], dWd [H, I] fp32)."""
    lib = L.load()
    T, H = x.shape
    I = Wg.shape[0]
    dt = _dtype_code(x)
    dev = x.device
    dx = torch.empty_like(x)
    dWg = torch.empty(I, H, dtype=torch.float32, device=dev)
    dWu = torch.empty(I, H, dtype=torch.float32, device=dev)
    dWd = torch.empty(H, I, dtype=torch.float32, device=dev)
    need = lib.mm_swiglu_ffn_backward_workspace_bytes(T, H, I, dt)
    if workspace is None:
        workspace = new_workspace(need, dev)
    rc = lib.mm_swiglu_ffn_backward(
        _dev(x, "x"), _dev(Wg, "Wg", x.dtype), _dev(Wu, "Wu", x.dtype), _dev(Wd, "Wd", x.dtype),
        _dev(dy, "dy", x.dtype), T, H, I, dt, dx.data_ptr(), dWg.data_ptr(), dWu.data_ptr(),
        dWd.data_ptr(), _dev(workspace, "workspace"), workspace.numel() * workspace.element_size(),
        _stream(stream))
    L.check(rc, "mm_swiglu_ffn_backward")
    return dx, dWg, dWu, dWd


def moe_backward(x: torch.Tensor, Wr: torch.Tensor, Wg: Sequence[torch.Tensor],
                 Wu: Sequence[torch.Tensor], Wd: Sequence[torch.Tensor], k: int, coef: float,
                 topk_idx: torch.Tensor, topk_w: torch.Tensor, probs: torch.Tensor,
                 dy: torch.Tensor, *, d_aux: float = 1.0, lse: Optional[torch.Tensor] = None,
                 z_coef: float = 0.0, d_z: float = 1.0, bias_grad: bool = False,
                 workspace: Optional[torch.Tensor] = None, stream=None) -> dict:
    """Backward of the MoE layer (mm_moe_backward, bf16) from the forward's
    saved routing (topk_idx, topk_w, and the `stats` probs / lse of
    moe_forward).  Returns a dict: dx, dWr, dWg / dWu / dWd (lists of E
    fp32 tensors) and, with bias_grad, d_bias."""
    lib = L.load()
    T, H = x.shape
    E = len(Wg)
    I = Wg[0].shape[0]
    dt = _dtype_code(x)
    dev = x.device
    dx = torch.empty_like(x)
    dWr = torch.empty(E, H, dtype=torch.float32, device=dev)
    dWg = [torch.empty(I, H, dtype=torch.float32, device=dev) for _ in range(E)]
    dWu = [torch.empty(I, H, dtype=torch.float32, device=dev) for _ in range(E)]
    dWd = [torch.empty(H, I, dtype=torch.float32, device=dev) for _ in range(E)]
    d_bias = torch.empty(E, dtype=torch.float32, device=dev) if bias_grad else None
    need = lib.mm_moe_backward_workspace_bytes(T, H, I, E, k, dt)
    if workspace is None:
        workspace = new_workspace(need, dev)
    pg, ag = L.ptr_array([_dev(w, "Wg", x.dtype) for w in Wg])
    pu, au = L.ptr_array([_dev(w, "Wu", x.dtype) for w in Wu])
    pd, ad = L.ptr_array([_dev(w, "Wd", x.dtype) for w in Wd])
    qg, bg = L.ptr_array([t.data_ptr() for t in dWg])
    qu, bu = L.ptr_array([t.data_ptr() for t in dWu])
    qd, bd = L.ptr_array([t.data_ptr() for t in dWd])
    rc = lib.mm_moe_backward(
        _dev(x, "x"), _dev(Wr, "Wr", x.dtype), pg, pu, pd, T, H, I, E, k, float(coef), dt,
        _dev(topk_idx, "topk_idx", torch.int32), _dev(topk_w, "topk_w", torch.float32),
        _dev(probs, "probs", torch.float32),
        None if lse is None else _dev(lse, "lse", torch.float32), _dev(dy, "dy", x.dtype),
        float(d_aux), float(z_coef), float(d_z), dx.data_ptr(), dWr.data_ptr(), qg, qu, qd,
        None if d_bias is None else d_bias.data_ptr(), _dev(workspace, "workspace"),
        workspace.numel() * workspace.element_size(), _stream(stream))
    del ag, au, ad, bg, bu, bd
    L.check(rc, "mm_moe_backward")
    out = {"dx": dx, "dWr": dWr, "dWg": dWg, "dWu": dWu, "dWd": dWd}
    if d_bias is not None:
        out["d_bias"] = d_bias
    return out


def check_status(workspace: torch.Tensor, stream=None) -> int:
    """Synchronise and return the device watchdog status (0 = fine); clears it."""
    return int(L.load().mm_check_status(_dev(workspace, "workspace"), _stream(stream)))


def watchdog_selftest(workspace: torch.Tensor, limit_us: int, stream=None) -> None:
    rc = L.load().mm_watchdog_selftest(_dev(workspace, "workspace"),
                                       workspace.numel() * workspace.element_size(),
                                       int(limit_us), _stream(stream))
    L.check(rc, "mm_watchdog_selftest")
