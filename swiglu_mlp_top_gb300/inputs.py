"""Seeded synthetic inputs and the named workloads.

This module holds no arithmetic of the method: it only draws random numbers
(CPU ``torch.Generator``, seed 0 unless told otherwise), rounds them to the
compute dtype and lays them out.  Both the CUDA path (through the tests and
the benchmark) and the fp64 oracle consume what it returns.

Recipe (the same for every workload):
  * draw order: x, then the router Wr (MoE only), then per expert e:
    Wg[e], Wu[e], Wd[e];
  * x ~ N(0, 1); every weight ~ N(0, 0.02);
  * drawn in float32; bf16 workloads round each tensor to bf16
    (round-to-nearest-even) and that rounded value is the input of both
    sides;
  * nn.Linear layout: Wg, Wu [I, H]; Wd [H, I]; Wr [E, H]; x [T, H].
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional, Sequence

import torch

WEIGHT_STD = 0.02


def intermediate_size(hidden: int) -> int:
    """MiniMind's default I = ceil(H * pi / 64) * 64 (768 -> 2432)."""
    return int(math.ceil(hidden * math.pi / 64) * 64)


@dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "dense" or "moe"
    T: int
    H: int
    I: int
    dtype: str                # "bf16" or "f32"
    E: int = 1
    k: int = 1
    coef: float = 0.0
    logit_bias: Optional[Sequence[float]] = None
    note: str = ""
    shape_bs: tuple = field(default=(0, 0))   # (B, S) as stated for the workload


H_MM = 768
I_MM = intermediate_size(H_MM)   # 2432

WORKLOADS = {
    # Tiny fp32 MoE: B=2, S=16, H=64, I=256, E=4, k=1, coef 0.01.
    "tiny_moe_f32": Workload("tiny_moe_f32", "moe", 32, 64, 256, "f32", E=4, k=1,
                             coef=0.01, shape_bs=(2, 16)),
    # Dense SwiGLU, MiniMind default H=768, I=2432, B=8 x S=512.
    "dense_t4096": Workload("dense_t4096", "dense", 4096, H_MM, I_MM, "bf16",
                            shape_bs=(8, 512)),
    # Same FFN at the pages' example shape B=1, S=100.
    "dense_t100": Workload("dense_t100", "dense", 100, H_MM, I_MM, "bf16",
                           shape_bs=(1, 100)),
    # MiniMind-shaped MoE: E=4, k=1, B=8 x S=1024, near-uniform load.
    "moe_e4k1_t8192": Workload("moe_e4k1_t8192", "moe", 8192, H_MM, I_MM, "bf16",
                               E=4, k=1, coef=0.01, shape_bs=(8, 1024)),
    # Top-2 MoE with skewed load: E=8, B=16 x S=1024, logit bias +1.5 on expert 0
    # and +0.5 on expert 1.
    "moe_e8k2_t16384_skew": Workload("moe_e8k2_t16384_skew", "moe", 16384, H_MM, I_MM,
                                     "bf16", E=8, k=2, coef=0.01,
                                     logit_bias=(1.5, 0.5, 0, 0, 0, 0, 0, 0),
                                     shape_bs=(16, 1024)),
}
for _T in (1, 4, 16, 64):
    WORKLOADS[f"decode_dense_t{_T}"] = Workload(
        f"decode_dense_t{_T}", "dense", _T, H_MM, I_MM, "bf16", shape_bs=(_T, 1))
    WORKLOADS[f"decode_moe_e8k2_t{_T}"] = Workload(
        f"decode_moe_e8k2_t{_T}", "moe", _T, H_MM, I_MM, "bf16", E=8, k=2, coef=0.01,
        shape_bs=(_T, 1))


def torch_dtype(dtype: str) -> torch.dtype:
    if dtype == "bf16":
        return torch.bfloat16
    if dtype == "f32":
        return torch.float32
    raise ValueError(f"unknown dtype {dtype!r}")


def _draw(gen: torch.Generator, shape, std: float, dtype: str) -> torch.Tensor:
    t = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        t = t * std
    return t.to(torch_dtype(dtype)).contiguous()


def make_inputs(T: int, H: int, I: int, dtype: str, E: int = 0, seed: int = 0,
                logit_bias: Optional[Sequence[float]] = None) -> dict:
    """Draw one problem's inputs on the CPU.

    E = 0 gives a dense FFN problem (x, Wg, Wu, Wd); E >= 1 an MoE problem
    (x, Wr, per-expert lists Wg, Wu, Wd, and the optional float32 logit bias).
    """
    gen = torch.Generator().manual_seed(seed)
    out = {"x": _draw(gen, (T, H), 1.0, dtype)}
    if E == 0:
        out["Wg"] = _draw(gen, (I, H), WEIGHT_STD, dtype)
        out["Wu"] = _draw(gen, (I, H), WEIGHT_STD, dtype)
        out["Wd"] = _draw(gen, (H, I), WEIGHT_STD, dtype)
        return out
    out["Wr"] = _draw(gen, (E, H), WEIGHT_STD, dtype)
    Wg, Wu, Wd = [], [], []
    for _ in range(E):
        Wg.append(_draw(gen, (I, H), WEIGHT_STD, dtype))
        Wu.append(_draw(gen, (I, H), WEIGHT_STD, dtype))
        Wd.append(_draw(gen, (H, I), WEIGHT_STD, dtype))
    out["Wg"], out["Wu"], out["Wd"] = Wg, Wu, Wd
    out["logit_bias"] = (None if logit_bias is None
                         else torch.tensor(list(logit_bias), dtype=torch.float32))
    return out


def make_workload_inputs(w: Workload, seed: int = 0, T: Optional[int] = None) -> dict:
    """Inputs for a named workload (optionally with a different token count)."""
    return make_inputs(T if T is not None else w.T, w.H, w.I, w.dtype,
                       E=(w.E if w.kind == "moe" else 0), seed=seed,
                       logit_bias=w.logit_bias)


def to_f64(t) -> "numpy.ndarray":  # noqa: F821
    """Exact upcast of a CPU tensor (or list of tensors) to float64 numpy."""
    if isinstance(t, (list, tuple)):
        return [to_f64(a) for a in t]
    if t is None:
        return None
    return t.detach().to("cpu", torch.float64).numpy()


def make_router_noise(T: int, E: int, std: float, seed: int = 1) -> torch.Tensor:
    """Router noise draws: [T, E] float32 ~ N(0, std^2) from its own seeded
    CPU generator.  The method adds them to the logits; the draw itself is
    an input, shared by the CUDA path and the oracle."""
    gen = torch.Generator().manual_seed(seed)
    return (torch.randn(T, E, generator=gen, dtype=torch.float32) * std).contiguous()
