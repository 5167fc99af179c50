"""Seeded synthetic inputs for the RoPE + attention core.

This module only draws random numbers and encodes them as fp16/bf16 bit
patterns.  It holds none of the attention arithmetic: both the FP64 oracle
(``oracle/``) and the CUDA path (``diffusion_transformer_attention_rope_gb300``)
receive the very same bytes from here and neither imports the other.

The five named workloads are the Stable Audio 3 attention shapes:

* ``tiny``               B=1 H=2  L=64   d=64 fp16 standard attention
* ``dit_l1292``          B=1 H=16 L=1292 d=64 fp16 standard attention (DiT, ~120 s of audio)
* ``dit_l4096_outliers`` B=1 H=24 L=4096 d=64 fp16, 1% of K entries scaled by 8
* ``diff_l4096``         B=1 H=16 L=4096 differential, d=64 / d_v=128 bf16, lambda=0.8
* ``swa_diff_l8192``     B=1 H=16 L=8192 differential + |i-j|<=256 window, bf16,
                         per-head lambda ~ U(0.2, 0.8)

Two more on the same shape: SAME-L's own window of +-17 (bf16), and the FP32-input
form of the +-256 window workload (FP32 q, k, v: SAME-L's FP32 attention
projections, whose products the method runs in TF32).

Recipe (fixed order of draws from ``numpy.random.PCG64(seed)``):
q, k, v as float32 N(0, 1); then, if requested, a Bernoulli(p) outlier mask
over k that multiplies the hit entries by ``k_outlier_scale``; then lambda.
Each tensor is rounded once, round-to-nearest-even, from float32 to the
storage dtype (FP32 inputs keep the drawn float32 values).  Layouts: standard q/k/v ``[B, H, L, d]``; differential q/k
``[B, H, 2, L, d]`` (map 0 = Q1/K1, map 1 = Q2/K2) and v ``[B, H, L, d_v]``.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = ["Workload", "WORKLOADS", "get_workload", "make_inputs", "encode", "decode"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    L: int
    d: int = 64
    nmaps: int = 1           # 1 = standard attention, 2 = differential attention
    dv: int = 64
    dtype: str = "fp16"      # "fp16" | "bf16" | "fp32"
    window: int = -1         # < 0: full attention; else |i - j| <= window
    seed: int = 0
    k_outlier_frac: float = 0.0
    k_outlier_scale: float = 1.0
    lam: Optional[tuple] = None   # None | ("const", x) | ("uniform", lo, hi)

    @property
    def differential(self) -> bool:
        return self.nmaps == 2

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny", B=1, H=2, L=64, seed=0),
        Workload("dit_l1292", B=1, H=16, L=1292, seed=1),
        Workload("dit_l4096_outliers", B=1, H=24, L=4096, seed=2,
                 k_outlier_frac=0.01, k_outlier_scale=8.0),
        Workload("diff_l4096", B=1, H=16, L=4096, nmaps=2, dv=128, dtype="bf16",
                 seed=3, lam=("const", 0.8)),
        Workload("swa_diff_l8192", B=1, H=16, L=8192, nmaps=2, dv=128, dtype="bf16",
                 window=256, seed=4, lam=("uniform", 0.2, 0.8)),
        # SAME-L's own window, +-17 (HF discussion #6 "sm_120 SAME-L", "Three gotchas"), on the
        # shape of the window workload above: a measurement case beyond the five configurations
        Workload("swa17_diff_l8192", B=1, H=16, L=8192, nmaps=2, dv=128, dtype="bf16",
                 window=17, seed=5, lam=("uniform", 0.2, 0.8)),
        # the FP32-input form of the window workload (SAME-L's FP32 attention projections,
        # TF32 products; same page, "How the kernels differ")
        Workload("swa_diff_l8192_fp32", B=1, H=16, L=8192, nmaps=2, dv=128, dtype="fp32",
                 window=256, seed=6, lam=("uniform", 0.2, 0.8)),
    ]
}


def get_workload(name: str) -> Workload:
    return WORKLOADS[name]


def encode(x32: np.ndarray, dtype: str) -> np.ndarray:
    """float32 -> uint16 bit patterns of fp16 / bf16, round to nearest even (uint32 bit
    patterns of the float32 values themselves for "fp32")."""
    x32 = np.ascontiguousarray(x32, dtype=np.float32)
    if dtype == "fp32":
        return x32.view(np.uint32).copy()
    if dtype == "fp16":
        return x32.astype(np.float16).view(np.uint16)
    if dtype == "bf16":
        u = x32.view(np.uint32).astype(np.uint64)
        nan = np.isnan(x32)
        r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
        r = r.astype(np.uint16)
        r[nan] = 0x7FC0
        return r
    raise ValueError(f"unknown dtype {dtype!r}")


def decode(bits: np.ndarray, dtype: str) -> np.ndarray:
    """uint16 (uint32 for "fp32") bit patterns -> float32 (exact)."""
    if dtype == "fp32":
        return np.ascontiguousarray(bits, dtype=np.uint32).view(np.float32).copy()
    bits = np.ascontiguousarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float32)
    if dtype == "bf16":
        return (bits.astype(np.uint32) << 16).view(np.float32)
    raise ValueError(f"unknown dtype {dtype!r}")


def make_inputs(w: Workload, seed: Optional[int] = None) -> dict:
    """Draw the workload's inputs.

    Returns a dict with ``q``, ``k``, ``v`` (uint16 bit patterns, C-contiguous),
    ``lam`` (float32 [H] or None), ``positions`` (None: 0..L-1) and the workload.
    """
    seed = w.seed if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed))
    if w.nmaps == 1:
        qk_shape = (w.B, w.H, w.L, w.d)
    else:
        qk_shape = (w.B, w.H, 2, w.L, w.d)
    v_shape = (w.B, w.H, w.L, w.dv)
    q = rng.standard_normal(qk_shape, dtype=np.float32)
    k = rng.standard_normal(qk_shape, dtype=np.float32)
    v = rng.standard_normal(v_shape, dtype=np.float32)
    if w.k_outlier_frac > 0.0:
        hit = rng.random(qk_shape, dtype=np.float32) < np.float32(w.k_outlier_frac)
        k = np.where(hit, k * np.float32(w.k_outlier_scale), k).astype(np.float32)
    lam = None
    if w.lam is not None:
        if w.lam[0] == "const":
            lam = np.full((w.H,), w.lam[1], dtype=np.float32)
        elif w.lam[0] == "uniform":
            lam = rng.uniform(w.lam[1], w.lam[2], size=(w.H,)).astype(np.float32)
        else:
            raise ValueError(f"unknown lambda recipe {w.lam!r}")
    elif w.nmaps == 2:
        raise ValueError("differential workload needs a lambda recipe")
    return {
        "q": encode(q, w.dtype),
        "k": encode(k, w.dtype),
        "v": encode(v, w.dtype),
        "lam": lam,
        "positions": None,
        "workload": w,
    }
