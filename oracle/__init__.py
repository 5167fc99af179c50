"""FP64 CPU oracle for the RoPE + attention core -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path never does.

The arithmetic lives in ``sa_oracle.c`` (plain C, double precision, pthreads);
this module compiles it with gcc on first use and marshals numpy arrays.

Functions and what they follow:

* ``rope``        -- rotate-half RoPE in FP64, base 10000 (HF discussion #3,
                     "The bug": ``apply_rotary_pos_emb`` computes in FP32 and
                     casts back; here FP64 without a cast).
* ``round_to``    -- round-to-nearest-even cast to fp16 / bf16 (the cast-back of
                     the RoPE function's final cast, same section).
* ``rmsnorm``     -- FP64 RMSNorm of a row over the head dim with a learned
                     gamma (the pages keep RMSNorm next to attention in FP32,
                     sa3_trt README "Notes on the design").
* ``rope_attn``   -- the full core: RoPE, cast-back, exact two-pass softmax
                     attention, the differential subtraction (HF discussion #6,
                     "How the kernels differ") and the symmetric sliding window
                     (same page, "Three gotchas"); optionally RMSNorm of every
                     q and k row before RoPE.

Every function is pinned by ``tests/test_oracle_pins.py`` against library
routines (numpy fp16 casts, torch float64 SDPA), closed forms and invariants.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sa_oracle.c")
_LIB = os.path.join(_HERE, "libsa_oracle.so")
_lock = threading.Lock()
_lib = None

DTYPES = {"fp16": 0, "bf16": 1, "fp32": 2}
CASTS = {"method": 0, "exact": 1}


def build(force: bool = False) -> str:
    """Compile sa_oracle.c into libsa_oracle.so (gcc, -O2, IEEE semantics)."""
    if not force and os.path.exists(_LIB) and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-D_POSIX_C_SOURCE=200809L", "-fPIC", "-shared",
           "-fno-fast-math", "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.POINTER
            lib.sa_oracle_rope.argtypes = [P(ctypes.c_double), P(ctypes.c_int32), ctypes.c_int64,
                                           ctypes.c_int, ctypes.c_double, P(ctypes.c_double)]
            lib.sa_oracle_rope.restype = ctypes.c_int
            lib.sa_oracle_round_array.argtypes = [P(ctypes.c_double), ctypes.c_int64, ctypes.c_int,
                                                  P(ctypes.c_double)]
            lib.sa_oracle_round_array.restype = None
            lib.sa_oracle_fp16_to_double.argtypes = [ctypes.c_uint16]
            lib.sa_oracle_fp16_to_double.restype = ctypes.c_double
            lib.sa_oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            lib.sa_oracle_bf16_to_double.restype = ctypes.c_double
            lib.sa_oracle_fp32_to_double.argtypes = [ctypes.c_uint32]
            lib.sa_oracle_fp32_to_double.restype = ctypes.c_double
            lib.sa_oracle_rope_attn.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, P(ctypes.c_int32),
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, P(ctypes.c_double), ctypes.c_int, ctypes.c_int, ctypes.c_double,
                P(ctypes.c_int64), ctypes.c_int64, P(ctypes.c_double), ctypes.c_int]
            lib.sa_oracle_rope_attn.restype = ctypes.c_int
            lib.sa_oracle_rope_attn_qknorm.argtypes = [
                ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p, P(ctypes.c_int32),
                ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                ctypes.c_int, P(ctypes.c_double), ctypes.c_int, ctypes.c_int, ctypes.c_double,
                ctypes.c_int, P(ctypes.c_double), P(ctypes.c_double), ctypes.c_double,
                P(ctypes.c_int64), ctypes.c_int64, P(ctypes.c_double), ctypes.c_int]
            lib.sa_oracle_rope_attn_qknorm.restype = ctypes.c_int
            lib.sa_oracle_rmsnorm.argtypes = [P(ctypes.c_double), ctypes.c_int64, ctypes.c_int,
                                              P(ctypes.c_double), ctypes.c_double, P(ctypes.c_double)]
            lib.sa_oracle_rmsnorm.restype = ctypes.c_int
            _lib = lib
    return _lib


def _ptr(a: Optional[np.ndarray], ctype):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


def rope(x: np.ndarray, positions: Optional[np.ndarray] = None, base: float = 10000.0) -> np.ndarray:
    """FP64 rotate-half RoPE of rows x[..., d] at positions (default: row index)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32).reshape(-1)
    if pos is not None and pos.shape[0] != flat.shape[0]:
        raise ValueError("positions must have one entry per row")
    y = np.empty_like(flat)
    rc = lib.sa_oracle_rope(_ptr(flat, ctypes.c_double), _ptr(pos, ctypes.c_int32), flat.shape[0], d,
                            float(base), _ptr(y, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"sa_oracle_rope failed ({rc})")
    return y.reshape(x.shape)


def rmsnorm(x: np.ndarray, gamma: Optional[np.ndarray] = None, eps: float = 1e-6) -> np.ndarray:
    """FP64 RMSNorm of rows x[..., d]: x * gamma / sqrt(mean(x^2) + eps) (gamma None: ones)."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    d = x.shape[-1]
    flat = x.reshape(-1, d)
    g = None if gamma is None else np.ascontiguousarray(gamma, dtype=np.float64).reshape(-1)
    if g is not None and g.shape[0] != d:
        raise ValueError("gamma must have d entries")
    y = np.empty_like(flat)
    rc = lib.sa_oracle_rmsnorm(_ptr(flat, ctypes.c_double), flat.shape[0], d, _ptr(g, ctypes.c_double),
                               float(eps), _ptr(y, ctypes.c_double))
    if rc != 0:
        raise ValueError(f"sa_oracle_rmsnorm failed ({rc})")
    return y.reshape(x.shape)


def round_to(x: np.ndarray, dtype: str) -> np.ndarray:
    """Round doubles to the nearest fp16/bf16/FP32 value (ties to even), returned as double."""
    lib = _load()
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    lib.sa_oracle_round_array(_ptr(x, ctypes.c_double), x.size, DTYPES[dtype], _ptr(y, ctypes.c_double))
    return y


def bits_to_double(bits: np.ndarray, dtype: str) -> np.ndarray:
    lib = _load()
    if dtype == "fp32":
        b = np.ascontiguousarray(bits, dtype=np.uint32).reshape(-1)
        return np.array([lib.sa_oracle_fp32_to_double(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))
    f = lib.sa_oracle_bf16_to_double if dtype == "bf16" else lib.sa_oracle_fp16_to_double
    b = np.ascontiguousarray(bits, dtype=np.uint16).reshape(-1)
    return np.array([f(int(x)) for x in b], dtype=np.float64).reshape(np.shape(bits))


def rope_attn(q: np.ndarray, k: np.ndarray, v: np.ndarray, *, B: int, H: int, L: int, d: int = 64,
              nmaps: int = 1, dv: int = 64, dtype: str = "fp16", window: int = -1,
              lam: Optional[np.ndarray] = None, positions: Optional[np.ndarray] = None,
              cast: str = "method", base: float = 10000.0, rows: Optional[np.ndarray] = None,
              threads: Optional[int] = None, qk_norm: Optional[tuple] = None) -> np.ndarray:
    """RoPE + attention core in FP64.

    q, k: uint16 bits, [B, H, L, d] (nmaps=1) or [B, H, 2, L, d] (nmaps=2);
    v: uint16 bits [B, H, L, dv] (dtype "fp32": uint32 bits of FP32 values).  rows: flattened ids (b*H + h)*L + i, or None
    for every row.  qk_norm: None, or (gamma_q, gamma_k, eps) to RMSNorm every q
    and k row before RoPE (a gamma of None means ones).  Returns double
    [len(rows), dv] (or [B, H, L, dv] for None).
    """
    lib = _load()
    bt, ct = (np.uint32, ctypes.c_uint32) if dtype == "fp32" else (np.uint16, ctypes.c_uint16)
    q = np.ascontiguousarray(q, dtype=bt)
    k = np.ascontiguousarray(k, dtype=bt)
    v = np.ascontiguousarray(v, dtype=bt)
    if q.size != B * H * nmaps * L * d or k.size != q.size or v.size != B * H * L * dv:
        raise ValueError("shape mismatch")
    lam64 = None
    if nmaps == 2:
        if lam is None:
            raise ValueError("differential attention needs lambda")
        lam64 = np.ascontiguousarray(np.broadcast_to(np.asarray(lam, dtype=np.float64), (H,)))
    pos = None if positions is None else np.ascontiguousarray(positions, dtype=np.int32)
    if pos is not None and pos.shape != (L,):
        raise ValueError("positions must be [L]")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    nrows = B * H * L if r is None else r.shape[0]
    out = np.empty((nrows, dv), dtype=np.float64)
    gq = gk = None
    eps = 0.0
    if qk_norm is not None:
        gq, gk, eps = qk_norm
        gq = None if gq is None else np.ascontiguousarray(gq, dtype=np.float64).reshape(-1)
        gk = None if gk is None else np.ascontiguousarray(gk, dtype=np.float64).reshape(-1)
        if (gq is not None and gq.shape[0] != d) or (gk is not None and gk.shape[0] != d):
            raise ValueError("gamma must have d entries")
    rc = lib.sa_oracle_rope_attn_qknorm(
        ctypes.cast(_ptr(q, ct), ctypes.c_void_p), ctypes.cast(_ptr(k, ct), ctypes.c_void_p),
        ctypes.cast(_ptr(v, ct), ctypes.c_void_p),
        _ptr(pos, ctypes.c_int32), B, H, L, d, nmaps, dv, int(window), _ptr(lam64, ctypes.c_double),
        DTYPES[dtype], CASTS[cast], float(base), int(qk_norm is not None), _ptr(gq, ctypes.c_double),
        _ptr(gk, ctypes.c_double), float(eps), _ptr(r, ctypes.c_int64), nrows,
        _ptr(out, ctypes.c_double), int(threads or default_threads()))
    if rc != 0:
        raise ValueError(f"sa_oracle_rope_attn failed ({rc})")
    if r is None:
        return out.reshape(B, H, L, dv)
    return out


def rope_attn_workload(inputs: dict, rows: Optional[np.ndarray] = None, cast: str = "method",
                       threads: Optional[int] = None, qk_norm: Optional[tuple] = None) -> np.ndarray:
    """Convenience: run the oracle on a ``synth.make_inputs`` dict."""
    w = inputs["workload"]
    return rope_attn(inputs["q"], inputs["k"], inputs["v"], B=w.B, H=w.H, L=w.L, d=w.d,
                     nmaps=w.nmaps, dv=w.dv, dtype=w.dtype, window=w.window, lam=inputs["lam"],
                     positions=inputs["positions"], cast=cast, rows=rows, threads=threads,
                     qk_norm=qk_norm)
