"""GB300 (sm_103a) RoPE + attention core of the Stable Audio 3 DiT / SAME autoencoder.

Thin ctypes binding of ``libsa_attn.so`` (C ABI in ``include/sa_attn.h``).  The
functions below keep the C names and only marshal arguments; every step of the
computation runs in the library's CUDA kernels.  PyTorch is used only by the
``RopeAttention`` convenience wrapper, for device memory and streams.

There is no fallback: if the library has not been built, importing works but
every call raises ``SaAttnError`` with instructions.
"""

from __future__ import annotations

import ctypes
import os
import threading
from typing import Optional, Sequence

__all__ = [
    "SA_FP16", "SA_BF16", "SA_FP32", "SaAttnError", "sa_rope_attn_workspace_bytes", "sa_attn_fwd_workspace_bytes", "sa_rope_qkv_f32", "sa_attn_fwd_f32", "library_path", "load_library",
    "sa_attn_create", "sa_attn_destroy", "sa_rope_attn_workspace_size", "sa_attn_fwd_workspace_size", "sa_rope_table_bytes", "sa_rope_k", "sa_attn_fwd_rope_q", "sa_rope_attn",
    "sa_rope_qk", "sa_rope_attn_qknorm", "sa_qknorm_rope_qk", "sa_rope_attn_host",
    "sa_rope_attn_host_workspace_size", "sa_attn_fwd", "sa_rope_attn_noalloc", "sa_attn_check", "sa_attn_set_timeout", "sa_last_error", "sa_status_string", "RopeAttention",
]

SA_FP16 = 0
SA_BF16 = 1
SA_FP32 = 2   # differential attention with FP32 q, k, v, out (TF32 products)
STATUS_NAMES = {0: "SA_OK", 1: "SA_ERR_INVALID_ARG", 2: "SA_ERR_UNSUPPORTED", 3: "SA_ERR_CUDA",
                4: "SA_ERR_DEVICE_TIMEOUT", 5: "SA_ERR_NO_DEVICE", 6: "SA_ERR_WORKSPACE"}

_PKG = os.path.dirname(os.path.abspath(__file__))
_lock = threading.Lock()
_lib = None


class SaAttnError(RuntimeError):
    def __init__(self, status: int, message: str):
        self.status = status
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")


def library_path() -> str:
    return os.path.join(_PKG, "libsa_attn.so")


def load_library():
    """Load libsa_attn.so and declare the C signatures (raises if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise SaAttnError(3, f"{path} is missing: build it with "
                                 "`python -c 'import __graft_entry__ as g; g.build()'` "
                                 "(needs nvcc with sm_103a support)")
        lib = ctypes.CDLL(path)
        vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
        lib.sa_attn_create.argtypes = [ctypes.POINTER(vp), i, f]
        lib.sa_attn_create.restype = i
        lib.sa_attn_destroy.argtypes = [vp]
        lib.sa_attn_destroy.restype = i
        lib.sa_rope_attn_workspace_size.argtypes = [i, i, i, i, i]
        lib.sa_rope_attn_workspace_size.restype = sz
        lib.sa_rope_attn_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.sa_rope_attn_workspace_bytes.restype = sz
        lib.sa_attn_fwd_workspace_bytes.argtypes = [i, i, i, i, i, i]
        lib.sa_attn_fwd_workspace_bytes.restype = sz
        lib.sa_rope_qkv_f32.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, vp]
        lib.sa_rope_qkv_f32.restype = i
        lib.sa_attn_fwd_f32.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(f), vp]
        lib.sa_attn_fwd_f32.restype = i
        lib.sa_rope_attn.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                     ctypes.POINTER(f), i, vp, sz, vp]
        lib.sa_rope_attn.restype = i
        lib.sa_rope_qk.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.sa_rope_qk.restype = i
        lib.sa_rope_attn_host_workspace_size.argtypes = [i, i, i, i, i]
        lib.sa_rope_attn_host_workspace_size.restype = sz
        lib.sa_rope_attn_host.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(f), i, vp, sz, vp]
        lib.sa_rope_attn_host.restype = i
        lib.sa_rope_attn_qknorm.argtypes = [vp, vp, vp, vp, vp, ctypes.POINTER(f), ctypes.POINTER(f), f,
                                            vp, i, i, i, i, i, ctypes.POINTER(f), i, vp, sz, vp]
        lib.sa_rope_attn_qknorm.restype = i
        lib.sa_qknorm_rope_qk.argtypes = [vp, vp, vp, vp, ctypes.POINTER(f), ctypes.POINTER(f), f,
                                          vp, vp, i, i, i, i, i, i, vp]
        lib.sa_qknorm_rope_qk.restype = i
        lib.sa_rope_table_bytes.argtypes = [i]
        lib.sa_rope_table_bytes.restype = sz
        lib.sa_rope_k.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, vp]
        lib.sa_rope_k.restype = i
        lib.sa_attn_fwd_rope_q.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(f), i,
                                           vp, sz, vp]
        lib.sa_attn_fwd_rope_q.restype = i
        lib.sa_attn_fwd_workspace_size.argtypes = [i, i, i, i, i]
        lib.sa_attn_fwd_workspace_size.restype = sz
        lib.sa_attn_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, ctypes.POINTER(f), i, vp, sz, vp]
        lib.sa_attn_fwd.restype = i
        lib.sa_rope_attn_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i,
                                             ctypes.POINTER(f), i, vp]
        lib.sa_rope_attn_noalloc.restype = i
        lib.sa_attn_set_timeout.argtypes = [vp, ctypes.c_ulonglong]
        lib.sa_attn_set_timeout.restype = i
        lib.sa_attn_check.argtypes = [vp]
        lib.sa_attn_check.restype = i
        lib.sa_last_error.argtypes = []
        lib.sa_last_error.restype = ctypes.c_char_p
        lib.sa_status_string.argtypes = [i]
        lib.sa_status_string.restype = ctypes.c_char_p
        _lib = lib
        return lib


def _check(status: int) -> None:
    if status != 0:
        raise SaAttnError(status, sa_last_error())


def sa_last_error() -> str:
    return load_library().sa_last_error().decode()


def sa_status_string(status: int) -> str:
    return load_library().sa_status_string(int(status)).decode()


def sa_attn_create(device: int = 0, rope_base: float = 10000.0) -> int:
    h = ctypes.c_void_p()
    _check(load_library().sa_attn_create(ctypes.byref(h), int(device), float(rope_base)))
    return int(h.value)


def sa_attn_destroy(handle: int) -> None:
    _check(load_library().sa_attn_destroy(ctypes.c_void_p(handle)))


def sa_rope_attn_workspace_size(B: int, H: int, L: int, d: int, differential: bool) -> int:
    return int(load_library().sa_rope_attn_workspace_size(B, H, L, d, 1 if differential else 0))


def sa_rope_attn_workspace_bytes(B: int, H: int, L: int, d: int, differential: bool, dtype: int) -> int:
    return int(load_library().sa_rope_attn_workspace_bytes(B, H, L, d, 1 if differential else 0, int(dtype)))


def sa_attn_fwd_workspace_bytes(B: int, H: int, L: int, d: int, differential: bool, dtype: int) -> int:
    return int(load_library().sa_attn_fwd_workspace_bytes(B, H, L, d, 1 if differential else 0, int(dtype)))


def sa_rope_qkv_f32(handle: int, q: int, k: int, v: int, positions: Optional[int], q_rot: int, k_rot: int,
                    v_t: int, B: int, H: int, L: int, d: int, stream: Optional[int]) -> None:
    """The FP32 form's pre-pass: q', k' rotated and rounded to TF32, v transposed to v^T (TF32)."""
    _check(load_library().sa_rope_qkv_f32(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
        ctypes.c_void_p(positions), ctypes.c_void_p(q_rot), ctypes.c_void_p(k_rot), ctypes.c_void_p(v_t),
        int(B), int(H), int(L), int(d), ctypes.c_void_p(stream)))


def sa_attn_fwd_f32(handle: int, q_rot: int, k_rot: int, v_t: int, out: int, B: int, H: int, L: int, d: int,
                    window: int, lam: Sequence[float], stream: Optional[int]) -> None:
    """The FP32 form's TF32 attention kernel on the pre-pass's q', k', v^T."""
    _check(load_library().sa_attn_fwd_f32(
        ctypes.c_void_p(handle), ctypes.c_void_p(q_rot), ctypes.c_void_p(k_rot), ctypes.c_void_p(v_t),
        ctypes.c_void_p(out), int(B), int(H), int(L), int(d), int(window), _lam(lam), ctypes.c_void_p(stream)))


def sa_attn_fwd_workspace_size(B: int, H: int, L: int, d: int, differential: bool) -> int:
    return int(load_library().sa_attn_fwd_workspace_size(B, H, L, d, 1 if differential else 0))


def sa_rope_table_bytes(L: int) -> int:
    return int(load_library().sa_rope_table_bytes(int(L)))


def sa_rope_k(handle: int, k: int, positions: Optional[int], k_rot: int, cs_table: int, B: int, H: int,
              L: int, d: int, nmaps: int, dtype: int, stream: Optional[int]) -> None:
    """Enqueue the RoPE pass of k alone, also writing the (cos, sin) table for the Q prologue."""
    _check(load_library().sa_rope_k(
        ctypes.c_void_p(handle), ctypes.c_void_p(k), ctypes.c_void_p(positions), ctypes.c_void_p(k_rot),
        ctypes.c_void_p(cs_table), int(B), int(H), int(L), int(d), int(nmaps), int(dtype),
        ctypes.c_void_p(stream)))


def sa_attn_fwd_rope_q(handle: int, q: int, k_rot: int, cs_table: int, v: int, out: int, B: int, H: int,
                       L: int, d: int, window: int, lam: Optional[Sequence[float]], dtype: int,
                       stream: Optional[int], workspace: Optional[int] = None, workspace_bytes: int = 0) -> None:
    """Enqueue attention on raw q (rotated in the kernel's prologue with cs_table) and rotated k."""
    _check(load_library().sa_attn_fwd_rope_q(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k_rot), ctypes.c_void_p(cs_table),
        ctypes.c_void_p(v), ctypes.c_void_p(out), int(B), int(H), int(L), int(d), int(window), _lam(lam),
        int(dtype), ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes), ctypes.c_void_p(stream)))


def sa_rope_attn(handle: int, q: int, k: int, v: int, positions: Optional[int], out: int,
                 B: int, H: int, L: int, d: int, window: int, lam: Optional[Sequence[float]],
                 dtype: int, workspace: Optional[int], workspace_bytes: int,
                 stream: Optional[int]) -> None:
    """Enqueue RoPE + attention.  Pointer arguments are device addresses (ints) or None."""
    lam_arr = _lam(lam)
    _check(load_library().sa_rope_attn(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
        ctypes.c_void_p(positions), ctypes.c_void_p(out), int(B), int(H), int(L), int(d),
        int(window), lam_arr, int(dtype), ctypes.c_void_p(workspace), int(workspace_bytes),
        ctypes.c_void_p(stream)))


def _lam(lam):
    if lam is None:
        return None
    vals = [float(x) for x in lam]
    return (ctypes.c_float * len(vals))(*vals)


def sa_rope_qk(handle: int, q: int, k: int, positions: Optional[int], q_rot: int, k_rot: int,
               B: int, H: int, L: int, d: int, nmaps: int, dtype: int, stream: Optional[int]) -> None:
    """Enqueue the RoPE stage alone (q_rot/k_rot get the rotated, cast-back q/k)."""
    _check(load_library().sa_rope_qk(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(positions),
        ctypes.c_void_p(q_rot), ctypes.c_void_p(k_rot), int(B), int(H), int(L), int(d), int(nmaps),
        int(dtype), ctypes.c_void_p(stream)))


def sa_rope_attn_host_workspace_size(B: int, H: int, L: int, d: int, differential: bool) -> int:
    return int(load_library().sa_rope_attn_host_workspace_size(int(B), int(H), int(L), int(d), int(bool(differential))))


def sa_rope_attn_host(handle: int, q: int, k: int, v: int, positions: Optional[int], out: int,
                      B: int, H: int, L: int, d: int, window: int, lam: Optional[Sequence[float]],
                      dtype: int, workspace: Optional[int], workspace_bytes: int,
                      stream: Optional[int]) -> None:
    """Enqueue RoPE + attention on HOST q, k, v, out (ints: host addresses; page-locked memory
    overlaps the copies); positions and workspace are device addresses."""
    _check(load_library().sa_rope_attn_host(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
        ctypes.c_void_p(positions), ctypes.c_void_p(out), int(B), int(H), int(L), int(d),
        int(window), _lam(lam), int(dtype), ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes),
        ctypes.c_void_p(stream)))


def _gamma(g):
    if g is None:
        return None
    vals = [float(x) for x in g]
    return (ctypes.c_float * len(vals))(*vals)


def sa_rope_attn_qknorm(handle: int, q: int, k: int, v: int, positions: Optional[int],
                        gamma_q: Optional[Sequence[float]], gamma_k: Optional[Sequence[float]],
                        eps: float, out: int, B: int, H: int, L: int, d: int, window: int,
                        lam: Optional[Sequence[float]], dtype: int, workspace: Optional[int],
                        workspace_bytes: int, stream: Optional[int]) -> None:
    """Enqueue QK-RMSNorm (FP32, gamma per tensor, eps) + RoPE + attention; gammas are host lists."""
    for g in (gamma_q, gamma_k):
        if g is not None and len(g) != d:
            raise ValueError("gamma must have d entries")
    _check(load_library().sa_rope_attn_qknorm(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
        ctypes.c_void_p(positions), _gamma(gamma_q), _gamma(gamma_k), ctypes.c_float(eps),
        ctypes.c_void_p(out), int(B), int(H), int(L), int(d), int(window), _lam(lam), int(dtype),
        ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes), ctypes.c_void_p(stream)))


def sa_qknorm_rope_qk(handle: int, q: int, k: int, positions: Optional[int],
                      gamma_q: Optional[Sequence[float]], gamma_k: Optional[Sequence[float]], eps: float,
                      q_rot: int, k_rot: int, B: int, H: int, L: int, d: int, nmaps: int, dtype: int,
                      stream: Optional[int]) -> None:
    """Enqueue the QK-RMSNorm + RoPE stage alone (q_rot/k_rot: normalised, rotated, cast-back)."""
    for g in (gamma_q, gamma_k):
        if g is not None and len(g) != d:
            raise ValueError("gamma must have d entries")
    _check(load_library().sa_qknorm_rope_qk(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(positions),
        _gamma(gamma_q), _gamma(gamma_k), ctypes.c_float(eps), ctypes.c_void_p(q_rot),
        ctypes.c_void_p(k_rot), int(B), int(H), int(L), int(d), int(nmaps), int(dtype),
        ctypes.c_void_p(stream)))


def sa_attn_fwd(handle: int, q_rot: int, k_rot: int, v: int, out: int, B: int, H: int, L: int,
                d: int, window: int, lam: Optional[Sequence[float]], dtype: int,
                stream: Optional[int], workspace: Optional[int] = None, workspace_bytes: int = 0) -> None:
    """Enqueue the attention stage alone on already-rotated q/k (workspace: optional split region)."""
    _check(load_library().sa_attn_fwd(
        ctypes.c_void_p(handle), ctypes.c_void_p(q_rot), ctypes.c_void_p(k_rot), ctypes.c_void_p(v),
        ctypes.c_void_p(out), int(B), int(H), int(L), int(d), int(window), _lam(lam), int(dtype),
        ctypes.c_void_p(workspace), ctypes.c_size_t(workspace_bytes), ctypes.c_void_p(stream)))


def sa_rope_attn_noalloc(handle: int, q: int, k: int, v: int, positions: Optional[int], out: int,
                         B: int, H: int, L: int, d: int, window: int,
                         lam: Optional[Sequence[float]], dtype: int, stream: Optional[int]) -> None:
    """sa_rope_attn without a workspace: for callers that cannot allocate device memory.
    The library's built-in scratch (SA_NOALLOC_SCRATCH_BYTES) is used and shared by all calls."""
    _check(load_library().sa_rope_attn_noalloc(
        ctypes.c_void_p(handle), ctypes.c_void_p(q), ctypes.c_void_p(k), ctypes.c_void_p(v),
        ctypes.c_void_p(positions), ctypes.c_void_p(out), int(B), int(H), int(L), int(d),
        int(window), _lam(lam), int(dtype), ctypes.c_void_p(stream)))


SA_NOALLOC_SCRATCH_BYTES = 64 << 20


def sa_attn_set_timeout(handle: int, timeout_ns: int) -> None:
    """Limit of every pipeline wait in the attention kernel (default 1 s)."""
    _check(load_library().sa_attn_set_timeout(ctypes.c_void_p(handle), int(timeout_ns)))


def sa_attn_check(handle: int) -> None:
    _check(load_library().sa_attn_check(ctypes.c_void_p(handle)))


class RopeAttention:
    """Convenience wrapper over the C ABI for torch CUDA tensors.

    ``attn(q, k, v, positions=None, window=-1, lam=None)`` returns ``out``.
    Standard attention: q, k, v ``[B, H, L, 64]``.  Differential (``lam`` given,
    one float per head or a scalar): q, k ``[B, H, 2, L, 64]``, v ``[B, H, L, 128]``.
    fp16 / bf16 tensors, or float32 for differential attention (TF32 products).
    Output and workspace are allocated with torch on the current stream.
    """

    def __init__(self, device: int = 0, rope_base: float = 10000.0):
        self.device = int(device)
        self.handle = sa_attn_create(self.device, rope_base)
        self._ws = None

    def close(self) -> None:
        if self.handle:
            sa_attn_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def workspace(self, B: int, H: int, L: int, differential: bool, dtype: int = SA_FP16):
        import torch

        need = sa_rope_attn_workspace_bytes(B, H, L, 64, differential, dtype)
        if self._ws is None or self._ws.numel() < need:
            self._ws = torch.empty(need, dtype=torch.uint8, device=f"cuda:{self.device}")
        return self._ws

    def __call__(self, q, k, v, positions=None, window: int = -1, lam=None, out=None, stream=None):
        import torch

        dtype = {torch.float16: SA_FP16, torch.bfloat16: SA_BF16, torch.float32: SA_FP32}.get(q.dtype)
        if dtype is None:
            raise SaAttnError(1, f"unsupported dtype {q.dtype}")
        for name, t in (("q", q), ("k", k), ("v", v), ("positions", positions), ("out", out)):
            if t is not None and (not t.is_cuda or not t.is_contiguous()):
                raise SaAttnError(1, f"{name} must be a contiguous CUDA tensor")
        diff = lam is not None
        if diff:
            B, H, _, L, d = q.shape
        else:
            B, H, L, d = q.shape
        dv = v.shape[-1]
        if diff and not hasattr(lam, "__len__"):
            lam = [float(lam)] * H
        if out is None:
            out = torch.empty((B, H, L, dv), dtype=q.dtype, device=q.device)
        ws = self.workspace(B, H, L, diff, dtype)
        s = torch.cuda.current_stream(q.device).cuda_stream if stream is None else stream
        sa_rope_attn(self.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                     None if positions is None else positions.data_ptr(), out.data_ptr(),
                     B, H, L, d, window, lam, dtype, ws.data_ptr(), ws.numel(), s)
        return out

    def check(self) -> None:
        sa_attn_check(self.handle)
