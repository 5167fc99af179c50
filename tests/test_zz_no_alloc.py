"""sa_rope_attn_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (an engine plugin that only receives tensor pointers and a stream,
a real-time audio thread that must not block in an allocator) still pass
inputs and outputs, but no workspace: the library's built-in scratch array is
used instead.  This test calls it through the C ABI twice in a row, on two
different shapes, and checks each result against sa_rope_attn with a caller
workspace, within the parity tolerance of the other GPU tests.  It also checks
that a shape too large for the built-in scratch is refused before anything runs.

This file is collected last on purpose and runs alone or after the other tests.
"""

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_rope_gb300 as sa
import synth

pytestmark = pytest.mark.gpu

TOL_ABS = 4e-3
TOL_COS = 0.9999
TDT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(TDT[dtype])


def _close(a, b):
    a = a.float().cpu().numpy().astype(np.float64).reshape(-1, a.shape[-1])
    b = b.float().cpu().numpy().astype(np.float64).reshape(-1, b.shape[-1])
    assert np.all(np.isfinite(a))
    assert np.abs(a - b).max() <= TOL_ABS
    cos = (a * b).sum(1) / np.maximum(np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1), 1e-300)
    assert cos.min() >= TOL_COS


def test_noalloc_entry_point_matches_workspace_entry_point():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    h = sa.sa_attn_create(0)
    stream = torch.cuda.current_stream().cuda_stream
    cases = [
        synth.Workload("noalloc_std", B=1, H=3, L=777, seed=21),
        synth.Workload("noalloc_diff", B=2, H=2, L=600, nmaps=2, dv=128, dtype="bf16", window=129,
                       seed=22, lam=("uniform", 0.2, 0.8)),
    ]
    try:
        for w in cases:   # two calls in a row, different shapes and dtypes
            x = synth.make_inputs(w)
            q, k, v = _dev(x["q"], w.dtype), _dev(x["k"], w.dtype), _dev(x["v"], w.dtype)
            lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
            dtype = sa.SA_FP16 if w.dtype == "fp16" else sa.SA_BF16
            out_ref = torch.empty((w.B, w.H, w.L, w.dv), dtype=TDT[w.dtype], device="cuda")
            out_na = torch.full_like(out_ref, 3.0)
            nbytes = sa.sa_rope_attn_workspace_size(w.B, w.H, w.L, w.d, w.differential)
            assert nbytes <= sa.SA_NOALLOC_SCRATCH_BYTES
            ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
            sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out_ref.data_ptr(),
                            w.B, w.H, w.L, w.d, w.window, lam, dtype, ws.data_ptr(), nbytes, stream)
            sa.sa_rope_attn_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None,
                                    out_na.data_ptr(), w.B, w.H, w.L, w.d, w.window, lam, dtype, stream)
            torch.cuda.synchronize()
            sa.sa_attn_check(h)
            _close(out_na, out_ref)

        # a shape whose scratch exceeds the built-in array is refused up front
        w = cases[0]
        x = synth.make_inputs(w)
        q, k, v = _dev(x["q"], w.dtype), _dev(x["k"], w.dtype), _dev(x["v"], w.dtype)
        out = torch.full((1, 3, 777, 64), 5.0, dtype=torch.float16, device="cuda")
        big_L = 1 << 20
        assert sa.sa_rope_attn_workspace_size(1, 3, big_L, 64, False) > sa.SA_NOALLOC_SCRATCH_BYTES
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_rope_attn_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(),
                                    1, 3, big_L, 64, -1, None, sa.SA_FP16, stream)
        assert e.value.status == 6
        assert "scratch" in sa.sa_last_error()
        torch.cuda.synchronize()
        assert torch.all(out == 5.0)
    finally:
        sa.sa_attn_destroy(h)
