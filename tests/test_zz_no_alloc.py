"""sa_rope_attn_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (an engine plugin that only receives tensor pointers and a stream,
a real-time audio thread that must not block in an allocator) still pass
inputs and outputs, but no workspace: the library's built-in scratch array is
used instead.  This test calls it through the C ABI several times in a row, on
different shapes, and checks each result against sa_rope_attn with a caller
workspace and against the FP64 oracle, within the parity tolerance of the other
GPU tests.  The shapes include the largest the built-in scratch accepts (the
SWA differential workload, B*H*maps*L = 262,144 rows of 64 values) and a call
with explicit positions; one row more is refused before anything runs.

This file is collected last on purpose and runs alone or after the other tests.
"""

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_rope_gb300 as sa
import oracle
import synth

pytestmark = pytest.mark.gpu

TOL_ABS = 4e-3
TOL_COS = 0.9999
TDT = {"fp16": torch.float16, "bf16": torch.bfloat16}


def _dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(TDT[dtype])


def _rows(a, dv):
    return np.asarray(a, dtype=np.float64).reshape(-1, dv)


def _close(a, b):
    a, b = _rows(a, b.shape[-1]), _rows(b, b.shape[-1])
    assert np.all(np.isfinite(a))
    err = np.abs(a - b).max()
    assert err <= TOL_ABS, f"max-abs {err:.3e}"
    cos = (a * b).sum(1) / np.maximum(np.linalg.norm(a, axis=1) * np.linalg.norm(b, axis=1), 1e-300)
    assert cos.min() >= TOL_COS, f"min row cosine {cos.min():.6f}"


def _scratch_need(B, H, L, maps):
    """Bytes of built-in scratch a shape takes: q' and k', each rounded up to 256 bytes."""
    a256 = lambda n: (n + 255) // 256 * 256
    return 2 * a256(B * H * maps * L * 64 * 2)


def _run_both(h, stream, w, x, positions=None):
    """sa_rope_attn (caller workspace) and sa_rope_attn_noalloc on the same inputs."""
    q, k, v = _dev(x["q"], w.dtype), _dev(x["k"], w.dtype), _dev(x["v"], w.dtype)
    pos = None if positions is None else torch.from_numpy(positions.astype(np.int32)).cuda()
    pos_ptr = None if pos is None else pos.data_ptr()
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    dtype = sa.SA_FP16 if w.dtype == "fp16" else sa.SA_BF16
    out_ref = torch.empty((w.B, w.H, w.L, w.dv), dtype=TDT[w.dtype], device="cuda")
    out_na = torch.full_like(out_ref, 3.0)
    nbytes = sa.sa_rope_attn_workspace_size(w.B, w.H, w.L, w.d, w.differential)
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), pos_ptr, out_ref.data_ptr(),
                    w.B, w.H, w.L, w.d, w.window, lam, dtype, ws.data_ptr(), nbytes, stream)
    sa.sa_rope_attn_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), pos_ptr, out_na.data_ptr(),
                            w.B, w.H, w.L, w.d, w.window, lam, dtype, stream)
    torch.cuda.synchronize()
    sa.sa_attn_check(h)
    to_np = lambda t: t.float().cpu().numpy().astype(np.float64)
    return to_np(out_na), to_np(out_ref)


def test_noalloc_entry_point_matches_workspace_entry_point_and_oracle():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    h = sa.sa_attn_create(0)
    stream = torch.cuda.current_stream().cuda_stream
    rng = np.random.default_rng(23)
    try:
        # several calls in a row on different shapes and dtypes, the last one with explicit
        # positions; every output against the workspace entry point and the FP64 oracle
        cases = [
            (synth.Workload("noalloc_std", B=1, H=3, L=777, seed=21), None),
            (synth.Workload("noalloc_diff", B=2, H=2, L=600, nmaps=2, dv=128, dtype="bf16", window=129,
                            seed=22, lam=("uniform", 0.2, 0.8)), None),
            (synth.Workload("noalloc_pos", B=1, H=2, L=333, seed=24), (rng.permutation(333) * 3 + 11)),
        ]
        for w, pos in cases:
            x = synth.make_inputs(w)
            if pos is not None:
                x["positions"] = pos.astype(np.int32)
            assert _scratch_need(w.B, w.H, w.L, w.nmaps) <= sa.SA_NOALLOC_SCRATCH_BYTES
            got, ref_ws = _run_both(h, stream, w, x, positions=x["positions"] if pos is not None else None)
            _close(got, ref_ws)
            _close(got, oracle.rope_attn_workload(x))

        # the largest shape the built-in scratch holds: the SWA differential workload (16 heads,
        # two maps, L = 8192, window 256), whose q' and k' fill the array exactly
        w = synth.WORKLOADS["swa_diff_l8192"]
        assert w.B * w.H * w.nmaps * w.L == 262144
        assert _scratch_need(w.B, w.H, w.L, w.nmaps) == sa.SA_NOALLOC_SCRATCH_BYTES
        x = synth.make_inputs(w)
        got, ref_ws = _run_both(h, stream, w, x)
        _close(got, ref_ws)
        fixed = [0, 1, 255, 256, 4095, 4096, 8190, 8191]
        rows = np.array([bh * w.L + i for bh in range(w.B * w.H)
                         for i in sorted(set(fixed) | set(rng.integers(0, w.L, 4).tolist()))], dtype=np.int64)
        _close(_rows(got, w.dv)[rows], oracle.rope_attn_workload(x, rows=rows))

        # one row more than the array holds is refused up front and nothing is written
        w = cases[0][0]
        x = synth.make_inputs(w)
        q, k, v = _dev(x["q"], w.dtype), _dev(x["k"], w.dtype), _dev(x["v"], w.dtype)
        out = torch.full((1, 3, 777, 64), 5.0, dtype=torch.float16, device="cuda")
        big_L = 262145
        assert _scratch_need(1, 1, big_L, 1) > sa.SA_NOALLOC_SCRATCH_BYTES
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_rope_attn_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(),
                                    1, 1, big_L, 64, -1, None, sa.SA_FP16, stream)
        assert e.value.status == 6
        assert "scratch" in sa.sa_last_error()
        # an oversized call with a bad head dim reports the head dim, as sa_rope_attn would
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_rope_attn_noalloc(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(),
                                    1, 1, big_L, 128, -1, None, sa.SA_FP16, stream)
        assert e.value.status == 2   # SA_ERR_UNSUPPORTED
        torch.cuda.synchronize()
        assert torch.all(out == 5.0)
    finally:
        sa.sa_attn_destroy(h)
