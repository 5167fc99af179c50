"""Failure detection on the GPU without a GPU fault.

Every wait inside the attention kernel is bounded.  Shrinking the bound to
500 ns (sa_attn_set_timeout) makes real pipeline waits run out: the kernel must
give up cleanly, report SA_ERR_DEVICE_TIMEOUT through sa_attn_check, and leave
the context usable -- the next call with the default bound is checked against
the FP64 oracle.  No trap, no bad address, no endless loop is involved.
"""

import numpy as np
import pytest
import torch

import diffusion_transformer_attention_rope_gb300 as sa
import oracle
import synth

pytestmark = pytest.mark.gpu

TDT = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}
SA_DT = {"fp16": sa.SA_FP16, "bf16": sa.SA_BF16, "fp32": sa.SA_FP32}


def _dev(bits, dtype):
    raw = np.ascontiguousarray(bits).view(np.int32 if dtype == "fp32" else np.int16)
    return torch.from_numpy(raw).cuda().view(TDT[dtype])


def _run(h, x, stream):
    w = x["workload"]
    q, k, v = _dev(x["q"], w.dtype), _dev(x["k"], w.dtype), _dev(x["v"], w.dtype)
    out = torch.zeros((w.B, w.H, w.L, w.dv), dtype=TDT[w.dtype], device="cuda")
    nbytes = sa.sa_rope_attn_workspace_bytes(w.B, w.H, w.L, w.d, w.differential, SA_DT[w.dtype])
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(), w.B, w.H, w.L,
                    w.d, w.window, lam, SA_DT[w.dtype], ws.data_ptr(), nbytes, stream)
    torch.cuda.synchronize()
    return out


# one shape per attention kernel: the general kernel (standard and differential), the
# narrow-window kernel (differential, window 17: persistent CTAs, output warps) and the TF32
# kernel (FP32 inputs)
@pytest.mark.parametrize("variant", ["standard", "differential", "narrow_window", "fp32"])
def test_pipeline_timeout_is_reported_and_recoverable(variant):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    if variant == "standard":
        w = synth.Workload("fail_std", B=1, H=8, L=2048, seed=41)
    elif variant == "differential":
        w = synth.Workload("fail_diff", B=1, H=4, L=2048, nmaps=2, dv=128, dtype="bf16", seed=42,
                           lam=("uniform", 0.2, 0.8))
    elif variant == "narrow_window":
        w = synth.Workload("fail_swa", B=1, H=8, L=4096, nmaps=2, dv=128, dtype="bf16", window=17, seed=44,
                           lam=("uniform", 0.2, 0.8))
    else:
        w = synth.Workload("fail_f32", B=1, H=4, L=2048, nmaps=2, dv=128, dtype="fp32", window=256, seed=45,
                           lam=("uniform", 0.2, 0.8))
    x = synth.make_inputs(w)
    stream = torch.cuda.current_stream().cuda_stream
    h = sa.sa_attn_create(0)
    try:
        sa.sa_attn_set_timeout(h, 500)          # far below a single tile's latency
        _run(h, x, stream)
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_attn_check(h)
        assert e.value.status == 4
        assert "pipeline wait" in sa.sa_last_error()

        sa.sa_attn_set_timeout(h, 1_000_000_000)
        sa.sa_attn_check(h)                     # the word was cleared by the previous check
        tiny = synth.make_inputs(synth.WORKLOADS["tiny"])
        got = _run(h, tiny, stream).float().cpu().numpy().astype(np.float64)
        sa.sa_attn_check(h)
        ref = oracle.rope_attn_workload(tiny)
        assert np.abs(got - ref).max() <= 4e-3
    finally:
        sa.sa_attn_destroy(h)


def test_set_timeout_rejects_bad_values():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    h = sa.sa_attn_create(0)
    try:
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_attn_set_timeout(h, 10)
        assert e.value.status == 1
    finally:
        sa.sa_attn_destroy(h)


def test_timeout_through_the_host_entry_is_reported():
    # the host-buffer entry runs its chunks on the handle's internal streams: a device-side
    # timeout there reaches the same error word, and the handle stays usable
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = synth.Workload("fail_host", B=1, H=12, L=8192, window=129, seed=43)   # 3 chunks of 4 planes
    x = synth.make_inputs(w)
    host = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).pin_memory()
    qh, kh, vh = host(x["q"]), host(x["k"]), host(x["v"])
    oh = torch.zeros((w.B, w.H, w.L, w.dv), dtype=torch.float16).pin_memory()
    n = sa.sa_rope_attn_host_workspace_size(w.B, w.H, w.L, w.d, False)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream().cuda_stream
    h = sa.sa_attn_create(0)

    def run():
        sa.sa_rope_attn_host(h, qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), None, oh.data_ptr(), w.B, w.H, w.L,
                             w.d, w.window, None, sa.SA_FP16, ws.data_ptr(), n, stream)
        torch.cuda.synchronize()

    try:
        sa.sa_attn_set_timeout(h, 500)
        run()
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_attn_check(h)
        assert e.value.status == 4
        sa.sa_attn_set_timeout(h, 1_000_000_000)
        run()
        sa.sa_attn_check(h)
        rows = np.arange(0, w.B * w.H * w.L, 997)
        ref = oracle.rope_attn_workload(x, rows=rows)
        got = oh.float().numpy().astype(np.float64).reshape(-1, w.dv)[rows]
        assert np.abs(got - ref).max() <= 4e-3
    finally:
        sa.sa_attn_destroy(h)
