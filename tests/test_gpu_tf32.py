"""GPU parity of the FP32-input form (TF32 products) against the FP64 oracle.

SAME-L's attention projections are FP32 and its shipped kernel runs both attention products as
TF32 MMAs with FP32 accumulation (HF discussion #6 "sm_120 SAME-L", "How the kernels differ"),
on the differential attention with the symmetric window of the same page ("Three gotchas").
Everything goes through the C ABI with dtype SA_FP32.  The bar is the one of the 16-bit paths:
max-abs error <= 4e-3 and per-row cosine >= 0.9999 against the unrounded FP64 oracle (TF32
keeps 10 explicit mantissa bits, as fp16 does).
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


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    a = sa.RopeAttention(0)
    yield a
    a.check()
    a.close()


def f32(bits):
    return torch.from_numpy(synth.decode(bits, "fp32")).cuda()


def run(attn, x, positions=None, window=None):
    w = x["workload"]
    pos = None if positions is None else torch.from_numpy(positions.astype(np.int32)).cuda()
    out = attn(f32(x["q"]), f32(x["k"]), f32(x["v"]), positions=pos,
               window=w.window if window is None else window, lam=[float(t) for t in x["lam"]])
    torch.cuda.synchronize()
    return out.cpu().numpy().astype(np.float64)


def compare(got, ref, tag=""):
    g = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    assert np.all(np.isfinite(g)), f"{tag}: non-finite output"
    err = np.abs(g - r).max()
    cos = (g * r).sum(1) / np.maximum(np.linalg.norm(g, axis=1) * np.linalg.norm(r, axis=1), 1e-300)
    assert err <= TOL_ABS, f"{tag}: max-abs {err:.3e}"
    assert cos.min() >= TOL_COS, f"{tag}: row {int(np.argmin(cos))} cosine {cos.min():.6f}"
    return err, cos.min()


def wl(name, L, window=-1, B=1, H=2, seed=0):
    return synth.Workload(name, B=B, H=H, L=L, nmaps=2, dv=128, dtype="fp32", window=window, seed=seed,
                          lam=("uniform", 0.2, 0.8))


def test_rope_prepass_matches_oracle(attn):
    # sa_rope_qk in FP32: q', k' = RoPE in FP32 rounded to TF32, against the FP64 rotation.
    # Bound per value: the FP32 angle theta = fl(fl(p) * fl(inv_freq)) is off by at most
    # |theta| * 2^-22, which moves the rotated pair by that much times its norm; the TF32
    # rounding adds half a unit of the 11-bit significand (2^-11 relative); FMA roundings 2^-22.
    w = wl("rope32", L=300, H=3, seed=70)
    x = synth.make_inputs(w)
    pos = (np.arange(w.L) * 27 + 5).astype(np.int32)
    q, k = f32(x["q"]), f32(x["k"])
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    s = torch.cuda.current_stream().cuda_stream
    sa.sa_rope_qk(attn.handle, q.data_ptr(), k.data_ptr(), torch.from_numpy(pos).cuda().data_ptr(),
                  qr.data_ptr(), kr.data_ptr(), w.B, w.H, w.L, 64, 2, sa.SA_FP32, s)
    torch.cuda.synchronize()
    i = np.arange(32)
    inv_freq = 10000.0 ** (-2.0 * i / 64)
    theta = pos[:, None].astype(np.float64) * inv_freq[None, :]          # [L, 32]
    dtheta = np.abs(theta) * 2.0 ** -22 + 1e-12
    for src, got in ((x["q"], qr), (x["k"], kr)):
        xin = synth.decode(src, "fp32").astype(np.float64).reshape(-1, w.L, 64)
        ref = oracle.rope(xin.reshape(-1, 64), np.tile(pos, xin.shape[0])).reshape(xin.shape)
        g = got.cpu().numpy().astype(np.float64).reshape(xin.shape)
        r_pair = np.sqrt(xin[..., :32] ** 2 + xin[..., 32:] ** 2)          # pair norms
        bound_pair = dtheta[None] * r_pair
        bound = np.concatenate([bound_pair, bound_pair], axis=-1) + 2.0 ** -11 * np.abs(ref) + \
            2.0 ** -22 * np.concatenate([r_pair, r_pair], axis=-1)
        assert np.all(np.abs(g - ref) <= bound * 1.01 + 1e-30)
        # every value is a TF32 number: its low 13 mantissa bits are zero
        bits = got.cpu().numpy().view(np.uint32)
        assert np.all((bits & 0x1FFF) == 0)


@pytest.mark.parametrize("L", [1, 2, 63, 64, 65, 127, 128, 129, 200, 333, 513])
def test_length_sweep_full_attention(attn, L):
    x = synth.make_inputs(wl("len32", L=L, seed=80 + L))
    compare(run(attn, x), oracle.rope_attn_workload(x), f"L={L}")


@pytest.mark.parametrize("win", [0, 1, 17, 63, 64, 65, 129, 256, 299, 300, 1000])
def test_window_sweep(attn, win):
    x = synth.make_inputs(wl("win32", L=301, window=win, seed=90))
    compare(run(attn, x), oracle.rope_attn_workload(x), f"window={win}")


def test_batches_heads_and_positions(attn):
    w = wl("bhp32", L=190, window=40, B=2, H=5, seed=100)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(101)
    pos = (rng.permutation(w.L) * 7 + 3000).astype(np.int32)
    x["positions"] = pos
    compare(run(attn, x, positions=pos), oracle.rope_attn_workload(x), "batches/heads/positions")


def test_full_size_workload(attn):
    w = synth.WORKLOADS["swa_diff_l8192_fp32"]
    x = synth.make_inputs(w)
    got = run(attn, x)
    rng = np.random.default_rng(110)
    fixed = [0, 1, 127, 128, 255, 256, 4095, 4096, 8064, 8191]
    rows = np.array([bh * w.L + i for bh in range(w.B * w.H)
                     for i in sorted(set(fixed) | set(rng.integers(0, w.L, 6).tolist()))], dtype=np.int64)
    compare(got.reshape(-1, w.dv)[rows], oracle.rope_attn_workload(x, rows=rows), w.name)
    # every row: out is a difference of two convex combinations of v rows
    g = got.reshape(w.B, w.H, w.L, w.dv)
    vmax = np.abs(synth.decode(x["v"], "fp32")).max(axis=2, keepdims=True)
    bound = (1 + x["lam"].astype(np.float64))[None, :, None, None] * vmax * (1 + 1e-2) + 1e-3
    assert np.all(np.abs(g) <= bound)


def test_two_stages_equal_public_call_and_reproducible(attn):
    # sa_rope_qk then sa_attn_fwd has the bits of sa_rope_attn; repeated calls agree bit for bit
    w = wl("stages32", L=701, window=100, H=3, seed=120)
    x = synth.make_inputs(w)
    q, k, v = f32(x["q"]), f32(x["k"]), f32(x["v"])
    lam = [float(t) for t in x["lam"]]
    s = torch.cuda.current_stream().cuda_stream
    out1 = attn(q, k, v, window=w.window, lam=lam)
    out2 = attn(q, k, v, window=w.window, lam=lam)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    out3, out4 = torch.empty_like(out1), torch.empty_like(out1)
    # sa_rope_qk then sa_attn_fwd (which transposes v into its workspace first)
    sa.sa_rope_qk(attn.handle, q.data_ptr(), k.data_ptr(), None, qr.data_ptr(), kr.data_ptr(),
                  w.B, w.H, w.L, 64, 2, sa.SA_FP32, s)
    nws = sa.sa_attn_fwd_workspace_bytes(w.B, w.H, w.L, 64, True, sa.SA_FP32)
    ws = torch.empty(nws, dtype=torch.uint8, device="cuda")
    sa.sa_attn_fwd(attn.handle, qr.data_ptr(), kr.data_ptr(), v.data_ptr(), out3.data_ptr(), w.B, w.H, w.L, 64,
                   w.window, lam, sa.SA_FP32, s, ws.data_ptr(), nws)
    # the FP32 stage entry points: pre-pass (q', k', v^T), then the TF32 kernel
    L4 = (w.L + 3) // 4 * 4
    vt = torch.empty((w.B * w.H, 128, L4), dtype=torch.float32, device="cuda")
    qr2, kr2 = torch.empty_like(q), torch.empty_like(k)
    sa.sa_rope_qkv_f32(attn.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, qr2.data_ptr(), kr2.data_ptr(),
                       vt.data_ptr(), w.B, w.H, w.L, 64, s)
    sa.sa_attn_fwd_f32(attn.handle, qr2.data_ptr(), kr2.data_ptr(), vt.data_ptr(), out4.data_ptr(), w.B, w.H, w.L,
                       64, w.window, lam, s)
    torch.cuda.synchronize()
    assert torch.equal(out1.view(torch.int32), out2.view(torch.int32))
    assert torch.equal(out1.view(torch.int32), out3.view(torch.int32))
    assert torch.equal(out1.view(torch.int32), out4.view(torch.int32))
    # v^T is the TF32-rounded transpose of v, zero past L
    vt_ref = torch.from_numpy(synth.decode(x["v"], "fp32")).cuda().reshape(w.B * w.H, w.L, 128).transpose(1, 2)
    assert torch.all(vt[:, :, w.L:] == 0)
    assert torch.all((vt[:, :, :w.L] - vt_ref).abs() <= vt_ref.abs() * 2.0 ** -11)
    assert torch.all((vt.view(torch.int32) & 0x1FFF) == 0)


def test_output_guard_bands_untouched(attn):
    w = wl("guard32", L=77, window=9, seed=130)
    x = synth.make_inputs(w)
    n = w.B * w.H * w.L * w.dv
    buf = torch.full((n + 2 * 1024,), 7.5, dtype=torch.float32, device="cuda")
    out = buf[1024:1024 + n].view(w.B, w.H, w.L, w.dv)
    attn(f32(x["q"]), f32(x["k"]), f32(x["v"]), window=w.window, lam=[float(t) for t in x["lam"]], out=out)
    torch.cuda.synchronize()
    assert torch.all(buf[:1024] == 7.5) and torch.all(buf[1024 + n:] == 7.5)
    compare(out.cpu().numpy(), oracle.rope_attn_workload(x), "guard")


def test_noalloc_fp32_matches_workspace_call(attn):
    w = wl("noalloc32", L=400, window=50, H=3, seed=140)
    x = synth.make_inputs(w)
    q, k, v = f32(x["q"]), f32(x["k"]), f32(x["v"])
    lam = [float(t) for t in x["lam"]]
    ref = attn(q, k, v, window=w.window, lam=lam)
    out = torch.full_like(ref, 3.0)
    sa.sa_rope_attn_noalloc(attn.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(),
                            w.B, w.H, w.L, 64, w.window, lam, sa.SA_FP32, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int32), ref.view(torch.int32))


def test_fp32_host_checks(attn):
    s = torch.cuda.current_stream().cuda_stream
    t = torch.zeros(4096, dtype=torch.float32, device="cuda")
    p = t.data_ptr()
    ws = sa.sa_rope_attn_workspace_bytes(1, 1, 8, 64, True, sa.SA_FP32)
    a256 = lambda n: (n + 255) // 256 * 256
    assert ws == 2 * a256(1 * 1 * 2 * 8 * 64 * 4) + a256(1 * 1 * 128 * 8 * 4)
    assert sa.sa_attn_fwd_workspace_bytes(1, 1, 9, 64, True, sa.SA_FP32) == a256(128 * 12 * 4)
    assert sa.sa_rope_attn_workspace_bytes(1, 1, 8, 64, False, sa.SA_FP32) == 0
    with pytest.raises(sa.SaAttnError) as e:    # standard attention has no FP32 form
        sa.sa_rope_attn(attn.handle, p, p, p, None, p, 1, 1, 8, 64, -1, None, sa.SA_FP32, p, 1 << 16, s)
    assert e.value.status == 2
    with pytest.raises(sa.SaAttnError) as e:    # workspace too small
        sa.sa_rope_attn(attn.handle, p, p, p, None, p, 1, 1, 8, 64, -1, [0.5], sa.SA_FP32, p, ws - 256, s)
    assert e.value.status == 6
    with pytest.raises(sa.SaAttnError) as e:    # the QK-RMSNorm form is 16-bit only
        sa.sa_rope_attn_qknorm(attn.handle, p, p, p, None, None, None, 1e-6, p, 1, 1, 8, 64, -1, [0.5],
                               sa.SA_FP32, p, 1 << 16, s)
    assert e.value.status == 2
    with pytest.raises(sa.SaAttnError) as e:    # the Q-prologue stage is 16-bit only
        sa.sa_rope_k(attn.handle, p, None, p, p, 1, 1, 8, 64, 2, sa.SA_FP32, s)
    assert e.value.status == 2
    torch.cuda.synchronize()
    assert torch.all(t == 0)
