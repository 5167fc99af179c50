"""Pins of the FP64 oracle against things other than itself.

Each test ties one piece of the oracle to a library routine (numpy's fp16
cast, torch's float64 scaled_dot_product_attention), to a closed form, to an
invariant the pages fix, to brute force, or to a number printed on the pages.
The comment on each test names the plausible mistake it would catch.
"""

import math

import numpy as np
import pytest
import torch

import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


# ----------------------------------------------------------------------------- helpers

def _sdpa64(q, k, v, mask=None):
    """torch float64 SDPA, [..., L, d] arrays (library routine, default scale 1/sqrt(d))."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)) for a in (q, k, v))
    m = None if mask is None else torch.from_numpy(mask)
    return torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=m).numpy()


def _rand_bits(rng, shape, dtype, scale=1.0):
    return synth.encode((rng.standard_normal(shape) * scale).astype(np.float32), dtype)


def _decode64(bits, dtype):
    return synth.decode(bits, dtype).astype(np.float64)


def _window_mask(L, w):
    i = np.arange(L)[:, None]
    j = np.arange(L)[None, :]
    return np.abs(i - j) <= w


# ----------------------------------------------------------------------------- bit decoding

def test_fp16_decode_exhaustive(oracle_mod):
    # catches: wrong exponent bias, subnormal scale, sign handling
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.bits_to_double(bits, "fp16")
    ref = bits.view(np.float16).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def test_bf16_decode_exhaustive(oracle_mod):
    # bf16 is the upper half of an IEEE float32 (library decode via a float32 view)
    bits = np.arange(65536, dtype=np.uint16)
    got = oracle_mod.bits_to_double(bits, "bf16")
    ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


# ----------------------------------------------------------------------------- rounding

def _fp16_test_values(rng):
    halves = np.arange(0, 0x7C00, dtype=np.uint16).view(np.float16).astype(np.float64)
    mids = (halves[:-1] + halves[1:]) / 2.0            # exact ties
    off = mids * (1 + 2.0 ** -40)                      # just above ties (needs a direct rounding)
    rnd = np.concatenate([rng.standard_normal(20000) * s for s in (1e-6, 1e-3, 1.0, 300.0, 3e4)])
    edge = np.array([0.0, 65504.0, 65519.999, 65520.0, 7e4, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26])
    v = np.concatenate([mids, off, rnd, edge])
    return np.concatenate([v, -v])


def test_round_fp16_matches_numpy(oracle_mod):
    # numpy rounds double -> half directly, to nearest even.  Catches: ties
    # rounded away from zero, double rounding, wrong subnormal quantum, overflow.
    x = _fp16_test_values(np.random.default_rng(1))
    with np.errstate(over="ignore"):
        ref = x.astype(np.float16).astype(np.float64)
    got = oracle_mod.round_to(x, "fp16")
    np.testing.assert_array_equal(got, ref)


def test_round_bf16_brute_force(oracle_mod):
    # nearest bf16 value by exhaustive search over all finite bf16 values,
    # ties to the even mantissa.  Independent of the quantum arithmetic.
    rng = np.random.default_rng(2)
    finite = np.arange(0, 0x7F80, dtype=np.uint32)
    vals = (finite << 16).view(np.float32).astype(np.float64)      # sorted ascending
    mids = (vals[:-1] + vals[1:]) / 2.0
    x = np.concatenate([
        rng.choice(mids, 4000),                                      # exact ties
        rng.standard_normal(4000) * np.exp(rng.uniform(-80, 80, 4000)),
        np.array([4155.0, 4144.0, 4160.0, 1.0 + 2.0 ** -8 + 2.0 ** -40]),
    ])
    x = np.concatenate([x, -x])
    got = oracle_mod.round_to(x, "bf16")
    a = np.abs(x)
    hi = np.searchsorted(vals, a, side="left").clip(1, len(vals) - 1)
    lo = hi - 1
    dlo = a - vals[lo]
    dhi = vals[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (finite[hi] % 2 == 0))
    ref = np.where(pick_hi, vals[hi], vals[lo])
    ref = np.where(a == vals[hi], vals[hi], ref)
    np.testing.assert_array_equal(got, np.copysign(ref, x))


def test_round_bf16_matches_torch_on_float32_inputs(oracle_mod):
    # torch converts float32 -> bfloat16 with one RNE rounding (a library routine)
    rng = np.random.default_rng(3)
    x32 = (rng.standard_normal(50000) * np.exp(rng.uniform(-30, 30, 50000))).astype(np.float32)
    ref = torch.from_numpy(x32).to(torch.bfloat16).to(torch.float64).numpy()
    got = oracle_mod.round_to(x32.astype(np.float64), "bf16")
    np.testing.assert_array_equal(got, ref)


def test_bf16_spacing_from_the_pages(oracle_mod):
    # The sa3_trt README ("Retired: bf16") states that a RoPE angle of ~4155 rad
    # lies where bf16's spacing is 32 rad (> 2*pi).  Check the oracle's bf16
    # grid there: neighbouring representable values are 32 apart.
    grid = oracle_mod.round_to(np.arange(4096.0, 8192.0, 1.0), "bf16")
    steps = np.diff(np.unique(grid))
    assert np.all(steps == 32.0)
    assert oracle_mod.round_to(np.array([4155.0]), "bf16")[0] == 4160.0
    assert 32.0 > 2 * math.pi


# ----------------------------------------------------------------------------- RoPE

def test_rope_d2_is_rotation_by_p_radians(oracle_mod):
    # d = 2: the only frequency is base^0 = 1, so RoPE rotates (x0, x1) by p radians.
    # catches: wrong sign (rotation the other way), cos/sin swapped.
    p = np.array([0, 1, 2, 7, 100, 4091], dtype=np.int32)
    x = np.tile(np.array([[1.0, 0.0]]), (len(p), 1))
    y = oracle_mod.rope(x, p)
    np.testing.assert_allclose(y[:, 0], np.cos(p.astype(np.float64)), atol=1e-13)
    np.testing.assert_allclose(y[:, 1], np.sin(p.astype(np.float64)), atol=1e-13)
    x = np.tile(np.array([[0.0, 1.0]]), (len(p), 1))
    y = oracle_mod.rope(x, p)
    np.testing.assert_allclose(y[:, 0], -np.sin(p.astype(np.float64)), atol=1e-13)
    np.testing.assert_allclose(y[:, 1], np.cos(p.astype(np.float64)), atol=1e-13)


def test_rope_frequency_anchors_d64(oracle_mod):
    # At p = 1 the rotation angle of pair (i, i+32) is the frequency itself.
    # Anchors computable by hand for base 10000, d = 64: f_0 = 1, f_8 = 10000^-1/4 = 0.1,
    # f_16 = 10000^-1/2 = 0.01, f_24 = 0.001; and the frequencies form a geometric
    # series with ratio 10000^(-1/32).  catches: exponent -i/d instead of -2i/d,
    # interleaved pairs (i, i+1) instead of rotate-half (i, i+d/2).
    d = 64
    x = np.zeros((32, d))
    for i in range(32):
        x[i, i] = 1.0
    y = oracle_mod.rope(x, np.ones(32, dtype=np.int32))
    ang = np.array([math.atan2(y[i, i + 32], y[i, i]) for i in range(32)])
    np.testing.assert_allclose(ang[[0, 8, 16, 24]], [1.0, 0.1, 0.01, 0.001], rtol=1e-13)
    ratio = ang[1:] / ang[:-1]
    np.testing.assert_allclose(ratio, 10000.0 ** (-1.0 / 32.0), rtol=1e-12)
    # energy stays inside the pair: no leakage into other coordinates
    for i in range(32):
        others = np.delete(y[i], [i, i + 32])
        assert np.all(others == 0.0)


def test_rope_preserves_pair_norms(oracle_mod):
    rng = np.random.default_rng(4)
    x = rng.standard_normal((257, 64))
    p = rng.integers(0, 8192, 257).astype(np.int32)
    y = oracle_mod.rope(x, p)
    nx = x[:, :32] ** 2 + x[:, 32:] ** 2
    ny = y[:, :32] ** 2 + y[:, 32:] ** 2
    np.testing.assert_allclose(ny, nx, rtol=1e-12, atol=1e-12)


def test_rope_relative_position(oracle_mod):
    # <R_m q, R_n k> depends only on m - n.  catches: any absolute-position leak,
    # sign error between the two halves.
    rng = np.random.default_rng(5)
    q = rng.standard_normal(64)
    k = rng.standard_normal(64)
    for (m, n) in [(3, 11), (1000, 17), (4095, 0), (100, 100)]:
        base = oracle_mod.rope(q[None], np.array([m], np.int32))[0] @ oracle_mod.rope(k[None], np.array([n], np.int32))[0]
        for t in [1, 37, 2048, 4000]:
            sh = oracle_mod.rope(q[None], np.array([m + t], np.int32))[0] @ oracle_mod.rope(k[None], np.array([n + t], np.int32))[0]
            assert abs(sh - base) < 1e-9 * max(1.0, abs(base))


def test_rope_position_zero_is_identity(oracle_mod):
    rng = np.random.default_rng(6)
    x = rng.standard_normal((9, 64))
    y = oracle_mod.rope(x, np.zeros(9, dtype=np.int32))
    np.testing.assert_array_equal(y, x)


# ----------------------------------------------------------------------------- attention

def _std_case(rng, B, H, L, dtype="fp16", dv=64):
    q = _rand_bits(rng, (B, H, L, 64), dtype)
    k = _rand_bits(rng, (B, H, L, 64), dtype)
    v = _rand_bits(rng, (B, H, L, dv), dtype)
    return q, k, v


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_attention_matches_torch_sdpa_at_position_zero(oracle_mod, dtype):
    # positions all zero -> RoPE is the identity, so the oracle must equal
    # torch's float64 SDPA on the decoded inputs.  catches: missing 1/sqrt(d),
    # transposed V, softmax over the wrong axis.
    rng = np.random.default_rng(7)
    B, H, L = 2, 3, 37
    q, k, v = _std_case(rng, B, H, L, dtype)
    pos = np.zeros(L, dtype=np.int32)
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, dtype=dtype, positions=pos)
    ref = _sdpa64(_decode64(q, dtype), _decode64(k, dtype), _decode64(v, dtype))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_rope_then_cast_then_sdpa(oracle_mod, dtype):
    # composition: oracle RoPE (pinned above) -> RNE cast (numpy / torch library
    # casts) -> torch SDPA equals the oracle's fused pipeline in "method" mode.
    rng = np.random.default_rng(8)
    B, H, L = 1, 2, 50
    q, k, v = _std_case(rng, B, H, L, dtype)
    pos = np.arange(L, dtype=np.int32) * 37 + 5
    qr = oracle_mod.rope(_decode64(q, dtype).reshape(-1, 64), np.tile(pos, B * H)).reshape(q.shape)
    kr = oracle_mod.rope(_decode64(k, dtype).reshape(-1, 64), np.tile(pos, B * H)).reshape(k.shape)
    if dtype == "fp16":
        cast = lambda a: a.astype(np.float16).astype(np.float64)
    else:
        cast = lambda a: oracle_mod.round_to(a, "bf16")
    ref = _sdpa64(cast(qr), cast(kr), _decode64(v, dtype))
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, dtype=dtype, positions=pos)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    # exact mode skips the cast: it must differ from method mode, but only slightly
    ex = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, dtype=dtype, positions=pos, cast="exact")
    ref_ex = _sdpa64(qr, kr, _decode64(v, dtype))
    np.testing.assert_allclose(ex, ref_ex, rtol=1e-12, atol=1e-13)
    assert np.abs(ex - got).max() > 0
    assert np.abs(ex - got).max() < (2e-3 if dtype == "fp16" else 2e-2)


def test_softmax_rows_sum_to_one(oracle_mod):
    # V = identity turns the output row into the probability row.
    rng = np.random.default_rng(9)
    L = 64
    q = _rand_bits(rng, (1, 1, L, 64), "fp16", 2.0)
    k = _rand_bits(rng, (1, 1, L, 64), "fp16", 2.0)
    v = synth.encode(np.eye(L, 64, dtype=np.float32)[None, None], "fp16")
    P = oracle_mod.rope_attn(q, k, v, B=1, H=1, L=L)[0, 0]
    np.testing.assert_allclose(P.sum(axis=1), 1.0, atol=1e-12)
    assert np.all(P > 0)


def test_constant_v_returns_v(oracle_mod):
    rng = np.random.default_rng(10)
    L = 40
    q = _rand_bits(rng, (1, 2, L, 64), "fp16", 3.0)
    k = _rand_bits(rng, (1, 2, L, 64), "fp16", 3.0)
    c = rng.standard_normal(64).astype(np.float32)
    v = synth.encode(np.broadcast_to(c, (1, 2, L, 64)), "fp16")
    out = oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L)
    np.testing.assert_allclose(out, np.broadcast_to(_decode64(synth.encode(c, "fp16"), "fp16"), out.shape),
                               rtol=1e-13, atol=1e-14)


def test_single_key_returns_v0(oracle_mod):
    rng = np.random.default_rng(11)
    q, k, v = _std_case(rng, 1, 3, 1)
    out = oracle_mod.rope_attn(q, k, v, B=1, H=3, L=1)
    np.testing.assert_array_equal(out, _decode64(v, "fp16"))


def test_zero_query_is_uniform_average(oracle_mod):
    rng = np.random.default_rng(12)
    L = 33
    _, k, v = _std_case(rng, 1, 1, L)
    q = np.zeros((1, 1, L, 64), dtype=np.uint16)
    out = oracle_mod.rope_attn(q, k, v, B=1, H=1, L=L)[0, 0]
    mean = _decode64(v, "fp16")[0, 0].mean(axis=0)
    np.testing.assert_allclose(out, np.broadcast_to(mean, out.shape), rtol=1e-12, atol=1e-14)
    # with a window the average is over the window only
    w = 3
    outw = oracle_mod.rope_attn(q, k, v, B=1, H=1, L=L, window=w)[0, 0]
    vd = _decode64(v, "fp16")[0, 0]
    for i in [0, 1, 16, L - 1]:
        np.testing.assert_allclose(outw[i], vd[max(0, i - w):min(L, i + w + 1)].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_dominant_logit_selects_its_value(oracle_mod):
    # one key aligned with a large query dominates: out ~= that key's value
    L = 16
    q = np.zeros((1, 1, L, 64), np.float32)
    k = np.zeros((1, 1, L, 64), np.float32)
    q[..., 0] = 200.0
    k[0, 0, 5, 0] = 200.0
    rng = np.random.default_rng(13)
    v = rng.standard_normal((1, 1, L, 64)).astype(np.float32)
    pos = np.zeros(L, np.int32)
    out = oracle_mod.rope_attn(synth.encode(q, "bf16"), synth.encode(k, "bf16"), synth.encode(v, "bf16"),
                               B=1, H=1, L=L, dtype="bf16", positions=pos)[0, 0]
    vd = _decode64(synth.encode(v, "bf16"), "bf16")[0, 0]
    np.testing.assert_allclose(out, np.broadcast_to(vd[5], out.shape), atol=1e-12)


def test_shift_invariance_of_logits(oracle_mod):
    # adding the same vector u to every key adds q.u/sqrt(d) to a whole logit row,
    # which softmax ignores (positions 0 so RoPE is the identity; exact cast mode).
    rng = np.random.default_rng(14)
    L = 29
    q = rng.standard_normal((1, 1, L, 64)).astype(np.float32)
    k = rng.standard_normal((1, 1, L, 64)).astype(np.float32)
    u = rng.standard_normal(64).astype(np.float32)
    v = rng.standard_normal((1, 1, L, 64)).astype(np.float32)
    pos = np.zeros(L, np.int32)
    # choose values exactly representable in bf16 so k + u stays exact
    enc = lambda a: synth.encode(a, "bf16")
    qb, vb = enc(q), enc(v)
    kb = enc(np.round(k * 4) / 4)
    ub = np.round(u * 4) / 4
    ku = enc(_decode64(kb, "bf16").astype(np.float32) + ub)
    assert np.array_equal(_decode64(ku, "bf16"), _decode64(kb, "bf16") + ub)
    a = oracle_mod.rope_attn(qb, kb, vb, B=1, H=1, L=L, dtype="bf16", positions=pos, cast="exact")
    b = oracle_mod.rope_attn(qb, ku, vb, B=1, H=1, L=L, dtype="bf16", positions=pos, cast="exact")
    np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_position_shift_invariance(oracle_mod):
    # whole pipeline: shifting every position by t leaves the output unchanged
    # (RoPE makes q_m . k_n depend on m - n only), in exact cast mode.
    rng = np.random.default_rng(15)
    L = 45
    q, k, v = _std_case(rng, 1, 2, L)
    p0 = np.arange(L, dtype=np.int32)
    a = oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L, positions=p0, cast="exact")
    b = oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L, positions=p0 + 3001, cast="exact")
    np.testing.assert_allclose(a, b, rtol=1e-9, atol=1e-11)
    # explicit arange equals the default positions bit for bit
    c = oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L, positions=p0)
    d = oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L)
    np.testing.assert_array_equal(c, d)


# ----------------------------------------------------------------------------- differential

def _diff_case(rng, B, H, L, dtype="bf16"):
    q = _rand_bits(rng, (B, H, 2, L, 64), dtype)
    k = _rand_bits(rng, (B, H, 2, L, 64), dtype)
    v = _rand_bits(rng, (B, H, L, 128), dtype)
    return q, k, v


def test_differential_lambda_zero_is_standard(oracle_mod):
    rng = np.random.default_rng(16)
    B, H, L = 1, 2, 31
    q, k, v = _diff_case(rng, B, H, L)
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, nmaps=2, dv=128, dtype="bf16", lam=np.zeros(H))
    std = oracle_mod.rope_attn(np.ascontiguousarray(q[:, :, 0]), np.ascontiguousarray(k[:, :, 0]), v,
                               B=B, H=H, L=L, dv=128, dtype="bf16")
    np.testing.assert_array_equal(got, std)


def test_differential_equal_maps_scale_by_one_minus_lambda(oracle_mod):
    # Q2 = Q1, K2 = K1 -> out = (1 - lambda_h) * standard.  catches: + instead of -,
    # lambda applied to the wrong map or the wrong head.
    rng = np.random.default_rng(17)
    B, H, L = 2, 3, 23
    q, k, v = _diff_case(rng, B, H, L)
    q[:, :, 1] = q[:, :, 0]
    k[:, :, 1] = k[:, :, 0]
    lam = np.array([0.2, 0.5, 0.8])
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, nmaps=2, dv=128, dtype="bf16", lam=lam)
    std = oracle_mod.rope_attn(np.ascontiguousarray(q[:, :, 0]), np.ascontiguousarray(k[:, :, 0]), v,
                               B=B, H=H, L=L, dv=128, dtype="bf16")
    np.testing.assert_allclose(got, (1 - lam)[None, :, None, None] * std, rtol=1e-12, atol=1e-14)


def test_differential_matches_two_sdpa_calls(oracle_mod):
    rng = np.random.default_rng(18)
    B, H, L = 1, 2, 40
    q, k, v = _diff_case(rng, B, H, L)
    lam = np.array([0.3, 0.7])
    pos = np.zeros(L, np.int32)
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, nmaps=2, dv=128, dtype="bf16", lam=lam, positions=pos)
    qd, kd, vd = _decode64(q, "bf16"), _decode64(k, "bf16"), _decode64(v, "bf16")
    ref = _sdpa64(qd[:, :, 0], kd[:, :, 0], vd) - lam[None, :, None, None] * _sdpa64(qd[:, :, 1], kd[:, :, 1], vd)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)


# ----------------------------------------------------------------------------- window

@pytest.mark.parametrize("w", [0, 1, 3, 17, 40])
def test_window_matches_masked_sdpa(oracle_mod, w):
    # catches: off-by-one at the window edge, one-sided window
    rng = np.random.default_rng(19 + w)
    B, H, L = 1, 2, 41
    q, k, v = _std_case(rng, B, H, L)
    pos = np.zeros(L, np.int32)
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, window=w, positions=pos)
    ref = _sdpa64(_decode64(q, "fp16"), _decode64(k, "fp16"), _decode64(v, "fp16"), mask=_window_mask(L, w))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_window_zero_returns_own_value(oracle_mod):
    rng = np.random.default_rng(30)
    L = 20
    q, k, v = _std_case(rng, 1, 1, L)
    out = oracle_mod.rope_attn(q, k, v, B=1, H=1, L=L, window=0)
    np.testing.assert_array_equal(out, _decode64(v, "fp16"))


def test_window_at_least_l_minus_one_is_full(oracle_mod):
    rng = np.random.default_rng(31)
    L = 26
    q, k, v = _std_case(rng, 1, 2, L)
    full = oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L)
    for w in [L - 1, L, 10 * L]:
        np.testing.assert_array_equal(oracle_mod.rope_attn(q, k, v, B=1, H=2, L=L, window=w), full)


# ----------------------------------------------------------------------------- plumbing

# ----------------------------------------------------------------------------- QK-RMSNorm

def test_rmsnorm_matches_torch_rms_norm(oracle_mod):
    # library routine: torch's float64 rms_norm with a weight.  catches: sum
    # instead of mean, eps outside the square root, a missing weight.
    rng = np.random.default_rng(40)
    x = rng.standard_normal((33, 64)) * np.exp(rng.uniform(-6, 6, (33, 1)))
    g = rng.uniform(0.5, 1.5, 64)
    for eps in (0.0, 1e-6, 1e-2):
        got = oracle_mod.rmsnorm(x, g, eps)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (64,), weight=torch.from_numpy(g),
                                           eps=eps).numpy()
        np.testing.assert_allclose(got, ref, rtol=1e-13, atol=0)


def test_rmsnorm_closed_forms(oracle_mod):
    # eps = 0, gamma = 1: unit mean square and invariance to a positive row scale;
    # a constant row c gives c / sqrt(c^2 + eps) in every entry; a zero row stays 0.
    rng = np.random.default_rng(41)
    x = rng.standard_normal((9, 64))
    y = oracle_mod.rmsnorm(x, None, 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=1), 1.0, rtol=1e-14)
    np.testing.assert_allclose(oracle_mod.rmsnorm(x * 1234.5, None, 0.0), y, rtol=1e-13, atol=1e-15)
    for c in (3.0, -0.25, 6.0e4):
        row = np.full((1, 64), c)
        np.testing.assert_allclose(oracle_mod.rmsnorm(row, None, 1e-6), c / math.sqrt(c * c + 1e-6),
                                   rtol=1e-15)
    assert np.all(oracle_mod.rmsnorm(np.zeros((1, 64)), None, 1e-6) == 0.0)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_qknorm_then_rope_then_cast_then_sdpa(oracle_mod, dtype):
    # composition: RMSNorm (pinned above) -> RoPE (pinned) -> RNE cast (library
    # casts) -> torch SDPA equals the oracle's pipeline with qk_norm.  Distinct,
    # non-uniform gammas for q and k make the order (norm before RoPE), the
    # tensor each gamma belongs to, and eps (small-magnitude rows) all matter;
    # fp16 rows near 6e4 would overflow a 16-bit sum of squares.
    rng = np.random.default_rng(42)
    B, H, L = 1, 2, 40
    q, k, v = _std_case(rng, B, H, L, dtype)
    scale = np.exp(rng.uniform(-9, 10, (B, H, L, 1)))
    qd = np.clip(_decode64(q, dtype) * scale, -6.0e4, 6.0e4)
    q = synth.encode(qd.astype(np.float32), dtype)
    pos = np.arange(L, dtype=np.int32) * 13 + 2
    gq = rng.uniform(0.25, 2.0, 64)
    gk = rng.uniform(0.25, 2.0, 64)
    eps = 1e-6
    cast = (lambda a: a.astype(np.float16).astype(np.float64)) if dtype == "fp16" else \
        (lambda a: oracle_mod.round_to(a, "bf16"))

    def prep(bits, g):
        n = oracle_mod.rmsnorm(_decode64(bits, dtype).reshape(-1, 64), g, eps)
        return cast(oracle_mod.rope(n, np.tile(pos, B * H)).reshape(bits.shape))

    ref = _sdpa64(prep(q, gq), prep(k, gk), _decode64(v, dtype))
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, dtype=dtype, positions=pos, qk_norm=(gq, gk, eps))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)
    swapped = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, dtype=dtype, positions=pos,
                                   qk_norm=(gk, gq, eps))
    assert np.abs(swapped - got).max() > 1e-3
    plain = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, dtype=dtype, positions=pos)
    assert np.abs(plain - got).max() > 1e-2


def test_qknorm_differential_and_window(oracle_mod):
    # the norm applies to both maps of q and k; windowed rows agree with a
    # masked torch SDPA on the normalised, rotated, cast operands.
    rng = np.random.default_rng(43)
    B, H, L, w = 1, 2, 33, 5
    q, k, v = _diff_case(rng, B, H, L)
    lam = rng.uniform(0.2, 0.8, H)
    gq, gk, eps = rng.uniform(0.5, 1.5, 64), rng.uniform(0.5, 1.5, 64), 1e-6
    cast = lambda a: oracle_mod.round_to(a, "bf16")

    def prep(bits, g):
        n = oracle_mod.rmsnorm(_decode64(bits, "bf16").reshape(-1, 64), g, eps)
        return cast(oracle_mod.rope(n, np.tile(np.arange(L, dtype=np.int32), B * H * 2)).reshape(bits.shape))

    qn, kn = prep(q, gq), prep(k, gk)
    vd = _decode64(v, "bf16")
    mask = _window_mask(L, w)
    o1 = _sdpa64(qn[:, :, 0], kn[:, :, 0], vd, mask)
    o2 = _sdpa64(qn[:, :, 1], kn[:, :, 1], vd, mask)
    ref = o1 - np.asarray(lam).reshape(1, H, 1, 1) * o2
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, nmaps=2, dv=128, dtype="bf16", window=w,
                               lam=lam, qk_norm=(gq, gk, eps))
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-13)


def test_row_subset_and_threads_are_consistent(oracle_mod):
    rng = np.random.default_rng(32)
    B, H, L = 2, 2, 30
    q, k, v = _std_case(rng, B, H, L)
    full = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, threads=1).reshape(-1, 64)
    rows = np.array([0, 5, 29, 30, 77, B * H * L - 1])
    sub = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, rows=rows, threads=5)
    np.testing.assert_array_equal(sub, full[rows])


def test_golden_tiny_rows(oracle_mod):
    # regression fixture written by tests/golden/make_golden.py (oracle only)
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "tiny_oracle_rows.txt")
    data = np.loadtxt(path)
    rows = data[:, 0].astype(np.int64)
    x = synth.make_inputs(synth.WORKLOADS["tiny"])
    got = oracle_mod.rope_attn_workload(x, rows=rows)
    np.testing.assert_allclose(got, data[:, 1:], rtol=0, atol=1e-15)


# ----------------------------------------------------------------------------- FP32-input form

def test_fp32_decode_matches_numpy(oracle_mod):
    # catches: wrong FP32 exponent bias or mantissa width, subnormal scale, sign, specials
    rng = np.random.default_rng(41)
    bits = np.concatenate([rng.integers(0, 2 ** 32, 20000, dtype=np.uint64).astype(np.uint32),
                           np.array([0, 1, 0x7FFFFF, 0x800000, 0x3F800000, 0x7F7FFFFF, 0x7F800000,
                                     0x80000000, 0x80000001, 0xFF800000], dtype=np.uint32)])
    bits = bits[((bits & 0x7F800000) != 0x7F800000) | ((bits & 0x7FFFFF) == 0)]   # no NaNs
    got = oracle_mod.bits_to_double(bits, "fp32")
    ref = bits.view(np.float32).astype(np.float64)
    np.testing.assert_array_equal(got, ref)


def test_round_fp32_matches_numpy(oracle_mod):
    # the method's cast for FP32 storage: numpy's float64 -> float32 cast (RNE) is the library
    # routine; includes exact ties (midpoints between adjacent floats) and subnormals
    rng = np.random.default_rng(42)
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-90, 90, 20000))
    f = rng.standard_normal(2000).astype(np.float32)
    ties = (f.astype(np.float64) + np.nextafter(f, np.float32(np.inf)).astype(np.float64)) / 2
    sub = rng.uniform(-1, 1, 500) * 2.0 ** -130
    x = np.concatenate([x, ties, sub, [0.0, -0.0, 3.4028234663852886e38]])
    got = oracle_mod.round_to(x, "fp32")
    np.testing.assert_array_equal(got, x.astype(np.float32).astype(np.float64))


def _f32_bits(rng, shape):
    return synth.encode(rng.standard_normal(shape).astype(np.float32), "fp32")


def test_fp32_differential_window_is_rope_cast_two_masked_sdpa(oracle_mod):
    # composition in the FP32-input form: oracle RoPE (pinned above) -> numpy float32 cast ->
    # torch float64 SDPA with the window mask, map 1 weighted by -lambda_h.  catches: FP32 bits
    # read as 16-bit elements, a 16-bit cast applied to FP32 storage, lambda on the wrong map
    rng = np.random.default_rng(43)
    B, H, L, w = 1, 2, 45, 6
    q, k, v = _f32_bits(rng, (B, H, 2, L, 64)), _f32_bits(rng, (B, H, 2, L, 64)), _f32_bits(rng, (B, H, L, 128))
    lam = np.array([0.35, 0.65])
    pos = np.arange(L, dtype=np.int32) * 11 + 3
    got = oracle_mod.rope_attn(q, k, v, B=B, H=H, L=L, nmaps=2, dv=128, dtype="fp32", lam=lam, window=w,
                               positions=pos)
    cast = lambda a: a.astype(np.float32).astype(np.float64)
    rot = lambda bits: cast(oracle_mod.rope(_decode64(bits, "fp32").reshape(-1, 64),
                                            np.tile(pos, bits.size // (64 * L))).reshape(bits.shape))
    qr, kr, vd = rot(q), rot(k), _decode64(v, "fp32")
    m = _window_mask(L, w)
    ref = _sdpa64(qr[:, :, 0], kr[:, :, 0], vd, m) - lam[None, :, None, None] * _sdpa64(qr[:, :, 1], kr[:, :, 1], vd, m)
    np.testing.assert_allclose(got, ref, rtol=1e-11, atol=1e-13)


def test_fp32_form_on_fp16_values_equals_fp16_form_exact(oracle_mod):
    # inputs that fp16 represents exactly: with the cast skipped ("exact" mode) only the decoding
    # differs, so the FP32 and fp16 forms must agree bit for bit
    rng = np.random.default_rng(44)
    B, H, L = 1, 2, 33
    h = [_rand_bits(rng, s, "fp16") for s in [(B, H, 2, L, 64), (B, H, 2, L, 64), (B, H, L, 128)]]
    f = [synth.encode(synth.decode(b, "fp16"), "fp32") for b in h]
    lam = np.array([0.4, 0.6])
    a = oracle_mod.rope_attn(*h, B=B, H=H, L=L, nmaps=2, dv=128, dtype="fp16", lam=lam, window=9, cast="exact")
    b = oracle_mod.rope_attn(*f, B=B, H=H, L=L, nmaps=2, dv=128, dtype="fp32", lam=lam, window=9, cast="exact")
    np.testing.assert_array_equal(a, b)
