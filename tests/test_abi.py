"""Host-side checks of the C ABI (no GPU needed): the library builds, loads and
exports exactly what include/sa_attn.h declares; host validation rejects bad
arguments before any device work."""

import os
import re
import subprocess

import pytest

import diffusion_transformer_attention_rope_gb300 as sa
from diffusion_transformer_attention_rope_gb300 import build as sa_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sa_attn.h")


@pytest.fixture(scope="module")
def lib():
    sa_build.build()
    return sa.load_library()


def _declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^SA_API\s+[\w\s\*]+?\b(sa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ["sa_attn_create", "sa_rope_attn", "sa_attn_destroy"]:
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", sa.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(sa_\w+)$", out, flags=re.M))
    declared = set(_declared_functions())
    assert declared == exported, (declared ^ exported)
    for name in declared:
        assert hasattr(lib, name)


def test_library_is_built_for_sm103a_only():
    # the build compiles every translation unit for sm_103a alone (one -gencode, no PTX for
    # other targets); on a GPU, sa_attn_create checks each attention kernel's binary version
    # (cudaFuncGetAttributes) is 10.3 and refuses to run otherwise
    assert sa_build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    src = open(os.path.join(ROOT, "diffusion_transformer_attention_rope_gb300", "csrc", "sa_fmha.cu")).read()
    assert "attr.binaryVersion != 103" in src


def _a256(x):
    return (x + 255) // 256 * 256


def _split_bytes(B, H, L, diff):
    # one 8-byte counter per query block (256 rows standard, 128 differential), then 160
    # FP32 partial-result slots of 2*128*(d_v + 2) values
    rows = 128 if diff else 256
    dv = 128 if diff else 64
    units = B * H * ((L + rows - 1) // rows)
    return _a256(units * 8) + _a256(160 * 2 * 128 * (dv + 2) * 4)


def test_workspace_size():
    # the (cos, sin) table of L * 32 FP32 pairs, k' (B*H*nmaps*L*64 two-byte elements), each
    # rounded up to 256 bytes, then the split region
    assert sa.sa_rope_table_bytes(1292) == 1292 * 32 * 8
    assert sa.sa_rope_table_bytes(0) == 0
    n = 1 * 16 * 1292 * 64 * 2
    assert sa.sa_rope_attn_workspace_size(1, 16, 1292, 64, False) == \
        _a256(1292 * 256) + _a256(n) + _split_bytes(1, 16, 1292, False)
    n = 1 * 16 * 2 * 4096 * 64 * 2
    assert sa.sa_rope_attn_workspace_size(1, 16, 4096, 64, True) == 4096 * 256 + n + _split_bytes(1, 16, 4096, True)
    assert sa.sa_attn_fwd_workspace_size(1, 24, 4096, 64, False) == _split_bytes(1, 24, 4096, False)
    assert sa.sa_attn_fwd_workspace_size(2, 3, 777, 64, True) == _split_bytes(2, 3, 777, True)
    assert sa.sa_rope_attn_workspace_size(1, 16, 4096, 128, True) == 0
    assert sa.sa_attn_fwd_workspace_size(1, 16, 4096, 128, True) == 0
    assert sa.sa_rope_attn_workspace_size(0, 16, 4096, 64, False) == 0
    assert sa.sa_attn_fwd_workspace_size(0, 16, 4096, 64, False) == 0
    assert sa.sa_rope_attn_workspace_size(1, 1, -5, 64, False) == 0


def test_status_strings():
    assert sa.sa_status_string(0) == "SA_OK"
    assert sa.sa_status_string(6) == "SA_ERR_WORKSPACE"
    assert sa.sa_status_string(99) == "SA_ERR_UNKNOWN"


def test_null_handle_is_rejected_on_the_host():
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_rope_attn(0, 256, 256, 256, None, 256, 1, 1, 64, 64, -1, None, sa.SA_FP16, 256, 1 << 20, None)
    assert e.value.status == 1
    assert "handle" in sa.sa_last_error()


def test_qknorm_parameters_are_checked_on_the_host():
    # eps and gamma are validated before anything else; nothing is enqueued
    args = (256, 256, 256, None)
    for gq, eps, word in (([1.0] * 64, -1.0, "eps"), ([1.0] * 64, float("nan"), "eps"),
                          ([1.0] * 63 + [float("inf")], 1e-6, "gamma")):
        with pytest.raises(sa.SaAttnError) as e:
            sa.sa_rope_attn_qknorm(0, *args, gq, None, eps, 256, 1, 1, 64, 64, -1, None, sa.SA_FP16,
                                   256, 1 << 20, None)
        assert e.value.status == 1
        assert word in sa.sa_last_error()
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_rope_attn_qknorm(0, *args, None, None, 1e-6, 256, 1, 1, 64, 64, -1, None, sa.SA_FP16,
                               256, 1 << 20, None)
    assert e.value.status == 1 and "handle" in sa.sa_last_error()
    with pytest.raises(ValueError):
        sa.sa_qknorm_rope_qk(0, 256, 256, None, [1.0] * 32, None, 1e-6, 256, 256, 1, 1, 64, 64, 1,
                             sa.SA_FP16, None)


def test_create_without_a_gpu_reports_no_device():
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_attn_create(0)
    assert e.value.status == 5


def test_create_rejects_bad_rope_base():
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_attn_create(0, rope_base=0.5)
    assert e.value.status == 1


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    # the product path has no fallback: a missing .so is an error, not a slow path
    monkeypatch.setattr(sa, "_lib", None)
    monkeypatch.setattr(sa, "library_path", lambda: str(tmp_path / "libsa_attn.so"))
    with pytest.raises(sa.SaAttnError):
        sa.load_library()


def test_set_timeout_null_handle_is_rejected():
    with pytest.raises(sa.SaAttnError) as e:
        sa.sa_attn_set_timeout(0, 1000)
    assert e.value.status == 1


def _host_chunks(B, H, L, diff):
    # the host-buffer call's chunks: about one per 16 MiB of copies (two from 8 MiB up), at
    # most 4, more when a chunk would exceed 128 planes; returns (chunks, planes of the largest)
    P = B * H
    total = P * 2.0 * L * 64 * (2 if diff else 1) * 4
    mib16 = 16 * 1024 * 1024
    by_size = int(total / mib16) if total >= mib16 else (2 if total >= mib16 / 2 else 1)
    n = max(min(min(4, by_size), P), -(-P // 128))
    return n, -(-P // n)


@pytest.mark.parametrize("B,H,L,diff,chunks", [
    (2, 3, 300, False, 1),      # 3.7 MB of copies: one chunk
    (1, 16, 1292, False, 2),    # 10.6 MB: two chunks of 8 planes
    (1, 24, 4096, False, 3),    # 50 MB: three chunks
    (1, 16, 4096, True, 4),     # 67 MB: at most four
    (5, 128, 64, True, 5),      # 640 planes: chunks of at most 128 planes
])
def test_host_workspace_follows_the_chunk_rule(B, H, L, diff, chunks):
    # device copies of q, k (both maps), v and out, then one sa_rope_attn workspace (for the
    # largest chunk) per compute stream in use
    n, max_len = _host_chunks(B, H, L, diff)
    assert n == chunks
    nqk = B * H * (2 if diff else 1) * L * 64
    nv = B * H * L * (128 if diff else 64)
    per = sa.sa_rope_attn_workspace_size(1, max_len, L, 64, diff)
    assert sa.sa_rope_attn_host_workspace_size(B, H, L, 64, diff) == \
        2 * _a256(nqk * 2) + 2 * _a256(nv * 2) + min(n, 4) * per
    assert sa.sa_rope_attn_host_workspace_size(0, H, L, 64, diff) == 0
