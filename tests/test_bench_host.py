"""Host-side checks of bench.py's accounting (no GPU): the per-row FLOP count used for the
oracle's sample adds up to the closed form, the algorithmic bytes of each workload, and the
bookkeeping that ties the committed ncu traffic to the kernel source it was captured on."""

import json
import os
import shutil

import numpy as np
import pytest

import bench
import synth

W = synth.WORKLOADS


@pytest.mark.parametrize("name", ["tiny", "dit_l1292", "swa_diff_l8192", "swa17_diff_l8192"])
def test_row_flops_over_all_rows_is_the_closed_form(name):
    w = W[name]
    rows = np.arange(w.B * w.H * w.L, dtype=np.int64)
    assert bench.row_flops(w, rows) == bench.flops(w)


def test_algorithmic_bytes():
    # q and k (both maps), v read and out written once, 2 bytes per element
    assert bench.io_bytes(W["dit_l1292"]) == 2 * 16 * 1292 * (64 + 64 + 64 + 64)
    assert round(bench.io_bytes(W["dit_l1292"]) / 1e6, 2) == 10.58
    assert round(bench.io_bytes(W["dit_l4096_outliers"]) / 1e6, 2) == 50.33
    assert round(bench.io_bytes(W["diff_l4096"]) / 1e6, 2) == 67.11
    assert round(bench.io_bytes(W["swa_diff_l8192"]) / 1e6, 1) == 134.2


def _copy_tree(tmp_path):
    # the files bench reads for its bookkeeping, under a scratch root
    src_dir = os.path.join(bench.ROOT, "diffusion_transformer_attention_rope_gb300", "csrc")
    dst_dir = tmp_path / "diffusion_transformer_attention_rope_gb300" / "csrc"
    dst_dir.mkdir(parents=True)
    for name in os.listdir(src_dir):
        if name.endswith((".cu", ".cuh", ".h")):
            shutil.copy(os.path.join(src_dir, name), dst_dir / name)
    (tmp_path / "profiles").mkdir()
    shutil.copy(os.path.join(bench.ROOT, "profiles", "traffic.json"), tmp_path / "profiles" / "traffic.json")
    return dst_dir / "sa_fmha.cu"


def test_kernel_sha_ignores_comments_but_not_code(tmp_path, monkeypatch):
    src = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_sha()
    text = src.read_text()
    src.write_text("// a comment line\n\n" + text.replace("\n", "  // trailing note\n", 3) + "\n\n")
    assert bench.kernel_sha() == base
    src.write_text(text + "\nstatic int sa_unused_marker = 1;\n")
    assert bench.kernel_sha() != base


def test_kernel_sha_covers_the_device_headers_a_kernel_includes(tmp_path, monkeypatch):
    src = _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    base = bench.kernel_sha()
    hdr = src.parent / "sa_ptx.cuh"      # included through sa_pipe.cuh as well as directly
    text = hdr.read_text()
    hdr.write_text(text + "\n// a comment only\n")
    assert bench.kernel_sha() == base
    hdr.write_text(text + "\nstatic int sa_unused_marker = 1;\n")
    assert bench.kernel_sha() != base
    # a header no attention kernel includes does not count
    hdr.write_text(text)
    (src.parent / "sa_unrelated.cuh").write_text("static int sa_other = 2;\n")
    assert bench.kernel_sha() == base


def test_traffic_is_reported_only_for_the_captured_kernel(tmp_path, monkeypatch):
    _copy_tree(tmp_path)
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    stored = json.load(open(tmp_path / "profiles" / "traffic.json"))
    entry = stored["dit_l1292"]
    monkeypatch.setattr(bench, "kernel_sha", lambda w=None: entry["kernel_sha"])
    assert bench.load_traffic(W["dit_l1292"]) == entry["bytes"]
    assert bench.load_traffic(W["tiny"]) is None
    monkeypatch.setattr(bench, "kernel_sha", lambda w=None: "0" * 16)
    assert bench.load_traffic(W["dit_l1292"]) is None


def test_kernel_source_follows_the_library_routing():
    # the FP32-input form runs the TF32 kernel; differential windows up to 256 the narrow-window
    # kernel; everything else the general kernel
    assert bench.kernel_source(W["swa_diff_l8192_fp32"]) == "sa_tf32.cu"
    assert bench.kernel_source(W["swa_diff_l8192"]) == "sa_swa.cu"
    assert bench.kernel_source(W["swa17_diff_l8192"]) == "sa_swa.cu"
    assert bench.kernel_source(W["diff_l4096"]) == "sa_fmha.cu"
    assert bench.kernel_source(W["dit_l4096_outliers"]) == "sa_fmha.cu"
    src = open(os.path.join(bench.ROOT, "diffusion_transformer_attention_rope_gb300", "csrc", "sa_kernels.h")).read()
    assert f"constexpr int kSwaMaxWindow = {bench.SWA_MAX_WINDOW};" in src


def test_committed_traffic_is_at_least_the_compulsory_reads():
    # every capture in profiles/traffic.json carries the kernel hash it was taken on, and its
    # DRAM bytes are at least the compulsory reads of q, k', v (no capture can read less)
    stored = json.load(open(os.path.join(bench.ROOT, "profiles", "traffic.json")))
    for name, entry in stored.items():
        assert len(entry["kernel_sha"]) == 16, name
        w = W[name]
        n = w.B * w.H * w.L
        elem = 4 if w.dtype == "fp32" else 2
        compulsory = elem * (n * w.nmaps * w.d * 2 + n * w.dv)
        assert entry["bytes"] >= 0.99 * compulsory, name


def test_peaks_fall_back_without_the_measured_file(tmp_path, monkeypatch):
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    p = bench.load_peaks()
    assert p["source"] == "fallback" and p["hbm_gbs"] == 6800.0 and p["tflops"] == 1900.0
    (tmp_path / "MEASURED_PEAKS.json").write_text(json.dumps({"hbm_gbs": 7000.0, "bf16_tflops": 2000.0}))
    p = bench.load_peaks()
    assert p["source"] == "measured" and p["tflops"] == 2000.0 and p["tflops_sustained"] == 2000.0
