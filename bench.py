"""Benchmark of the RoPE + attention core on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step = one pass of the whole hot path over one batch of synthetic input:
the RoPE stage (q, k rotated in FP32, cast back) and the attention stage
(QK^T/sqrt(d), FP32 softmax, P.V; differential / windowed per workload).
Default workload: the DiT standard attention at L=1292 (B=1, H=16, d=64, fp16).

The default run also measures the L=4096 DiT workload (the configuration the
60%-of-peak target is quoted on), differential attention and the two sliding
windows, each with the same fields, under the line's ``workloads`` map
(``--headline-only`` skips them).

Prints ONE JSON line (rank 0).  ``value`` is attention TFLOP/s of the whole job
(algorithmic FLOPs, inputs resident in HBM, L2 flushed between steps, CUDA
events on the launching stream, max over ranks).  ``e2e`` is the same metric
through the public C-ABI call with pinned host buffers and the host<->device
copies inside the timed region.  ``roofline`` is for the attention kernel,
timed live between events recorded around its own launch.  ``cpu_baseline``
times the FP64 oracle on the host cores on a bounded sample.

``--impl reference`` times the FP64 CPU oracle (the reference arm of this
repository) on the same workload; each step is a bounded sample of it.
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(the path shards by (batch, head) with no exchange), so scaling is weak.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "attention TFLOP/s and % of GB300 FP16/BF16 tensor peak at L=1292/4096"
DEFAULT_WORKLOAD = "dit_l1292"
DEFAULT_WORKLOADS_HEADLINE = DEFAULT_WORKLOAD
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------------------- accounting

def allowed_pairs_per_head(w) -> int:
    """(query, key) pairs the mask admits per head: all L^2, or |i - j| <= window."""
    L, win = w.L, w.window
    if win < 0 or win >= L - 1:
        return L * L
    i = np.arange(L, dtype=np.int64)
    return int((np.minimum(L - 1, i + win) - np.maximum(0, i - win) + 1).sum())


def flops(w) -> int:
    """Algorithmic FLOPs: per softmax map and allowed pair, 2*d (QK^T) + 2*d_v (P.V)."""
    return w.B * w.H * w.nmaps * allowed_pairs_per_head(w) * (2 * w.d + 2 * w.dv)


def io_bytes(w) -> int:
    """q', k' (both maps), v read once and out written once, in the storage dtype."""
    n = w.B * w.H * w.L
    elem = 4 if w.dtype == "fp32" else 2
    return elem * (n * w.nmaps * w.d * 2 + n * w.dv + n * w.dv)


# Dense TF32 / dense BF16 tensor rate, nominal (GB300: 1.1 and 2.25 PFLOP/s): the FP32-input
# workloads' products run as TF32 MMAs, so their peak is the measured bf16 rate times this.
TF32_OVER_BF16 = 1.1 / 2.25


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": float(p["hbm_gbs"]), "tflops": float(p["bf16_tflops"]),
                "tflops_sustained": float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "tflops": 1900.0, "tflops_sustained": 1700.0, "source": "fallback"}


# Differential windows up to this width run the narrow-window kernel (the library's rule).
SWA_MAX_WINDOW = 256


def kernel_source(w=None) -> str:
    """Source file of the attention kernel a workload runs: the FP32-input (TF32) kernel, the
    narrow-window differential kernel, or the general one."""
    if w is not None and w.dtype == "fp32":
        return "sa_tf32.cu"
    if w is not None and w.nmaps == 2 and 0 <= w.window <= SWA_MAX_WINDOW and w.window < w.L - 1:
        return "sa_swa.cu"
    return "sa_fmha.cu"


def kernel_sha(w=None, read=None) -> str:
    """Hash of the workload's attention kernel source and of the device headers it includes
    (sa_*.cuh, transitively), with comments and blank lines removed, so that the stored ncu
    counters stay valid across comment-only edits and no others.  `read(name)` returns a source
    file's text (default: the file in the package's csrc)."""
    import hashlib
    import re

    csrc = os.path.join(ROOT, "diffusion_transformer_attention_rope_gb300", "csrc")
    if read is None:
        def read(name):
            with open(os.path.join(csrc, name)) as f:
                return f.read()
    names, todo = [], [kernel_source(w)]
    while todo:
        name = todo.pop(0)
        if name in names:
            continue
        names.append(name)
        todo += re.findall(r'^#include "(sa_\w+\.cuh)"', read(name), flags=re.M)
    h = hashlib.sha256()
    for name in [names[0]] + sorted(names[1:]):
        code = [re.sub(r"\s*//.*$", "", ln).rstrip() for ln in read(name).splitlines()]
        h.update(("\n".join(ln for ln in code if ln) + "\n").encode())
    return h.hexdigest()[:16]


def load_traffic(w):
    """DRAM bytes per attention launch from the committed ncu summary, or None when no
    capture exists for this workload or the kernel source changed since it was taken."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f).get(w.name)
        if t and t.get("kernel_sha") == kernel_sha(w):
            return t["bytes"]
    except Exception:
        pass
    return None


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """SM clock and throttle reasons sampled DURING the timed region.

    A thread polls NVML (libnvidia-ml through ctypes) every ~0.5 ms, so even a
    millisecond-long timed region gets samples; nvidia-smi (-lms 200) is the fallback.
    Only reads are made: no clock or other GPU setting is changed.
    """

    REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, cuda_index: int):
        self.cuda_index = cuda_index
        self.samples = []
        self.max_mhz = None
        self._stop = False
        self._thread = None
        self._nv = None
        self._smi = None

    def _nvml_handle(self):
        import ctypes

        import torch

        nv = ctypes.CDLL("libnvidia-ml.so.1")
        if nv.nvmlInit_v2() != 0:
            return None
        props = torch.cuda.get_device_properties(self.cuda_index)
        bus = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), props.pci_bus_id, props.pci_device_id)
        h = ctypes.c_void_p()
        if nv.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(h)) != 0:
            return None
        mx = ctypes.c_uint()
        if nv.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0:
            self.max_mhz = float(mx.value)
        self._nv = nv
        return h

    def _poll(self, h):
        import ctypes

        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        get_reasons = getattr(self._nv, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            self._nv.nvmlDeviceGetCurrentClocksThrottleReasons
        while not self._stop:
            if self._nv.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(clk)) == 0:
                r = rs.value if get_reasons(h, ctypes.byref(rs)) == 0 else 0
                self.samples.append((float(clk.value), int(r)))
            time.sleep(0.0005)

    def start(self):
        import threading

        try:
            h = self._nvml_handle()
        except Exception:
            h = None
        if h is not None:
            self._thread = threading.Thread(target=self._poll, args=(h,), daemon=True)
            self._thread.start()
            while not self.samples and self._thread.is_alive():
                time.sleep(0.0005)
            return
        try:
            self._path = os.path.join("/tmp", f"sa_clocks_{os.getpid()}.csv")
            self._f = open(self._path, "w")
            self._smi = subprocess.Popen(
                ["nvidia-smi", f"--id={self.cuda_index}", "--query-gpu=clocks.sm,clocks.max.sm,"
                 "clocks_event_reasons.active", "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=self._f, stderr=subprocess.DEVNULL)
        except Exception:
            self._smi = None

    def stop(self):
        if self._thread is not None:
            self._stop = True
            self._thread.join(timeout=5)
        elif self._smi is not None:
            self._smi.terminate()
            try:
                self._smi.wait(timeout=5)
            except Exception:
                self._smi.kill()
            self._f.close()
            for line in open(self._path):
                parts = [p.strip() for p in line.split(",")]
                try:
                    self.samples.append((float(parts[0]), int(parts[2], 16)))
                    self.max_mhz = float(parts[1])
                except (ValueError, IndexError):
                    continue
            os.unlink(self._path)
        if not self.samples:
            return None
        reasons = sorted({name for _, r in self.samples for bit, name in self.REASONS.items() if r & bit})
        return {"sm_mhz": statistics.median(c for c, _ in self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples), "reasons": reasons,
                "source": "nvml" if self._thread is not None else "nvidia-smi"}


# ----------------------------------------------------------------------------- distributed

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(world, backend):
    if world > 1:
        import torch.distributed as dist

        os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
        dist.init_process_group(backend=backend)
        return dist
    return None


def reduce_max(dist, value: float, device=None) -> float:
    """Max over ranks (device None: a CPU tensor, for the gloo backend)."""
    if dist is None:
        return value
    import torch

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, flops_per_rank_step: int, steps: int, max_total_ms: float) -> float:
    """Whole-job TFLOP/s: the work of every rank divided by the slowest rank's time."""
    return world * flops_per_rank_step * steps / (max_total_ms * 1e-3) / 1e12


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ----------------------------------------------------------------------------- CPU baseline (oracle)

def row_flops(w, rows: np.ndarray) -> int:
    i = rows % w.L
    if w.window < 0 or w.window >= w.L - 1:
        keys = np.full(i.shape, w.L, dtype=np.int64)
    else:
        keys = np.minimum(w.L - 1, i + w.window) - np.maximum(0, i - w.window) + 1
    return int(keys.sum()) * w.nmaps * (2 * w.d + 2 * w.dv)


def qk_norm_params(enabled: bool):
    """The QK-RMSNorm of --qk-norm: seeded gammas ~ U(0.5, 1.5) for q and k, eps 1e-6 (the
    pages give no values; these stand in for learned weights)."""
    if not enabled:
        return None
    rng = np.random.default_rng(60)
    return (rng.uniform(0.5, 1.5, 64).astype(np.float32), rng.uniform(0.5, 1.5, 64).astype(np.float32), 1e-6)


def oracle_sample(w, x, budget_s: float, rng, threads=None, qk_norm=None):
    """Time the FP64 oracle on a random row sample sized to ~budget_s of work.
    Returns (tflops, seconds, rows_done, threads)."""
    import oracle

    oracle.build()
    threads = threads or oracle.default_threads()
    total = w.B * w.H * w.L
    nrm = None if qk_norm is None else (qk_norm[0].astype(np.float64), qk_norm[1].astype(np.float64), qk_norm[2])
    probe = rng.choice(total, size=min(total, max(64, total // 200)), replace=False)
    t0 = time.perf_counter()
    oracle.rope_attn_workload(x, rows=probe, threads=threads, qk_norm=nrm)
    dt = max(time.perf_counter() - t0, 1e-3)
    n = int(min(total, max(len(probe), len(probe) * budget_s / dt)))
    rows = rng.choice(total, size=n, replace=False)
    t0 = time.perf_counter()
    oracle.rope_attn_workload(x, rows=rows, threads=threads, qk_norm=nrm)
    dt = time.perf_counter() - t0
    return row_flops(w, rows) / dt / 1e12, dt, n, threads


# ----------------------------------------------------------------------------- our arm

def workload_of(args):
    w = synth.WORKLOADS[args.workload]
    if args.batch is not None and args.batch != w.B:
        w = w.with_(B=args.batch)
    return w


# Workloads measured beside the headline one in the default run (each in the line's `workloads`
# map): the long-sequence DiT configuration that the 60% target is quoted on, differential
# attention, the two sliding windows, and the FP32-input form (TF32 products) of the first.
EXTRA_WORKLOADS = ["dit_l4096_outliers", "diff_l4096", "swa_diff_l8192", "swa17_diff_l8192", "swa_diff_l8192_fp32"]


def run_ours(args):
    import torch

    world, rank, local = dist_env()
    dist = dist_init(world, "nccl")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    w = workload_of(args)
    res = measure(args, w, dist, world, rank, local, device, cpu_budget=args.cpu_budget)
    if args.all_workloads and args.workload == DEFAULT_WORKLOADS_HEADLINE and args.batch is None:
        extra = {}
        for name in EXTRA_WORKLOADS:
            r = measure(args, synth.WORKLOADS[name], dist, world, rank, local, device,
                        cpu_budget=args.extra_cpu_budget)
            if r is not None:
                extra[name] = {k: r[k] for k in ("value", "unit", "ms_per_step", "step_ms", "frac_of_peak", "dtype",
                                                 "config", "roofline", "stages_ms", "graph", "cpu_baseline", "e2e",
                                                 "gpu_launches", "clocks")}
        if res is not None:
            res["workloads"] = extra
    return res


def measure(args, w, dist, world, rank, local, device, cpu_budget):
    """One workload: the timed regions below; the JSON fields of rank 0 (None elsewhere)."""
    import torch

    import diffusion_transformer_attention_rope_gb300 as sa

    x = synth.make_inputs(w, seed=w.seed + rank)
    tdt = {"fp16": torch.float16, "bf16": torch.bfloat16, "fp32": torch.float32}[w.dtype]
    dtype = {"fp16": sa.SA_FP16, "bf16": sa.SA_BF16, "fp32": sa.SA_FP32}[w.dtype]
    fp32 = w.dtype == "fp32"

    def to_dev(bits):
        if fp32:
            return torch.from_numpy(bits.view(np.int32)).to(device).view(tdt)
        return torch.from_numpy(bits.view(np.int16)).to(device).view(tdt)

    q, k, v = to_dev(x["q"]), to_dev(x["k"]), to_dev(x["v"])
    out = torch.empty((w.B, w.H, w.L, w.dv), dtype=tdt, device=device)
    lam = None if x["lam"] is None else [float(t) for t in x["lam"]]
    ws_bytes = sa.sa_rope_attn_workspace_bytes(w.B, w.H, w.L, w.d, w.differential, dtype)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device=device)
    nqk = q.numel()
    # the workspace of sa_rope_attn: the (cos, sin) table, k', the split region; region 2 runs
    # the same two stages through their own entry points on the same buffers
    a256 = lambda n: (n + 255) // 256 * 256
    off_k = a256(sa.sa_rope_table_bytes(w.L))
    off_split = off_k + a256(nqk * 2)
    cs_table = ws[:off_k]
    k_rot = ws[off_k:off_k + nqk * 2]
    split = ws[off_split:]
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=device)
    h = sa.sa_attn_create(local)
    stream = torch.cuda.current_stream(device)
    s = stream.cuda_stream

    nrm = qk_norm_params(args.qk_norm)
    if fp32:
        # the FP32-input form: its two stages are the FP32 RoPE pass (q' and k' into the
        # workspace) and the TF32 attention kernel on them
        if nrm is not None:
            raise SystemExit("--qk-norm has no FP32 form")
        off_k32 = a256(nqk * 4)
        off_v32 = 2 * a256(nqk * 4)

        def rope():
            sa.sa_rope_qkv_f32(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, ws.data_ptr(),
                               ws.data_ptr() + off_k32, ws.data_ptr() + off_v32, w.B, w.H, w.L, w.d, s)

        def attn():
            sa.sa_attn_fwd_f32(h, ws.data_ptr(), ws.data_ptr() + off_k32, ws.data_ptr() + off_v32, out.data_ptr(),
                               w.B, w.H, w.L, w.d, w.window, lam, s)

        def full():
            sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(), w.B, w.H,
                            w.L, w.d, w.window, lam, dtype, ws.data_ptr(), ws_bytes, s)
    elif nrm is None:
        def rope():
            sa.sa_rope_k(h, k.data_ptr(), None, k_rot.data_ptr(), cs_table.data_ptr(),
                         w.B, w.H, w.L, w.d, w.nmaps, dtype, s)

        def attn():
            sa.sa_attn_fwd_rope_q(h, q.data_ptr(), k_rot.data_ptr(), cs_table.data_ptr(), v.data_ptr(),
                                  out.data_ptr(), w.B, w.H, w.L, w.d, w.window, lam, dtype, s,
                                  split.data_ptr(), split.numel())

        def full():
            sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(), w.B, w.H,
                            w.L, w.d, w.window, lam, dtype, ws.data_ptr(), ws_bytes, s)
    else:
        # QK-RMSNorm: region 2 times the two-stage form (normalised, rotated q' and k' from the
        # pre-pass, then the attention kernel on them), the only split form this variant has
        gq, gk, eps = nrm[0].tolist(), nrm[1].tolist(), nrm[2]
        q_rot = torch.empty_like(q)

        def rope():
            sa.sa_qknorm_rope_qk(h, q.data_ptr(), k.data_ptr(), None, gq, gk, eps, q_rot.data_ptr(),
                                 k_rot.data_ptr(), w.B, w.H, w.L, w.d, w.nmaps, dtype, s)

        def attn():
            sa.sa_attn_fwd(h, q_rot.data_ptr(), k_rot.data_ptr(), v.data_ptr(), out.data_ptr(), w.B, w.H,
                           w.L, w.d, w.window, lam, dtype, s, split.data_ptr(), split.numel())

        def full():
            sa.sa_rope_attn_qknorm(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, gq, gk, eps,
                                   out.data_ptr(), w.B, w.H, w.L, w.d, w.window, lam, dtype,
                                   ws.data_ptr(), ws_bytes, s)

    for _ in range(args.warmup):
        flush.zero_()
        full()
        flush.zero_()
        rope()
        attn()
    torch.cuda.synchronize(device)
    sa.sa_attn_check(h)

    # timed region 1 (value): the whole path as one public call per step
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    clocks = ClockSampler(local)
    barrier(dist)
    torch.cuda.synchronize(device)
    clocks.start()
    for i in range(args.steps):
        flush.zero_()                      # L2 flush outside the timed events
        ev[i][0].record(stream)
        full()
        ev[i][1].record(stream)
    torch.cuda.synchronize(device)
    barrier(dist)
    clk = clocks.stop()
    sa.sa_attn_check(h)
    step_ms = [e[0].elapsed_time(e[1]) for e in ev]
    total_ms = reduce_max(dist, float(sum(step_ms)), device)

    # the same step replayed from a CUDA graph (the call enqueues no host work, so it captures
    # whole): what the launches themselves cost at small sizes.  Reported beside `value`.
    graph_ms = None
    if nrm is None:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            sa.sa_rope_attn(h, q.data_ptr(), k.data_ptr(), v.data_ptr(), None, out.data_ptr(), w.B, w.H,
                            w.L, w.d, w.window, lam, dtype, ws.data_ptr(), ws_bytes,
                            torch.cuda.current_stream(device).cuda_stream)
        evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for _ in range(args.warmup):
            flush.zero_()
            g.replay()
        torch.cuda.synchronize(device)
        for i in range(args.steps):
            flush.zero_()
            evg[i][0].record(stream)
            g.replay()
            evg[i][1].record(stream)
        torch.cuda.synchronize(device)
        sa.sa_attn_check(h)
        graph_ms = reduce_max(dist, float(sum(e[0].elapsed_time(e[1]) for e in evg)), device) / args.steps
        del g

    # timed region 2 (roofline): the two stages with events around the attention launch
    ev3 = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        flush.zero_()
        ev3[i][0].record(stream)
        rope()
        ev3[i][1].record(stream)
        attn()
        ev3[i][2].record(stream)
    torch.cuda.synchronize(device)
    sa.sa_attn_check(h)
    attn_ms = [e[1].elapsed_time(e[2]) for e in ev3]
    rope_ms = [e[0].elapsed_time(e[1]) for e in ev3]

    # e2e: the C-ABI call on pinned HOST buffers (sa_rope_attn_host: copies in, the path, copy out,
    # pipelined over chunks of planes), the copies inside the timed region.  The QK-norm variant
    # and the FP32 form have no host entry: their copies are plain stream copies around the
    # device call.
    qh, kh, vh = (t.cpu().pin_memory() for t in (q, k, v))
    oh = torch.empty(out.shape, dtype=tdt).pin_memory()
    ev2 = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    hws_bytes = sa.sa_rope_attn_host_workspace_size(w.B, w.H, w.L, w.d, w.differential)
    hws = torch.empty(hws_bytes, dtype=torch.uint8, device=device) if nrm is None and not fp32 else None

    def e2e_step(e=None):
        if e is not None:
            e[0].record(stream)
        if nrm is None and not fp32:
            sa.sa_rope_attn_host(h, qh.data_ptr(), kh.data_ptr(), vh.data_ptr(), None, oh.data_ptr(), w.B, w.H,
                                 w.L, w.d, w.window, lam, dtype, hws.data_ptr(), hws_bytes, s)
        else:
            q.copy_(qh, non_blocking=True)
            k.copy_(kh, non_blocking=True)
            v.copy_(vh, non_blocking=True)
            full()
            oh.copy_(out, non_blocking=True)
        if e is not None:
            e[1].record(stream)

    for _ in range(args.warmup):
        flush.zero_()
        e2e_step()
    barrier(dist)
    torch.cuda.synchronize(device)
    for i in range(args.steps):
        flush.zero_()
        e2e_step(ev2[i])
    torch.cuda.synchronize(device)
    barrier(dist)
    sa.sa_attn_check(h)
    e2e_total = reduce_max(dist, float(sum(e[0].elapsed_time(e[1]) for e in ev2)), device)
    h2d = sum(t.numel() * t.element_size() for t in (q, k, v))
    d2h = out.numel() * out.element_size()
    sa.sa_attn_destroy(h)

    if rank != 0:
        return None
    fl = flops(w)
    peaks = load_peaks()
    if fp32:
        peaks = dict(peaks, tflops=peaks["tflops"] * TF32_OVER_BF16,
                     source=peaks["source"] + " bf16 burst x nominal tf32/bf16 (1.1/2.25); tf32")
    value = job_throughput(world, fl, args.steps, total_ms)
    attn_avg_s = statistics.mean(attn_ms) * 1e-3
    achieved = fl / attn_avg_s / 1e12
    cpu = None
    if not args.no_cpu_baseline and world == 1:
        tfl, dt, n, th = oracle_sample(w, x, cpu_budget, np.random.default_rng(0), qk_norm=nrm)
        cpu = {"value": tfl, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
               "sample": f"{n} of {w.B * w.H * w.L} query rows (random, all heads), {dt:.1f} s, FP64 C oracle"}
    return {
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": total_ms / args.steps,
        "step_ms": {"median": statistics.median(step_ms), "min": min(step_ms), "max": max(step_ms)},
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "d_v": w.dv,
                   "maps": w.nmaps, "window": w.window, "flops_per_step_per_gpu": fl,
                   "l2": "flushed before every step (256 MiB write, outside the events)",
                   "parallelism": f"replicas x{world}", "qk_norm": nrm is not None},
        "frac_of_peak": value / world / peaks["tflops"],
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peaks["tflops"], "unit": "TFLOP/s",
                     "frac": achieved / peaks["tflops"],
                     "traffic": load_traffic(w) if nrm is None else None,
                     "kernel": ("attention, TF32 (sa_attn_fwd_f32 on sa_rope_qkv_f32 output)" if fp32 else
                                "attention (sa_attn_fwd_rope_q)" if nrm is None else
                                "attention (sa_attn_fwd on sa_qknorm_rope_qk output)"),
                     "kernel_source": kernel_source(w), "kernel_sha": kernel_sha(w),
                     "peak_source": peaks["source"] if fp32 else peaks["source"] + " bf16 burst",
                     "avg_ms": attn_avg_s * 1e3,
                     # the same launch against the HBM roof: algorithmic bytes (q', k', v read once,
                     # out written once) over its duration, of the measured copy bandwidth
                     "hbm": {"achieved": io_bytes(w) / attn_avg_s / 1e9, "peak": peaks["hbm_gbs"],
                             "unit": "GB/s", "frac": io_bytes(w) / attn_avg_s / 1e9 / peaks["hbm_gbs"]}},
        "stages_ms": {"rope": statistics.mean(rope_ms), "attention": statistics.mean(attn_ms)},
        "graph": None if graph_ms is None else {"ms_per_step": graph_ms,
                                                "value": job_throughput(world, fl, 1, graph_ms)},
        "cpu_baseline": cpu,
        "e2e": {"value": job_throughput(world, fl, args.steps, e2e_total), "unit": "TFLOP/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "gpu_launches": 2 * args.steps,
        "clocks": clk,
    }


# ----------------------------------------------------------------------------- reference arm

def run_reference(args):
    """The FP64 CPU oracle, timed on the host cores; each step is a bounded row sample."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    w = workload_of(args)
    x = synth.make_inputs(w)
    rng = np.random.default_rng(1)
    per_step = max(0.2, min(2.0, 150.0 / max(1, args.steps + args.warmup)))
    nrm = qk_norm_params(args.qk_norm)
    for _ in range(args.warmup):
        oracle_sample(w, x, per_step / 4, rng, qk_norm=nrm)
    vals, secs, rows = [], [], 0
    th = None
    for _ in range(args.steps):
        tfl, dt, n, th = oracle_sample(w, x, per_step, rng, qk_norm=nrm)
        vals.append(tfl)
        secs.append(dt)
        rows += n
    value = statistics.mean(vals)
    return {
        "impl": "reference",
        "metric": METRIC,
        "value": value,
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": statistics.mean(secs) * 1e3,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic",
        "config": {"workload": w.name, "B": w.B, "H": w.H, "L": w.L, "d": w.d, "d_v": w.dv,
                   "maps": w.nmaps, "window": w.window, "qk_norm": nrm is not None},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": th, "kind": "oracle",
                         "sample": f"{rows} query rows over {args.steps} steps (random rows of "
                                   f"{w.B * w.H * w.L}), FP64 C oracle"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--batch", type=int, default=None, help="override the workload's batch size B")
    ap.add_argument("--cpu-budget", type=float, default=12.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--extra-cpu-budget", type=float, default=3.0,
                    help="seconds of oracle work for each extra workload's cpu_baseline")
    ap.add_argument("--headline-only", dest="all_workloads", action="store_false",
                    help="measure the selected workload only (no `workloads` map)")
    ap.add_argument("--qk-norm", action="store_true",
                    help="QK-RMSNorm (FP32, seeded gammas, eps 1e-6) before RoPE: sa_rope_attn_qknorm")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "ours":
        ap.error("--warmup must be >= 3")
    res = run_reference(args) if args.impl == "reference" else run_ours(args)
    if res is not None:
        print(json.dumps(res), flush=True)
    world, _, _ = dist_env()
    if world > 1 and args.impl == "ours":
        import torch.distributed as dist

        dist.destroy_process_group()


if __name__ == "__main__":
    main()
