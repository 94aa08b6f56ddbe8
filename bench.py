"""Benchmark of the row-wise reduce-then-rescale kernels on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--no-suite]

Prints ONE JSON line.  Metric: achieved HBM bandwidth counting minimum bytes
(each input read once, each output written once, gamma once) and its fraction
of the GB300 HBM peak.  A step is one call of the operation over the
workload's whole batch; the default workload is the fused residual-add +
RMSNorm, bf16, 8192 x 4096.  `per_kernel` repeats the measurement for every
named workload (RMSNorm, fused, attention softmax, vocabulary softmax and the
row-length sweep), one dispatcher leaf each.

Inputs are resident in HBM; consecutive steps rotate over enough distinct
input/output sets that no step finds its data in L2 (more than twice the L2
capacity of traffic between two uses of a set).  The K timed steps are
captured once in a CUDA graph before the timed region (`--stream-launches`:
issued one by one instead); device time comes from CUDA events on the
launching stream around one replay.

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(rows are independent: weak scaling, no collective on the data path); the
reported time is the maximum over ranks.

`--impl reference` times the fp64 CPU oracle (the only reference there is)
on bounded samples of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import ctypes
import dataclasses
import glob
import hashlib
import json
import math
import os
import re
import shutil
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "achieved HBM GB/s (min bytes) and % of GB300 HBM peak per kernel, 1 GPU"
NOMINAL_HBM_GBS = 8000.0          # NVIDIA's public per-GPU HBM3e figure for GB300
FALLBACK_HBM_GBS = 6800.0         # used only when no measured peak file exists
DEFAULT_WORKLOAD = "fused_add_rmsnorm_bf16_8192x4096"
OP_CODE = {"rmsnorm": 0, "fused_add_rmsnorm": 1, "softmax": 2, "log_softmax": 3, "logsumexp": 4,
           "layernorm": 5, "topk": 6}
DT = {"f32": torch.float32, "bf16": torch.bfloat16}


# ------------------------------------------------------------------ helpers

def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def aggregate_over_ranks(elapsed_ms: float, units: float, world: int):
    """Max of the per-rank elapsed times and the sum of units over ranks
    (whole-job throughput = sum of units / slowest rank's time)."""
    if world > 1 and torch.distributed.is_initialized():
        dev = "cuda" if torch.distributed.get_backend() == "nccl" else "cpu"
        t = torch.tensor([elapsed_ms], dtype=torch.float64, device=dev)
        u = torch.tensor([units], dtype=torch.float64, device=dev)
        torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
        torch.distributed.all_reduce(u, op=torch.distributed.ReduceOp.SUM)
        return float(t.item()), float(u.item())
    return elapsed_ms, units


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: torch copy, 2 GiB)"
    return FALLBACK_HBM_GBS, "fallback"


CSRC = os.path.join(ROOT, "online_softmax_row_gb300", "csrc")


def kernel_units(w) -> list[str]:
    """The translation units whose kernels a call of workload w can run."""
    d = {"f32": "f", "bf16": "b"}
    if w.op in ("softmax", "log_softmax"):
        return [f"k_softmax_{d[w.in_dtype]}{d[w.out_dtype]}.cu", "k_staged.cu"]
    if w.op == "logsumexp":
        return ["k_lse.cu"]
    if w.op == "topk":
        return ["k_topk.cu"]
    prefix = {"rmsnorm": "k_rms", "fused_add_rmsnorm": "k_fused", "layernorm": "k_ln"}[w.op]
    return [f"{prefix}_{d[w.in_dtype]}.cu"]


def _include_closure(paths):
    seen, todo = set(), [os.path.normpath(p) for p in paths]
    while todo:
        p = todo.pop()
        # kernel sources only: the public C header declares, it compiles no kernel
        if p in seen or not os.path.exists(p) or os.path.dirname(p) != CSRC:
            continue
        seen.add(p)
        for inc in re.findall(r'^#include "([^"]+)"', open(p, encoding="utf-8").read(), re.M):
            todo.append(os.path.normpath(os.path.join(os.path.dirname(p), inc)))
    return sorted(seen)


def source_hash(w) -> str:
    """Hash of the sources the workload's kernels are compiled from (their
    translation units and the kernel headers those include)."""
    h = hashlib.sha256()
    for f in _include_closure([os.path.join(CSRC, u) for u in kernel_units(w)]):
        with open(f, "rb") as fh:
            h.update(os.path.basename(f).encode())
            h.update(fh.read())
    return h.hexdigest()[:12]


def profiled_traffic(w, plan: str):
    """Per-launch DRAM bytes of the workload's kernel from the committed ncu
    summary (profiles/dram_traffic.md), if it was captured on the current
    sources of that kernel and with the same plan; else None."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.md")
    if not os.path.exists(path):
        return None
    want = source_hash(w)
    for line in open(path, encoding="utf-8"):
        cells = [c.strip().strip("`") for c in line.strip().strip("|").split("|")]
        if len(cells) >= 5 and cells[0] == w.name and cells[1] == want and cells[2] == plan:
            try:
                return int(cells[4].replace(",", ""))
            except ValueError:
                return None
    return None


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 200 ms while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        exe = shutil.which("nvidia-smi")
        if exe:
            self.proc = subprocess.Popen([exe, f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                                          "-i", str(self.index), "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        return self

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        if not self.lines:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for l in self.lines:
            c = [x.strip() for x in l.split(",")]
            try:
                sm.append(float(c[1]))
                smax.append(float(c[2]))
                power.append(float(c[3]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, c[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ our arm

def add_outputs(w, s, device):
    """Output tensors of one call of workload w, added to the set s."""
    if w.op in ("softmax", "log_softmax"):
        s["y"] = torch.empty(w.M, w.N, dtype=DT[w.out_dtype], device=device)
    elif w.op == "logsumexp":
        s["y"] = torch.empty(w.M, dtype=torch.float32, device=device)
        s["arg"] = torch.empty(w.M, dtype=torch.int64, device=device)
    elif w.op == "topk":
        s["y"] = torch.empty(w.M, w.k, dtype=torch.float32, device=device)
        s["arg"] = torch.empty(w.M, w.k, dtype=torch.int64, device=device)
        s["probs"] = torch.empty(w.M, w.k, dtype=torch.float32, device=device)
        s["lse"] = torch.empty(w.M, dtype=torch.float32, device=device)
    else:
        s["y"] = torch.empty_like(s["x"])
    return s


def make_sets(w, n_sets, device):
    """n_sets independent input/output sets of workload w, on device.  Many
    small sets (short decode batches) are cut from one generated batch of
    n_sets * M rows, each set its own contiguous rows."""
    sets = []
    if n_sets > 16 and not w.mask:
        big = workloads.make(dataclasses.replace(w, M=w.M * n_sets, shift_rows=w.shift_rows * n_sets),
                             seed=0, device=device)
        for i in range(n_sets):
            s = {k: (v[i * w.M:(i + 1) * w.M] if v.dim() == 2 else v) for k, v in big.items()}
            sets.append(add_outputs(w, s, device))
        return sets
    for i in range(n_sets):
        sets.append(add_outputs(w, dict(workloads.make(w, seed=i, device=device)), device))
    return sets


def n_sets_for(w, l2_bytes):
    per_set = w.min_bytes
    return max(2, math.ceil(2 * l2_bytes / max(per_set, 1)) + 1)


def call(osr, w, s):
    if w.op == "softmax":
        return osr.softmax_rows(s["x"], out=s["y"])
    if w.op == "log_softmax":
        return osr.log_softmax_rows(s["x"], out=s["y"])
    if w.op == "logsumexp":
        lib = osr.library()
        x = s["x"]
        st = lib.osr_row_logsumexp(x.data_ptr(), s["y"].data_ptr(), s["arg"].data_ptr(), w.M, w.N,
                                   1 if x.dtype == torch.bfloat16 else 0,
                                   torch.cuda.current_stream(x.device).cuda_stream)
        if st != 0:
            raise RuntimeError(f"osr_row_logsumexp: status {st}")
        return s["y"]
    if w.op == "topk":
        lib = osr.library()
        x = s["x"]
        st = lib.osr_row_topk(x.data_ptr(), s["y"].data_ptr(), s["arg"].data_ptr(), s["probs"].data_ptr(),
                              s["lse"].data_ptr(), w.M, w.N, w.k, 1 if x.dtype == torch.bfloat16 else 0,
                              torch.cuda.current_stream(x.device).cuda_stream)
        if st != 0:
            raise RuntimeError(f"osr_row_topk: status {st}")
        return s["y"]
    if w.op == "rmsnorm":
        return osr.rmsnorm_fwd(s["x"], s["gamma"], w.eps, out=s["y"])
    if w.op == "layernorm":
        return osr.layernorm_fwd(s["x"], s["gamma"], s["beta"], w.eps, out=s["y"])
    return osr.fused_add_rmsnorm(s["x"], s["residual"], s["gamma"], w.eps, out=s["y"])


def launches_per_call(plan: str, M: int) -> int:
    if plan.startswith("split"):
        b = int(re.search(r"b=(\d+)", plan).group(1))
        return 2 * math.ceil(M / b)
    return 1


def time_graph(osr, w, steps, warmup, device, l2_bytes, replays=21):
    """Device time of `steps` calls captured once in a CUDA graph (rotating
    input sets), replayed `replays` times: the kernels' own time without host
    launch cost.  Returns the per-call milliseconds of every replay (CUDA
    events on the launching stream around each replay) and the step count."""
    sets = make_sets(w, n_sets_for(w, l2_bytes), device)
    steps = max(steps, len(sets))  # every set once: no call finds its inputs in L2
    for i in range(max(warmup, 3)):
        call(osr, w, sets[i % len(sets)])
    torch.cuda.synchronize(device)
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream(device)
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s, capture_error_mode="relaxed"):
            for i in range(steps):
                call(osr, w, sets[i % len(sets)])
    g.replay()
    torch.cuda.synchronize(device)
    cur = torch.cuda.current_stream(device)
    per_call = []
    for _ in range(replays):
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(cur)
        g.replay()
        stop.record(cur)
        torch.cuda.synchronize(device)
        per_call.append(start.elapsed_time(stop) / steps)
    del g, sets
    torch.cuda.empty_cache()
    return per_call, steps


def quantile(v, q):
    """The q-quantile of v (linear between order statistics)."""
    v = sorted(v)
    pos = q * (len(v) - 1)
    lo = int(math.floor(pos))
    hi = min(lo + 1, len(v) - 1)
    return v[lo] + (v[hi] - v[lo]) * (pos - lo)


# The five configurations of the metric: C1 RMSNorm fp32, C2 fused bf16,
# C3 attention softmax fp32, C4 vocabulary softmax bf16 -> fp32, C5 the
# fp32 row-length sweep
BASELINE_CONFIGS = [("C1", "rmsnorm_f32_64x3584"), ("C2", "fused_add_rmsnorm_bf16_8192x4096"),
                    ("C3", "softmax_attn_f32_114688x4096"), ("C4", "softmax_vocab_bf16_f32_64x152064")] + \
    [(f"C5 N={n}", f"softmax_sweep_f32_N{n}") for n in (32, 128, 1024, 4096, 32768, 152064)]


def time_workload(osr, w, steps, warmup, device, l2_bytes, sampler_index=None, sustain_s=0.0,
                  graph=True, replay_warm=True, pre_load=True, post_load=True):
    """Device time of `steps` back-to-back calls (rotating input sets).
    graph: the `steps` calls are captured once in a CUDA graph (outside the
    timed region; launches with programmatic dependent launch become
    programmatic edges) and the timed region is one replay of it, so host
    launch gaps do not count; otherwise they are issued one by one.
    sustain_s: seconds of the same load before the timed region (pre_load)
    and after it (post_load), while the clock sampler runs."""
    sets = make_sets(w, n_sets_for(w, l2_bytes), device)
    stream = torch.cuda.current_stream(device)
    for i in range(max(warmup, 3)):
        call(osr, w, sets[i % len(sets)])
    torch.cuda.synchronize(device)
    g = None
    if graph:
        g = torch.cuda.CUDAGraph()
        cap = torch.cuda.Stream(device)
        with torch.cuda.stream(cap):
            with torch.cuda.graph(g, stream=cap, capture_error_mode="relaxed"):
                for i in range(steps):
                    call(osr, w, sets[i % len(sets)])
        if replay_warm:
            g.replay()
        torch.cuda.synchronize(device)
    sampler = ClockSampler(sampler_index) if sampler_index is not None else None
    clocks = None

    def sustain():
        if sustain_s <= 0:
            return
        t_end = time.time() + sustain_s
        i = 0
        while time.time() < t_end:
            for _ in range(50):
                call(osr, w, sets[i % len(sets)])
                i += 1
            torch.cuda.synchronize(device)

    if sampler:
        sampler.__enter__()
    try:
        if pre_load:
            sustain()  # same load, so the clock samples reflect the timed region
        if torch.distributed.is_initialized():
            torch.distributed.barrier()
        torch.cuda.synchronize(device)
        start = torch.cuda.Event(enable_timing=True)
        stop = torch.cuda.Event(enable_timing=True)
        start.record(stream)
        if g is not None:
            g.replay()
        else:
            for i in range(steps):
                call(osr, w, sets[i % len(sets)])
        stop.record(stream)
        torch.cuda.synchronize(device)
        elapsed_ms = start.elapsed_time(stop)
        if post_load:
            sustain()
    finally:
        if sampler:
            sampler.__exit__(None, None, None)
            clocks = sampler.summary()
    del g, sets
    torch.cuda.empty_cache()
    return elapsed_ms, clocks


def call_abi(lib, w, s, stream):
    """One call of workload w through the C ABI on the buffers of set s
    (pointers only: device or page-locked host memory alike)."""
    P = lambda k: s[k].data_ptr() if k in s and s[k] is not None else None
    dt = 1 if s["x"].dtype == torch.bfloat16 else 0
    odt = 1 if s["y"].dtype == torch.bfloat16 else 0
    eps = ctypes.c_float(w.eps)
    if w.op == "softmax":
        st = lib.osr_softmax_rows(P("x"), P("y"), w.M, w.N, dt, odt, stream)
    elif w.op == "log_softmax":
        st = lib.osr_log_softmax_rows(P("x"), P("y"), w.M, w.N, dt, odt, stream)
    elif w.op == "logsumexp":
        st = lib.osr_row_logsumexp(P("x"), P("y"), P("arg"), w.M, w.N, dt, stream)
    elif w.op == "topk":
        st = lib.osr_row_topk(P("x"), P("y"), P("arg"), P("probs"), P("lse"), w.M, w.N, w.k, dt, stream)
    elif w.op == "rmsnorm":
        st = lib.osr_rmsnorm_fwd(P("x"), P("gamma"), eps, P("y"), w.M, w.N, dt, stream)
    elif w.op == "layernorm":
        st = lib.osr_layernorm_fwd(P("x"), P("gamma"), P("beta"), eps, P("y"), w.M, w.N, dt, stream)
    else:
        st = lib.osr_fused_add_rmsnorm(P("x"), P("residual"), P("gamma"), eps, P("y"), w.M, w.N, dt, stream)
    if st != 0:
        raise RuntimeError(f"{w.op} through the C ABI: status {st}")


def time_e2e(osr, w, steps, warmup, device):
    """Same metric through the C ABI with HOST buffers: inputs and outputs live
    in page-locked host memory and every call's kernels read them from and
    write them to host memory over the host link (NVLink-C2C on GB300), with
    no staging copy; consecutive steps rotate over enough host sets that no
    step finds its data in L2."""
    l2 = torch.cuda.get_device_properties(device).L2_cache_size
    lib = osr.library()
    sets = []
    for i in range(n_sets_for(w, l2)):
        s = {k: v.pin_memory() for k, v in workloads.make(w, seed=i, device="cpu").items()}
        s = add_outputs(w, s, "cpu")
        sets.append({k: v if v.is_pinned() else v.pin_memory() for k, v in s.items()})
    ins = [k for k in ("x", "residual", "gamma", "beta") if k in sets[0]]
    outs = ["y"] + (["residual"] if w.op == "fused_add_rmsnorm" else []) + \
        (["arg"] if w.op in ("logsumexp", "topk") else []) + (["probs", "lse"] if w.op == "topk" else [])
    h2d = sum(sets[0][k].numel() * sets[0][k].element_size() for k in ins)
    d2h = sum(sets[0][k].numel() * sets[0][k].element_size() for k in outs)
    stream = torch.cuda.current_stream(device)
    raw = stream.cuda_stream
    for i in range(max(warmup, 3)):
        call_abi(lib, w, sets[i % len(sets)], raw)
    torch.cuda.synchronize(device)
    start = torch.cuda.Event(enable_timing=True)
    stop = torch.cuda.Event(enable_timing=True)
    start.record(stream)
    for i in range(steps):
        call_abi(lib, w, sets[i % len(sets)], raw)
    stop.record(stream)
    torch.cuda.synchronize(device)
    ms = start.elapsed_time(stop)
    return {"value": round(w.min_bytes * steps / (ms * 1e-3) / 1e9, 3), "unit": "GB/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
            "ms_per_step": round(ms / steps, 5), "host_sets": len(sets),
            "path": "C ABI call on page-locked host buffers: the kernels read the inputs from and "
                    "write the outputs to host memory over NVLink-C2C (no staging copy)"}


def copy_peak(osr, device, gib=2, copy=None):
    """Best of 10 device-to-device copies of `gib` GiB (read + write bytes
    over time), by the library's copy kernel or the runtime's memcpy."""
    copy = copy or osr.bench_copy
    n = gib * (1 << 30)
    a = torch.empty(n, dtype=torch.uint8, device=device)
    b = torch.empty(n, dtype=torch.uint8, device=device)
    a.fill_(1)
    for _ in range(3):
        copy(a, b)
    torch.cuda.synchronize(device)
    best = float("inf")
    for _ in range(10):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        s.record()
        copy(a, b)
        e.record()
        torch.cuda.synchronize(device)
        best = min(best, s.elapsed_time(e))
    del a, b
    torch.cuda.empty_cache()
    return 2 * n / (best * 1e-3) / 1e9


def time_single_calls(osr, w, device, l2_bytes, calls=21):
    """Device-side latency of one call issued alone: CUDA events around each
    of `calls` stream launches on rotating input sets (cold in L2),
    synchronised between calls.  A short GPU spin is queued before each start
    event, so that the host has enqueued the call by the time the GPU reaches
    the event and the figure is the device's, not the host's launch cost;
    returns the per-call microseconds."""
    sets = make_sets(w, n_sets_for(w, l2_bytes), device)
    for i in range(3):
        call(osr, w, sets[i % len(sets)])
    torch.cuda.synchronize(device)
    cur = torch.cuda.current_stream(device)
    us = []
    for i in range(calls):
        s = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        torch.cuda._sleep(200000)  # about 0.1 ms of GPU spin ahead of the timed call
        s.record(cur)
        call(osr, w, sets[(i + 3) % len(sets)])
        e.record(cur)
        torch.cuda.synchronize(device)
        us.append(s.elapsed_time(e) * 1e3)
    del sets
    torch.cuda.empty_cache()
    return us


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo", encoding="utf-8") as f:
            info = f.read()
    except OSError:
        return "unknown"
    m = re.search(r"^model name\s*:\s*(.+)$", info, re.M)
    if m:
        return m.group(1).strip()
    m = re.search(r"^CPU part\s*:\s*(\S+)$", info, re.M)  # Arm: the part number
    if m:
        part = m.group(1).lower()
        return {"0xd4f": "Arm Neoverse V2"}.get(part, f"Arm CPU part {part}")
    return "unknown"


def _oracle_sample(oracle, w, threads, budget_s):
    """Time the oracle with `threads` threads on about budget_s of rows."""
    oracle.set_threads(threads)
    probe = max(1, min(w.M, 4096 // max(1, w.N // 1024) or 1))
    t = _oracle_time(oracle, w, probe)
    per_row = max(t / probe, 1e-7)
    sample = int(max(1, min(w.M, budget_s / per_row)))
    t = _oracle_time(oracle, w, sample)
    return sample, t, w.min_bytes * sample / w.M / t / 1e9


def cpu_baseline_for(w, budget_s=6.0):
    """The oracle, as it stands, on a bounded sample of rows of the same
    workload: on every host core (OpenMP over rows) and on one; value in the
    workload's GB/s (min bytes of the sample)."""
    import oracle
    cores = os.cpu_count() or 1
    sample, t, gbs = _oracle_sample(oracle, w, cores, budget_s)
    s1, t1, gbs1 = _oracle_sample(oracle, w, 1, budget_s)
    oracle.set_threads(1)
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{sample} of {w.M} rows of {w.name} (seed 0), fp64 C oracle, {cores} threads, "
                      f"{t:.2f} s",
            "seconds": round(t, 3), "nproc": cores, "cpu_model": cpu_model(),
            "single_thread": {"value": round(gbs1, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{s1} of {w.M} rows, {t1:.2f} s"}}


def _oracle_inputs(w, rows):
    """Oracle-format inputs (float32, or uint16 bf16 bits) for the first rows."""
    if w.op in ("softmax", "log_softmax", "logsumexp", "topk"):
        inp = workloads.softmax_inputs(rows, w.N, w.in_dtype, w.sigma, 0, w.shift, w.spikes_per_row,
                                       w.spike, seed=0, mask=w.mask)
    elif w.op == "layernorm":
        inp = workloads.layernorm_inputs(rows, w.N, w.in_dtype, w.sigma, w.low, w.high, seed=0)
    else:
        inp = workloads.rmsnorm_inputs(rows, w.N, w.in_dtype, w.sigma, w.op == "fused_add_rmsnorm", seed=0)
    out = {}
    for k, v in inp.items():
        v = v.contiguous()
        out[k] = v.view(torch.int16).numpy().view(np.uint16) if v.dtype == torch.bfloat16 else v.numpy()
    return out


def _run_oracle(oracle, w, inp):
    if w.op == "softmax":
        y = oracle.softmax(inp["x"])
        return oracle.round_to(y, w.out_dtype)
    if w.op == "log_softmax":
        return oracle.round_to(oracle.log_softmax(inp["x"]), w.out_dtype)
    if w.op == "logsumexp":
        return oracle.logsumexp_argmax(inp["x"])
    if w.op == "topk":
        return oracle.topk(inp["x"], w.k)
    if w.op == "rmsnorm":
        y = oracle.rmsnorm(inp["x"], inp["gamma"], w.eps)
        return oracle.round_to(y, w.out_dtype)
    if w.op == "layernorm":
        return oracle.round_to(oracle.layernorm(inp["x"], inp["gamma"], inp["beta"], w.eps), w.out_dtype)
    h, y = oracle.fused_add_rmsnorm(inp["x"], inp["residual"], inp["gamma"], w.eps)
    return oracle.round_to(h, w.out_dtype), oracle.round_to(y, w.out_dtype)


def _oracle_time(oracle, w, rows):
    inp = _oracle_inputs(w, rows)
    t0 = time.perf_counter()
    _run_oracle(oracle, w, inp)
    return time.perf_counter() - t0


def ours(args):
    import online_softmax_row_gb300 as osr
    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local))
    device = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(device)
    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    peak, peak_src = measured_peaks()
    w = workloads.WORKLOADS[args.workload]
    capped = bool(args.max_rows and w.M > args.max_rows)
    if capped:
        # profiling a smaller case of the same kernel (same row length, plan
        # and per-row work): traffic then scales by rows
        w = dataclasses.replace(w, M=args.max_rows,
                                shift_rows=round(w.shift_rows * args.max_rows / w.M))
    osr.library()
    plan = osr.plan_describe(OP_CODE[w.op], w.M, w.N, w.in_dtype, w.out_dtype, True,
                             props.multi_processor_count)

    # The K steps are timed right after the warm-up, as the burst copy peak
    # they are compared with is (a kernel timed alone); the clock sampler
    # runs across them and 1.5 s of the same load after them.  `sustained`
    # repeats the timing after 1.5 s of the same load: the GPU warms, and
    # on some boxes that costs the short region up to 3 % at unchanged SM
    # clocks.
    elapsed_ms, clocks = time_workload(osr, w, args.steps, args.warmup, device, l2,
                                       sampler_index=None if args.profile else device.index,
                                       sustain_s=0.0 if args.profile else 1.5,
                                       graph=not args.stream_launches, replay_warm=not args.profile,
                                       pre_load=False)
    sustained = None
    if not args.profile:
        sus_ms, _ = time_workload(osr, w, args.steps, args.warmup, device, l2, sampler_index=None,
                                  sustain_s=1.5, graph=not args.stream_launches, pre_load=True,
                                  post_load=False)
        sus_ms, sus_bytes = aggregate_over_ranks(sus_ms, w.min_bytes * args.steps, world)
        sustained = {"value": round(sus_bytes / (sus_ms * 1e-3) / 1e9, 3), "unit": "GB/s",
                     "ms_per_step": round(sus_ms / args.steps, 5),
                     "frac": round(sus_bytes / world / (sus_ms * 1e-3) / 1e9 / peak, 4),
                     "timing": "the same steps after 1.5 s of the same load"}
    max_ms, total_bytes = aggregate_over_ranks(elapsed_ms, w.min_bytes * args.steps, world)
    value = total_bytes / (max_ms * 1e-3) / 1e9
    per_launch_ms = elapsed_ms / args.steps / launches_per_call(plan, w.M)
    achieved = w.min_bytes / launches_per_call(plan, w.M) / (per_launch_ms * 1e-3) / 1e9

    result = {
        "metric": METRIC, "value": round(value, 3), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        # the arithmetic type: every kernel computes in binary32 (bf16 inputs
        # are widened exactly); the storage types are in_dtype / out_dtype
        "dtype": "f32", "data": "synthetic",
        "config": {"workload": w.name, "op": w.op, "M": w.M, "N": w.N, "in_dtype": w.in_dtype,
                   "out_dtype": w.out_dtype, "min_bytes_per_step": w.min_bytes, "kernel": plan,
                   "rows_capped": capped,
                   "timing": ("the steps issued one by one on the stream" if args.stream_launches else
                              "CUDA graph of the steps (programmatic dependent launch edges), captured "
                              "before the timed region; CUDA events around one replay"),
                   "l2": f"rotating {n_sets_for(w, l2)} input/output sets (> 2x L2 of traffic "
                         f"between reuses); no flush", "parallelism": f"rows; {world} GPU(s), weak"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                     # the committed captures are of the full-size workloads
                     "frac": round(achieved / peak, 4), "traffic": None if capped else profiled_traffic(w, plan),
                     "kernel_source_hash": source_hash(w),
                     "peak_source": peak_src + " -- of measured" if "measured" in peak_src else peak_src,
                     "algorithmic_bytes_per_launch": w.min_bytes // launches_per_call(plan, w.M)},
        "gpu_launches": args.steps * launches_per_call(plan, w.M),
        "clocks": clocks,
    }
    if sustained is not None:
        result["sustained"] = sustained
    if rank == 0 and not (args.no_suite or args.profile):
        ck = copy_peak(osr, device)
        mc = copy_peak(osr, device, copy=osr.bench_memcpy)
        result["peaks"] = {"nominal_gbs": NOMINAL_HBM_GBS, "driver_measured_gbs": peak,
                           "copy_kernel_same_run_gbs": round(ck, 1), "memcpy_d2d_same_run_gbs": round(mc, 1),
                           "copy_max_same_run_gbs": round(max(ck, mc), 1)}
        copy_gbs = result["peaks"]["copy_max_same_run_gbs"]
        suite = []
        for name, wl in workloads.WORKLOADS.items():
            steps = max(20, min(2000, int(1e10 / max(wl.min_bytes, 1))))
            per_call, steps = time_graph(osr, wl, steps, 5, device, l2)
            p = osr.plan_describe(OP_CODE[wl.op], wl.M, wl.N, wl.in_dtype, wl.out_dtype, True,
                                  props.multi_processor_count)
            us = [t * 1e3 for t in per_call]
            med = statistics.median(us)
            g = wl.min_bytes / (med * 1e-6) / 1e9
            suite.append({"workload": name, "kernel": p, "min_bytes": wl.min_bytes, "steps": steps,
                          "us_per_call": round(med, 3), "us_p10": round(quantile(us, 0.1), 3),
                          "us_p90": round(quantile(us, 0.9), 3), "replays": len(us), "gbs": round(g, 1),
                          "frac_measured": round(g / peak, 4), "frac_nominal": round(g / NOMINAL_HBM_GBS, 4),
                          "frac_copy_same_run": round(g / copy_gbs, 4),
                          "launches_per_call": launches_per_call(p, wl.M),
                          "traffic": profiled_traffic(wl, p)})
            if wl.min_bytes < (64 << 20):
                # small calls are latency-bound: one call issued alone as well
                lat = time_single_calls(osr, wl, device, l2)
                suite[-1]["latency_us"] = round(statistics.median(lat), 3)
        result["per_kernel"] = suite
        result["per_kernel_timing"] = ("per workload: CUDA graph of the steps over rotating sets, "
                                       "replayed 21 times with CUDA events around each replay; "
                                       "median and p10/p90 of the per-call time")
        by_name = {e["workload"]: e for e in suite}
        baseline_configs = {}
        for tag, name in BASELINE_CONFIGS:
            e = by_name[name]
            baseline_configs[tag] = {"us": e["us_per_call"], "p10": e["us_p10"], "p90": e["us_p90"],
                                     "gbs": e["gbs"], "frac": e["frac_measured"],
                                     "frac_copy": e["frac_copy_same_run"], "traffic": e["traffic"]}
            if "latency_us" in e:
                baseline_configs[tag]["latency_us"] = e["latency_us"]
    if rank == 0:
        if not args.profile:
            result["e2e"] = time_e2e(osr, w, max(3, min(args.steps, 50)), args.warmup, device)
            result["cpu_baseline"] = cpu_baseline_for(w)
        if not (args.no_suite or args.profile):
            # last, and compact, so that a reader keeping only the end of the
            # line still sees every configuration of the metric: median us
            # over 21 graph replays, p10/p90, GB/s, fraction of the measured
            # peak and of the copy kernel in this run, ncu DRAM bytes
            result["baseline_configs"] = baseline_configs
        print(json.dumps(result), flush=True)
    if world > 1:
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


# ------------------------------------------------------------------ reference arm

def reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)  # OpenMP over rows, every host core
    w = workloads.WORKLOADS[args.workload]
    # each step: a bounded sample of rows of the same workload
    rows = max(1, min(w.M, int(8_000_000 // max(w.N, 1))))
    inp = _oracle_inputs(w, rows)
    for _ in range(max(args.warmup, 0)):
        _run_oracle(oracle, w, inp)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _run_oracle(oracle, w, inp)
    dt = time.perf_counter() - t0
    sample_bytes = w.min_bytes * rows / w.M
    value = sample_bytes * args.steps / dt / 1e9
    sample = f"{rows} of {w.M} rows of {w.name} per step (seed 0), fp64 C oracle, {cores} threads"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "op": w.op, "M": w.M, "N": w.N, "in_dtype": w.in_dtype,
                   "out_dtype": w.out_dtype, "sample_rows_per_step": rows},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.get_threads(),
                         "kind": "oracle", "sample": sample, "nproc": cores, "cpu_model": cpu_model()},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=list(workloads.WORKLOADS))
    ap.add_argument("--no-suite", action="store_true", help="skip the per-workload table")
    ap.add_argument("--stream-launches", action="store_true",
                    help="time the steps launched one by one instead of one graph replay")
    ap.add_argument("--profile", action="store_true",
                    help="only the timed steps of the workload (for ncu captures): no clock "
                         "sampling, per-workload table, e2e or CPU baseline")
    ap.add_argument("--max-rows", type=int, default=0,
                    help="with --profile: run only the first MAX_ROWS rows of the workload "
                         "(a capture-sized case of the same kernel)")
    args = ap.parse_args(argv)
    if args.max_rows and not args.profile:
        ap.error("--max-rows is for profiling captures only (--profile)")
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
