"""Benchmark of the fused gated group-RMSNorm on GB300.

Prints ONE JSON line (rank 0).  A step is one call of the whole operation
(validate, select, one kernel: load y/gate, gate, group reduction,
normaliser, epilogue, store) over one batch of synthetic input.  Default
workload: the largest prefill shape that one GPU holds, the strided odd span
(65536 rows x 4800, groups of 100, bf16, y and gate column slices of a packed
[65536, 9664] in-proj output).

  value        algorithmic HBM GB/s (y + gate read once, out written once, the
               weight once) / device time of the K timed steps, summed over ranks
  per_config   the other prefill workloads, each timed the same way in its own
               window (max(K, 50) steps), with its roofline and clocks
  e2e          the same metric through the public Python API with pinned HOST
               buffers, every byte crossing the host link inside the timed region
  roofline     the kernel's achieved GB/s against the measured HBM copy peak;
               traffic = DRAM bytes per launch from the ncu range capture
               recorded in profiles/dram_traffic.txt (null when the kernels
               changed since)
  clocks       SM clock, power and clock-event reasons sampled in process
               (NVML, read-only) during each timed region
  cpu_baseline the single-threaded CPU oracle on a bounded sample

Timing: W warm-up steps, then K steps between two CUDA events on the
launching stream with a barrier and a synchronize on both sides, max over
ranks.  Inputs rotate over several copies whose total exceeds the L2, so
every step reads y and gate from HBM.

--impl reference times the CPU oracle instead (the reference arm of this
build): same metric and workload, each step a bounded sample of rows.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import ggrn_inputs  # noqa: E402

METRIC = "achieved HBM GB/s (% of GB300 peak) and rows/s; decode µs/call"
UNIT = "GB/s"
L2_BYTES = 129 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.txt")
CSRC = os.path.join(ROOT, "gated_group_rmsnorm_gb300", "csrc")
IO_DTYPE = {torch.bfloat16: "bf16", torch.float16: "f16", torch.float32: "f32"}


# ---------------------------------------------------------------------------
# Multi-rank plumbing (host logic; tested with gloo ranks on CPU).
# ---------------------------------------------------------------------------
def dist_env() -> tuple[int, int, int]:
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def reduce_max(value: float, device) -> float:
    """Max of a float over all ranks (identity without a process group)."""
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier() -> None:
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


def aggregate(bytes_per_step: int, rows_per_step: int, steps: int, max_ms: float,
              world: int) -> dict:
    """Whole-job throughput: units all ranks processed / the slowest rank's time."""
    secs = max_ms / 1e3
    return {"gbs": world * steps * bytes_per_step / secs / 1e9,
            "rows_per_s": world * steps * rows_per_step / secs,
            "ms_per_step": max_ms / steps}


# ---------------------------------------------------------------------------
# Clock sampling during the timed region.
# ---------------------------------------------------------------------------
class ClockSampler:
    """SM clock, power and clock-event reasons sampled in this process through
    NVML's read-only queries, about every millisecond, so that even a timed
    region of a fraction of a millisecond has samples around it.  Nothing is
    ever set: only nvmlDeviceGet* calls are made."""
    # clock-event reason bits of the NVML header
    REASONS = {0x8: "hw_slowdown", 0x40: "hw_thermal_slowdown", 0x20: "sw_thermal_slowdown",
               0x4: "sw_power_cap", 0x80: "hw_power_brake_slowdown"}
    NVML_CLOCK_SM = 1

    def __init__(self, uuid: str, period_s: float = 0.001):
        self.samples: list[tuple[float, int, int, int]] = []  # (time, sm MHz, reasons, mW)
        self.max_mhz = None
        self.error = None
        self._stop = threading.Event()
        self.thread = None
        try:
            L = ctypes.CDLL("libnvidia-ml.so.1")
            if L.nvmlInit_v2() != 0:
                raise OSError("nvmlInit_v2 failed")
            h = ctypes.c_void_p()
            u = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if L.nvmlDeviceGetHandleByUUID(u.encode(), ctypes.byref(h)) != 0:
                raise OSError(f"no NVML device with uuid {u}")
            mx = ctypes.c_uint()
            if L.nvmlDeviceGetMaxClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = mx.value
            self.L, self.h = L, h
        except (OSError, AttributeError) as e:
            self.error = str(e)
            return
        self.period = period_s
        self.thread = threading.Thread(target=self._run, daemon=True)
        self.thread.start()

    def _run(self):
        L, h = self.L, self.h
        mhz, rs, mw = ctypes.c_uint(), ctypes.c_ulonglong(), ctypes.c_uint()
        while not self._stop.is_set():
            ok = L.nvmlDeviceGetClockInfo(h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) == 0
            if ok and L.nvmlDeviceGetCurrentClocksEventReasons(h, ctypes.byref(rs)) != 0:
                rs.value = 0
            if L.nvmlDeviceGetPowerUsage(h, ctypes.byref(mw)) != 0:
                mw.value = 0
            if ok:
                self.samples.append((time.perf_counter(), mhz.value, rs.value, mw.value))
            time.sleep(self.period)

    def stop(self):
        self._stop.set()
        if self.thread is not None:
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float) -> dict:
        """Samples taken while the timed region ran (host clock, perf_counter);
        for a region shorter than a few sampling periods, the samples of the
        2 ms either side of it as well."""
        if self.error is not None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0,
                    "window": f"none (NVML unavailable: {self.error})"}
        win = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed region"
        if len(win) < 3:
            win = [s for s in self.samples if t0 - 0.002 <= s[0] <= t1 + 0.002]
            window = "timed region +-2 ms"
        if not win:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": [], "samples": 0,
                    "window": window}
        reasons = sorted({name for _, _, r, _ in win for bit, name in self.REASONS.items()
                          if r & bit})
        return {"sm_mhz": statistics.median(m for _, m, _, _ in win),
                "sm_min_mhz": min(m for _, m, _, _ in win),
                "sm_max_mhz": self.max_mhz,
                "power_w_max": round(max(p for _, _, _, p in win) / 1000.0, 1),
                "reasons": reasons, "samples": len(win), "window": window,
                "source": "NVML queries in the bench process, ~1 ms apart"}


# ---------------------------------------------------------------------------
# Roofline denominators and recorded ncu traffic.
# ---------------------------------------------------------------------------
def hbm_peak() -> tuple[float, str]:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            return float(json.load(fh)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    """Hash of the sources that define the norm kernels and how a call
    launches them (the host pipeline, ggrn_host.cu, only sequences copies
    around those launches, and ggrn_outproj.cu holds the separate fused
    out_proj kernels: both are left out)."""
    h = hashlib.sha256()
    for fn in sorted(os.listdir(CSRC)):
        if fn.endswith((".cu", ".cuh", ".h")) and fn not in ("ggrn_host.cu", "ggrn_outproj.cu"):
            with open(os.path.join(CSRC, fn), "rb") as fh:
                h.update(fn.encode() + b"\0" + _without_timeline(fh.read()))
    return h.hexdigest()[:16]


def _without_timeline(src: bytes) -> bytes:
    """The source as the product library compiles it: the blocks compiled
    only into the profiling build (#ifdef GGRN_TIMELINE ... #endif, not
    nested) are dropped."""
    out, skip = [], False
    for line in src.split(b"\n"):
        if line.strip() == b"#ifdef GGRN_TIMELINE":
            skip = True
        elif skip and line.strip() == b"#endif":
            skip = False
        elif not skip:
            out.append(line)
    return b"\n".join(out)


def recorded_traffic(workload: str) -> tuple[float | None, str]:
    """DRAM bytes per launch from profiles/dram_traffic.txt, if it was captured
    on the current kernel sources (else None)."""
    if not os.path.exists(TRAFFIC_FILE):
        return None, "no capture recorded"
    cur = kernel_source_hash()
    found = None
    with open(TRAFFIC_FILE) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if kv.get("workload") == workload:
                found = kv
    if found is None:
        return None, "no capture for this workload"
    if found.get("csrc_sha") != cur:
        return None, f"kernels changed since the capture ({found.get('csrc_sha')} != {cur})"
    return float(found["dram_bytes_per_launch"]), found.get("note", "ncu capture")


def recorded_ncu_gbs(workload: str) -> float | None:
    """(DRAM read + write bytes) / duration of the recorded ncu capture of the
    workload's kernel (one cold launch), if taken on the current sources."""
    if recorded_traffic(workload)[0] is None:
        return None
    with open(TRAFFIC_FILE) as fh:
        for line in fh:
            kv = dict(tok.split("=", 1) for tok in line.split() if "=" in tok)
            if kv.get("workload") == workload and "ncu_gbs" in kv:
                return float(kv["ncu_gbs"])
    return None


# ---------------------------------------------------------------------------
# Our arm.
# ---------------------------------------------------------------------------
def _raw_args(g, inp, out, wl, stream_handle):
    """Pre-marshalled C-ABI arguments of one step (the timed loop then only
    crosses ctypes once per step)."""
    from gated_group_rmsnorm_gb300 import binding
    width = wl.width
    rows, ys = binding._as_rows(inp.y, width, "y")
    _, gts = binding._as_rows(inp.gate, width, "gate")
    _, os_ = binding._as_rows(out, width, "out")
    return (inp.y.data_ptr(), inp.gate.data_ptr(), inp.w.data_ptr(), out.data_ptr(), rows, width,
            wl.group_size, ys, gts, os_, ctypes.c_float(wl.eps), binding.DTYPE_CODE[wl.dtype],
            wl.mode, stream_handle)


def _decode_numbers(g, device) -> dict:
    """µs per call of the batch-1 decode shape: eager, a 1-call graph, a 21-call
    graph (one Mamba-2 norm per layer of a 21-layer decode step)."""
    wl = ggrn_inputs.WORKLOADS["mamba2_decode"]
    layers = [ggrn_inputs.make_inputs(wl, device=device, seed=100 + i) for i in range(21)]
    outs = [torch.empty_like(l.y) for l in layers]
    stream = torch.cuda.current_stream(device)
    L = g.load()
    handle = ctypes.c_void_p(stream.cuda_stream)
    args = [_raw_args(g, l, o, wl, handle) for l, o in zip(layers, outs)]
    n_calls = 2100

    def timed(fn, n):
        for _ in range(50):
            fn()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        wall = time.perf_counter() - t0
        return e0.elapsed_time(e1) * 1e3, wall * 1e6

    i = [0]

    def eager():
        st = L.ggrn_forward(*args[i[0] % 21])
        i[0] += 1
        assert st == 0
    dev_us, wall_us = timed(eager, n_calls)
    g1 = g.DecodeGraph([dict(y=layers[0].y, gate=layers[0].gate, w=layers[0].w, out=outs[0],
                             group_size=wl.group_size, eps=wl.eps)])
    g21 = g.DecodeGraph([dict(y=l.y, gate=l.gate, w=l.w, out=o, group_size=wl.group_size,
                              eps=wl.eps) for l, o in zip(layers, outs)])
    g1_dev, g1_wall = timed(lambda: g1.replay(stream), n_calls)
    g21_dev, g21_wall = timed(lambda: g21.replay(stream), n_calls // 21)
    g1.close()
    g21.close()
    # the same step of a norm whose row is one 7680-wide group (a cluster of
    # CTAs per group): 21 calls in one graph
    lone = []
    for i in range(21):
        inp = ggrn_inputs.random_case(1, 7680, 7680, torch.bfloat16, 0, seed=300 + i)
        lone.append((inp.y.to(device), inp.gate.to(device), inp.w.to(device),
                     torch.empty((1, 7680), dtype=torch.bfloat16, device=device)))
    plan_lone = g.plan(lone[0][0], lone[0][1], lone[0][2], group_size=7680)
    gl = g.DecodeGraph([dict(y=y, gate=gt, w=w, out=o, group_size=7680, eps=1e-5)
                        for y, gt, w, o in lone])
    gl_dev, gl_wall = timed(lambda: gl.replay(stream), n_calls // 21)
    gl.close()
    return {"workload": "mamba2_decode (1 x 7680, groups of 960, bf16)",
            "eager_us_per_call": round(max(dev_us, wall_us) / n_calls, 3),
            "graph1_us_per_call": round(max(g1_dev, g1_wall) / n_calls, 3),
            "graph21_us_per_call": round(max(g21_dev, g21_wall) / (21 * (n_calls // 21)), 3),
            "lone_group_7680_graph21_us_per_call":
                round(max(gl_dev, gl_wall) / (21 * (n_calls // 21)), 3),
            "lone_group_path": plan_lone["path_name"],
            "note": "max(device time, host wall time) per call over back-to-back calls; "
                    "DecodeGraph of one call launches it directly (a graph of one small "
                    "kernel costs more to launch than the kernel)"}


def _outproj_numbers(g, device, steps: int, d_models=(3840, 7680)) -> dict:
    """The norm fused into the out_proj GEMM (ggrn_norm_outproj) on the
    Mamba-2 prefill shape, against the same two steps unfused: the norm
    kernel (ggrn_forward) then torch.matmul (cuBLAS) on its output; and the
    GEMM alone.  µs per step from CUDA events over `steps` back-to-back
    steps after warm-up; TFLOP/s = 2 M N K / time."""
    wl = ggrn_inputs.WORKLOADS["mamba2_prefill"]
    inp = ggrn_inputs.make_inputs(wl, device=device)
    out = {}
    for d_model in d_models:
        w_out = ggrn_inputs.make_outproj_weight(d_model, wl.width, device=device, seed=1)
        z = torch.empty((wl.rows, d_model), dtype=torch.bfloat16, device=device)
        ws = torch.empty(max(16, g.load().ggrn_norm_outproj_workspace_bytes(
            wl.rows, wl.width, wl.group_size)), dtype=torch.uint8, device=device)
        a = torch.empty((wl.rows, wl.width), dtype=torch.bfloat16, device=device)

        def fused():
            g.norm_outproj(inp.y, inp.gate, inp.w, w_out, group_size=wl.group_size, eps=wl.eps,
                           out=z, workspace=ws)

        def unfused():
            g.forward(inp.y, inp.gate, inp.w, group_size=wl.group_size, eps=wl.eps, out=a)
            torch.matmul(a, w_out.T, out=z)

        def gemm_only():
            torch.matmul(a, w_out.T, out=z)

        res = {}
        for name, fn in (("fused", fused), ("unfused_norm_then_cublas", unfused),
                         ("cublas_gemm_only", gemm_only)):
            for _ in range(5):
                fn()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            for _ in range(steps):
                fn()
            e1.record()
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) * 1e3 / steps
            res[name] = {"us": round(us, 2),
                         "tflops": round(2.0 * wl.rows * d_model * wl.width / us / 1e6, 1)}
        res["fused_vs_unfused"] = round(res["unfused_norm_then_cublas"]["us"] / res["fused"]["us"],
                                        3)
        out[f"d_model_{d_model}"] = res
        del w_out, z, ws, a
    return {"workload": "mamba2_prefill (4096 x 7680, groups of 960) -> out_proj [d_model, 7680], "
                        "bf16, f32 sums", "steps": steps, **out}


def _cpu_baseline(wl, budget_s: float = 10.0) -> dict:
    """The single-threaded oracle on host cores: sample rows of the workload,
    repeated until the budget is spent."""
    import oracle
    sample_rows = min(wl.rows, 256)
    swl = wl.with_rows(sample_rows)
    inp = ggrn_inputs.make_inputs(swl)
    orc = oracle.default()
    out = torch.empty((sample_rows, wl.width), dtype=wl.dtype)
    reps = 0
    t0 = time.perf_counter()
    while True:
        orc.forward(inp.y, inp.gate, inp.w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode,
                    out=out)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    bytes_ = swl.algorithmic_bytes() * reps
    return {"value": round(bytes_ / el / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "rows_per_s": round(sample_rows * reps / el, 1),
            "sample": f"{sample_rows} rows of {wl.name} (same recipe), {reps} passes, {el:.1f} s, "
                      f"single-threaded C++ oracle"}


def _cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.startswith("Model name:"):
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    try:
        with open("/proc/cpuinfo") as fh:
            for line in fh:
                if line.lower().startswith("model name"):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def _cpu_baseline_all_cores(wl, budget_s: float = 5.0) -> dict:
    """The same per-row oracle code on every host core: one thread per core,
    each running the single-threaded oracle over its own block of sample rows
    until the budget is spent (the oracle's C call releases the GIL)."""
    import concurrent.futures
    import oracle
    threads = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    per = max(1, min(64, wl.rows // threads))
    swl = wl.with_rows(per * threads)
    inp = ggrn_inputs.make_inputs(swl)
    out = torch.empty((swl.rows, wl.width), dtype=wl.dtype)
    orc = oracle.default()
    deadline = time.perf_counter() + budget_s

    def work(t):
        sl = slice(t * per, (t + 1) * per)
        reps = 0
        while True:
            orc.forward(inp.y[sl], inp.gate[sl], inp.w, group_size=wl.group_size, eps=wl.eps,
                        mode=wl.mode, out=out[sl])
            reps += 1
            if time.perf_counter() >= deadline:
                return reps

    t0 = time.perf_counter()
    with concurrent.futures.ThreadPoolExecutor(threads) as ex:
        reps = list(ex.map(work, range(threads)))
    el = time.perf_counter() - t0
    bytes_ = wl.with_rows(per).algorithmic_bytes() * sum(reps)
    return {"value": round(bytes_ / el / 1e9, 4), "unit": UNIT, "cores": threads,
            "kind": "oracle", "rows_per_s": round(per * sum(reps) / el, 1),
            "cpu_model": _cpu_model(), "hardware_threads": os.cpu_count(),
            "sample": f"{threads} threads x {per} rows of {wl.name} (same recipe), "
                      f"{sum(reps)} passes in all, {el:.1f} s, the single-threaded C++ oracle "
                      f"per thread"}


def _e2e(g, wl, steps: int, device) -> dict:
    """Public API with pinned host buffers: every step is one forward_host
    call (host y and gate in, host out back), timed between events on the
    stream.  For pinned buffers the library's kernel reads y and gate and
    writes out in place over the host link, so every byte of the step
    crosses the link inside the timed region."""
    host = ggrn_inputs.make_inputs(wl, device=device)
    width = wl.width
    if host.packed is not None:
        packed_h = host.packed.cpu().pin_memory()
        y_h, g_h = packed_h[:, :width], packed_h[:, width:2 * width]
    else:
        y_h, g_h = host.y.cpu().pin_memory(), host.gate.cpu().pin_memory()
    w_d = host.w
    out_h = torch.empty((wl.rows, width), dtype=wl.dtype).pin_memory()
    stream = torch.cuda.current_stream(device)

    def step():
        g.forward_host(y_h, g_h, w_d, group_size=wl.group_size, eps=wl.eps, mode=wl.mode,
                       out=out_h)
    for _ in range(5):
        step()
    torch.cuda.synchronize()
    # three timed windows of `steps` steps; the median is reported (the host
    # link shows occasional transients of a few tens of ms from outside this
    # process), all three are listed
    windows = []
    for _ in range(3):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        windows.append(e0.elapsed_time(e1))
    ms = sorted(windows)[1]
    es = out_h.element_size()
    h2d_bytes = 2 * wl.rows * width * es   # the y and gate columns of every row
    d2h_bytes = wl.rows * width * es
    return {"value": round(wl.algorithmic_bytes() * steps / (ms / 1e3) / 1e9, 2), "unit": UNIT,
            "h2d_bytes_per_step": h2d_bytes, "d2h_bytes_per_step": d2h_bytes, "steps": steps,
            "ms_per_step": round(ms / steps, 4),
            "windows_gbs": [round(wl.algorithmic_bytes() * steps / (t / 1e3) / 1e9, 2)
                            for t in windows],
            "api": "forward_host (ggrn_forward_host: pinned y, gate and out are read and "
                   "written in place by one kernel over the host link)"}


def unfused_chain_fn(wl):
    """Context, not a product path: the operation as separate PyTorch ops on
    the GPU, the multi-dispatch chain a fused kernel replaces (widen, y *
    silu(gate), per-group mean of squares and rsqrt, normalise and cast,
    weight and cast; ONNX: the normalised X times scale and silu(gate))."""
    import torch.nn.functional as F
    rows, width, gs = wl.rows, wl.width, wl.group_size

    def chain(inp):
        yf, gf = inp.y.float(), inp.gate.float()
        if wl.mode == 0:
            gated = (yf * F.silu(gf)).view(rows, width // gs, gs)
            nf = torch.rsqrt(gated.pow(2).mean(-1, keepdim=True) + wl.eps)
            t = (gated * nf).to(wl.dtype).view(rows, width)
            return (inp.w * t.float()).to(wl.dtype)
        x = yf.view(rows, width // gs, gs)
        nf = torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + wl.eps)
        r = (x * nf).view(rows, width) * inp.w.float().repeat(width // gs) * F.silu(gf)
        return r.to(wl.dtype)
    return chain


def _unfused_chain(wl, sets, steps: int) -> dict:
    """The unfused chain timed like the fused launch, on the same rotating inputs."""
    chain = unfused_chain_fn(wl)
    for i in range(3):
        chain(sets[i % len(sets)])
    torch.cuda.synchronize()
    ops = None
    try:  # dispatched ATen ops that are not views: one GPU kernel each here
        from torch.utils._python_dispatch import TorchDispatchMode

        class _Count(TorchDispatchMode):
            n = 0

            def __torch_dispatch__(self, func, types, args=(), kwargs=None):
                if not getattr(func, "is_view", False):
                    _Count.n += 1
                return func(*args, **(kwargs or {}))
        with _Count():
            chain(sets[0])
        ops = _Count.n
    except Exception:  # the count is optional context
        ops = None
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    for i in range(steps):
        chain(sets[i % len(sets)])
    e1.record()
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": round(wl.algorithmic_bytes() / (ms / 1e3) / 1e9, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps, "aten_ops_per_step": ops,
            "note": "the operation as separate PyTorch GPU ops (unfused chain), same "
                    "algorithmic bytes and inputs; context for the single fused launch"}


def _time_workload(g, L, wl, steps: int, warmup: int, device, sampler) -> dict:
    """W untimed steps, then exactly K steps of one workload between CUDA events
    on the launching stream, barrier + synchronize on both sides; inputs
    rotate over copies whose total exceeds the L2.  Returns the measurement
    (max over ranks) with the plan and the clock samples of the region."""
    bytes_per_step = wl.algorithmic_bytes()
    n_sets = max(2, -(-4 * L2_BYTES // bytes_per_step))
    sets = [ggrn_inputs.make_inputs(wl, device=device, seed=s) for s in range(n_sets)]
    outs = [torch.empty((wl.rows, wl.width), dtype=wl.dtype, device=device) for _ in range(n_sets)]
    stream = torch.cuda.current_stream(device)
    handle = ctypes.c_void_p(stream.cuda_stream)
    raw = [_raw_args(g, st, o, wl, handle) for st, o in zip(sets, outs)]
    plan = g.plan(sets[0].y, sets[0].gate, sets[0].w, group_size=wl.group_size, mode=wl.mode,
                  out=outs[0])
    for i in range(warmup):
        st = L.ggrn_forward(*raw[i % n_sets])
        if st != 0:
            raise RuntimeError(f"ggrn_forward: {g.status_string(st)}")
    torch.cuda.synchronize()
    barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_start = time.perf_counter()
    e0.record(stream)
    for i in range(steps):
        L.ggrn_forward(*raw[i % n_sets])
    e1.record(stream)
    torch.cuda.synchronize()
    t_end = time.perf_counter()
    barrier()
    ms = e0.elapsed_time(e1)
    max_ms = reduce_max(ms, device)
    res = {"ms": ms, "max_ms": max_ms, "plan": plan, "n_sets": n_sets,
           "bytes_per_step": bytes_per_step, "clocks": sampler.summary(t_start, t_end),
           "sets": sets}
    del outs, raw
    return res


def _roofline(wl, kernel_gbs: float) -> dict:
    peak, peak_src = hbm_peak()
    traffic, traffic_note = recorded_traffic(wl.name)
    return {"bound": "hbm", "achieved": round(kernel_gbs, 2), "peak": peak, "unit": "GB/s",
            "frac": round(kernel_gbs / peak, 4), "traffic": traffic, "peak_source": peak_src,
            "algorithmic_bytes_per_launch": wl.algorithmic_bytes(),
            "traffic_note": traffic_note,
            "ncu_dram_gbs": recorded_ncu_gbs(wl.name),
            "ncu_dram_gbs_note": "DRAM read+write bytes over the duration of a range of "
                                 "back-to-back launches under ncu (profiles/dram_traffic.txt)"}


def _config(wl, m) -> dict:
    plan = m["plan"]
    return {"workload": wl.name, "rows": wl.rows, "width": wl.width,
            "group_size": wl.group_size, "io_dtype": IO_DTYPE[wl.dtype],
            "mode": "mamba2" if wl.mode == 0 else "onnx", "eps": wl.eps,
            "row_stride": wl.packed_width or wl.width,
            "l2": f"inputs rotate over {m['n_sets']} copies "
                  f"({m['n_sets'] * m['bytes_per_step'] / 1e6:.0f} MB > {L2_BYTES / 1e6:.0f} MB L2)",
            "path": plan["path_name"], "block_threads": plan["block_threads"],
            "grid_blocks": plan["grid_blocks"]}


PER_CONFIG = ("mamba2_prefill", "wide_single_group", "gdn_onnx", "strided_odd_span")


def run_ours(args) -> None:
    rank, world, local_rank = dist_env()
    import torch.distributed as dist
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    torch.cuda.set_device(local_rank)
    device = torch.device("cuda", local_rank)
    import gated_group_rmsnorm_gb300 as g
    L = g.load(build_if_missing=True)
    props = torch.cuda.get_device_properties(device)
    sampler = ClockSampler(str(getattr(props, "uuid", "")))

    wl = ggrn_inputs.WORKLOADS[args.workload]
    if args.rows:
        wl = wl.with_rows(args.rows)
    m = _time_workload(g, L, wl, args.steps, args.warmup, device, sampler)
    sets = m.pop("sets")
    bytes_per_step = m["bytes_per_step"]
    agg = aggregate(bytes_per_step, wl.rows, args.steps, m["max_ms"], world)
    kernel_gbs = bytes_per_step / (m["ms"] / args.steps / 1e3) / 1e9
    peak, _ = hbm_peak()

    # the other prefill workloads, each timed the same way in its own window
    per_config = {}
    if not args.no_per_config and not args.rows:
        pc_steps, pc_warmup = max(args.steps, 50), max(args.warmup, 5)
        for name in PER_CONFIG:
            if name == wl.name:
                continue
            pwl = ggrn_inputs.WORKLOADS[name]
            pm = _time_workload(g, L, pwl, pc_steps, pc_warmup, device, sampler)
            pm.pop("sets")
            pagg = aggregate(pm["bytes_per_step"], pwl.rows, pc_steps, pm["max_ms"], world)
            pgbs = pm["bytes_per_step"] / (pm["ms"] / pc_steps / 1e3) / 1e9
            per_config[name] = {
                "value": round(pagg["gbs"], 2), "unit": UNIT, "steps": pc_steps,
                "warmup": pc_warmup, "ms_per_step": round(pagg["ms_per_step"], 6),
                "rows_per_s": round(pagg["rows_per_s"], 1),
                "pct_of_nominal_8TBs": round(100 * pgbs / NOMINAL_HBM_GBS, 2),
                "launches_per_step": 1, "share_of_timed_region": 1.0,
                "config": _config(pwl, pm), "roofline": _roofline(pwl, pgbs),
                "clocks": pm["clocks"]}
            torch.cuda.empty_cache()

    extra = {}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        extra["cpu_baseline"] = _cpu_baseline(wl, args.cpu_seconds)
        extra["cpu_baseline_all_cores"] = _cpu_baseline_all_cores(wl, args.cpu_seconds / 2)
    e2e = None
    if not args.no_e2e:
        t0 = time.perf_counter()
        e2e = _e2e(g, wl, args.e2e_steps, device)
        e2e["clocks"] = sampler.summary(t0, time.perf_counter())
        e2e_ms = reduce_max(e2e["ms_per_step"], device)
        e2e["value"] = round(world * bytes_per_step / (e2e_ms / 1e3) / 1e9, 2)
        e2e["ms_per_step"] = round(e2e_ms, 4)
    decode = _decode_numbers(g, device) if (rank == 0 and not args.no_decode) else None
    outproj = (_outproj_numbers(g, device, max(args.steps, 20))
               if (rank == 0 and not args.no_outproj) else None)
    if rank == 0 and world == 1 and not args.no_unfused:
        extra["unfused_chain"] = _unfused_chain(wl, sets, min(args.steps, 200))
    del sets
    sampler.stop()

    if rank != 0:
        return
    cfg = _config(wl, m)
    cfg["parallelism"] = f"replicas x{world} (rows are independent; no collective)"
    line = {
        "metric": METRIC, "value": round(agg["gbs"], 2), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(agg["ms_per_step"], 6),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": cfg,
        "rows_per_s": round(agg["rows_per_s"], 1),
        "pct_of_peak": {"of_measured_copy_peak": round(100 * kernel_gbs / peak, 2),
                        "of_nominal_8TBs": round(100 * kernel_gbs / NOMINAL_HBM_GBS, 2)},
        "roofline": _roofline(wl, kernel_gbs),
        "clocks": m["clocks"],
        "gpu_launches": args.steps,
        "e2e": e2e,
    }
    if per_config:
        line["per_config"] = per_config
    line.update(extra)
    if decode is not None:
        line["decode"] = decode
    if outproj is not None:
        line["norm_outproj"] = outproj
    print(json.dumps(line), flush=True)


def run_profile_range(args) -> None:
    """For an ncu range capture: W warm-up launches, then N back-to-back
    launches between cudaProfilerStart and cudaProfilerStop (an ncu range), so
    DRAM traffic is counted over consecutive launches, including each
    launch's output written back from L2 during the next one."""
    import gated_group_rmsnorm_gb300 as g
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    L = g.load(build_if_missing=True)
    wl = ggrn_inputs.WORKLOADS[args.workload]
    if args.rows:
        wl = wl.with_rows(args.rows)
    n_sets = max(2, -(-4 * L2_BYTES // wl.algorithmic_bytes()))
    sets = [ggrn_inputs.make_inputs(wl, device=device, seed=s) for s in range(n_sets)]
    outs = [torch.empty((wl.rows, wl.width), dtype=wl.dtype, device=device) for _ in range(n_sets)]
    stream = torch.cuda.current_stream(device)
    raw = [_raw_args(g, st, o, wl, ctypes.c_void_p(stream.cuda_stream))
           for st, o in zip(sets, outs)]
    for i in range(args.warmup):
        assert L.ggrn_forward(*raw[i % n_sets]) == 0
    torch.cuda.synchronize()
    torch.cuda.profiler.start()
    for i in range(args.profile_range):
        L.ggrn_forward(*raw[i % n_sets])
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    print(json.dumps({"workload": wl.name, "rows": wl.rows, "launches_in_range": args.profile_range,
                      "algorithmic_bytes_per_launch": wl.algorithmic_bytes(),
                      "csrc_sha": kernel_source_hash()}), flush=True)


def run_timeline(args) -> None:
    """Per-CTA timeline of N back-to-back launches of the workload, from the
    profiling build (libggrn_timeline.so, include/ggrn_timeline.h): where a
    launch's time goes besides moving its bytes.  One JSON line of medians
    over the launches after the first three: the period between dependency
    releases, the gap from the last CTA's end to the next release, when the
    first stage reaches the consumers, the spread of the CTAs' ends and the
    mean idle time of an SM at the tail."""
    from gated_group_rmsnorm_gb300 import build as gbuild
    torch.cuda.set_device(0)
    device = torch.device("cuda", 0)
    L = ctypes.CDLL(gbuild.build(timeline=True))
    i64, vp, f, ci = ctypes.c_int64, ctypes.c_void_p, ctypes.c_float, ctypes.c_int
    L.ggrn_forward.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, i64, i64, f, ci, ci, vp]
    L.ggrn_forward.restype = ci
    wl = ggrn_inputs.WORKLOADS[args.workload]
    if args.rows:
        wl = wl.with_rows(args.rows)
    tname = IO_DTYPE[wl.dtype]
    read, clear = getattr(L, f"ggrn_timeline_read_{tname}"), getattr(L, f"ggrn_timeline_clear_{tname}")
    n = min(args.timeline, 60)
    n_sets = max(2, -(-4 * L2_BYTES // wl.algorithmic_bytes()))
    sets = [ggrn_inputs.make_inputs(wl, device=device, seed=s) for s in range(n_sets)]
    outs = [torch.empty((wl.rows, wl.width), dtype=wl.dtype, device=device) for _ in range(n_sets)]
    stream = torch.cuda.current_stream(device)
    from gated_group_rmsnorm_gb300 import binding
    raw = [_raw_args(binding, st, o, wl, ctypes.c_void_p(stream.cuda_stream))
           for st, o in zip(sets, outs)]
    for i in range(max(args.warmup, 3)):
        assert L.ggrn_forward(*raw[i % n_sets]) == 0
    torch.cuda.synchronize()
    assert clear() == 0
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        L.ggrn_forward(*raw[i % n_sets])
    e1.record(stream)
    torch.cuda.synchronize()
    us_event = e0.elapsed_time(e1) * 1e3 / n
    buf = (ctypes.c_ulonglong * (64 * 320 * 5))()
    assert read(buf) == 0
    launches = []
    for e in range(64):
        ctas = [tuple(buf[(e * 320 + b) * 5 + k] for k in range(5)) for b in range(320)]
        ctas = [c for c in ctas if c[1]]
        if ctas:
            launches.append(ctas)
    launches.sort(key=lambda c: min(x[1] for x in c))
    per = []
    for i, c in enumerate(launches[:-1]):
        rel = min(x[1] for x in c)
        ends = sorted(x[3] for x in c)
        firsts = sorted(x[2] - rel for x in c)
        nrel = min(x[1] for x in launches[i + 1])
        per.append({"period": nrel - rel, "busy": ends[-1] - rel, "gap": nrel - ends[-1],
                    "first_min": firsts[0], "first_med": firsts[len(firsts) // 2],
                    "first_max": firsts[-1], "end_spread": ends[-1] - ends[0],
                    "tail_idle_mean": statistics.mean(ends[-1] - x for x in ends),
                    "entry_early": rel - min(x[0] for x in c),
                    "units": (min(x[4] for x in c), max(x[4] for x in c))})
    per = per[3:]
    med = {k: round(statistics.median(p[k] for p in per) / 1e3, 3) for k in per[0] if k != "units"}
    print(json.dumps({"workload": wl.name, "rows": wl.rows, "launches": len(per),
                      "event_us_per_launch": round(us_event, 3),
                      "bytes_at_event_rate_gbs": round(wl.algorithmic_bytes() / us_event / 1e3, 1),
                      "median_us": med, "units_per_cta_min_max": per[0]["units"],
                      "ctas": len(launches[0]), "csrc_sha": kernel_source_hash(),
                      "note": "global-timer stamps per CTA (profiling build); period = release "
                              "to next release, gap = last CTA end to next release, first_* = "
                              "first stage seen after release, tail_idle_mean = mean over CTAs "
                              "of (last end - own end)"}), flush=True)


# ---------------------------------------------------------------------------
# Reference arm: the CPU oracle.
# ---------------------------------------------------------------------------
def run_reference(args) -> None:
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import oracle
    wl = ggrn_inputs.WORKLOADS[args.workload]
    orc = oracle.default()
    # Calibrate rows per step so that W + K steps take about `ref_seconds`.
    cal = wl.with_rows(min(wl.rows, 16))
    cin = ggrn_inputs.make_inputs(cal)
    t0 = time.perf_counter()
    orc.forward(cin.y, cin.gate, cin.w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode)
    per_row = (time.perf_counter() - t0) / cal.rows
    total_steps = max(1, args.steps + args.warmup)
    rows = int(max(1, min(wl.rows, args.ref_seconds / total_steps / max(per_row, 1e-9))))
    swl = wl.with_rows(rows)
    inp = ggrn_inputs.make_inputs(swl)
    out = torch.empty((rows, wl.width), dtype=wl.dtype)

    def step():
        orc.forward(inp.y, inp.gate, inp.w, group_size=wl.group_size, eps=wl.eps, mode=wl.mode,
                    out=out)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    gbs = swl.algorithmic_bytes() * args.steps / el / 1e9
    sample = (f"{rows} of {wl.rows} rows of {wl.name} per step (same recipe), single-threaded "
              f"C++ oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": round(gbs, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": wl.name, "rows": wl.rows, "width": wl.width,
                   "group_size": wl.group_size, "io_dtype": IO_DTYPE[wl.dtype],
                   "mode": "mamba2" if wl.mode == 0 else "onnx", "sample_rows_per_step": rows},
        "rows_per_s": round(rows * args.steps / el, 1),
        "cpu_baseline": {"value": round(gbs, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(gbs, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_rows_sweep(args) -> None:
    """Per-launch time against the row count of one workload, for the
    automatic path and a forced family, with a CUDA-graph replay of the same
    launches; a least-squares line time = fixed + per_row * rows separates
    the fixed cost of a launch from its steady-state bandwidth.  One JSON
    line per measurement, then one per fit."""
    import gated_group_rmsnorm_gb300 as g
    from gated_group_rmsnorm_gb300 import binding
    torch.cuda.set_device(0)
    L = g.load(build_if_missing=True)
    base = ggrn_inputs.WORKLOADS[args.workload]
    paths = [g.PATH_AUTO] + ([args.sweep_path] if args.sweep_path else [])
    results = {}
    for path in paths:
        for rows in [int(r) for r in args.rows_sweep.split(",")]:
            wl = base.with_rows(rows)
            n_sets = max(2, -(-4 * L2_BYTES // wl.algorithmic_bytes()))
            sets = [ggrn_inputs.make_inputs(wl, device="cuda", seed=s) for s in range(n_sets)]
            outs = [torch.empty((rows, wl.width), dtype=wl.dtype, device="cuda") for _ in sets]
            stream = torch.cuda.current_stream()
            raw = [_raw_args(g, s, o, wl, ctypes.c_void_p(stream.cuda_stream)) for s, o in
                   zip(sets, outs)]
            for i in range(30):
                a = raw[i % n_sets]
                st = L.ggrn_forward_path(*a[:-1], path, a[-1])
                if st != 0:
                    raise RuntimeError(g.status_string(st))
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            n = args.steps
            e0.record(stream)
            for i in range(n):
                a = raw[i % n_sets]
                L.ggrn_forward_path(*a[:-1], path, a[-1])
            e1.record(stream)
            torch.cuda.synchronize()
            us = e0.elapsed_time(e1) / n * 1e3
            side = torch.cuda.Stream()
            side.wait_stream(stream)
            graph = torch.cuda.CUDAGraph()
            graph_calls = 20
            with torch.cuda.stream(side):
                raw_s = [a[:-1] + (ctypes.c_void_p(side.cuda_stream),) for a in raw]
                with torch.cuda.graph(graph, stream=side):
                    for i in range(graph_calls):
                        a = raw_s[i % n_sets]
                        L.ggrn_forward_path(*a[:-1], path, a[-1])
            torch.cuda.synchronize()
            for _ in range(3):
                graph.replay()
            torch.cuda.synchronize()
            reps = max(1, n // graph_calls)
            e0.record(stream)
            for _ in range(reps):
                graph.replay()
            e1.record(stream)
            torch.cuda.synchronize()
            us_g = e0.elapsed_time(e1) / (reps * graph_calls) * 1e3
            plan = g.plan(sets[0].y, sets[0].gate, sets[0].w, group_size=wl.group_size,
                          mode=wl.mode, path=path)
            line = {"workload": wl.name, "rows": rows, "path_requested": binding.PATH_NAMES[path],
                    "path": plan["path_name"], "us_per_launch": round(us, 3),
                    "us_per_launch_graph": round(us_g, 3),
                    "gbs": round(wl.algorithmic_bytes() / us / 1e3, 1)}
            print(json.dumps(line), flush=True)
            results.setdefault(binding.PATH_NAMES[path], []).append((rows, us))
            del sets, outs, graph
            torch.cuda.empty_cache()
    for name, pts in results.items():
        n = len(pts)
        mx = sum(r for r, _ in pts) / n
        my = sum(t for _, t in pts) / n
        b = sum((r - mx) * (t - my) for r, t in pts) / sum((r - mx) ** 2 for r, _ in pts)
        a = my - b * mx
        per_row_bytes = base.algorithmic_bytes() / base.rows
        print(json.dumps({"fit": name, "workload": base.name, "fixed_us": round(a, 3),
                          "per_row_ns": round(b * 1e3, 4),
                          "steady_state_gbs": round(per_row_bytes / (b * 1e3), 1)}), flush=True)


def main(argv=None) -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20000)
    ap.add_argument("--warmup", type=int, default=200)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(ggrn_inputs.WORKLOADS), default="strided_odd_span")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's row count (small profiling captures)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--outproj-only", action="store_true",
                    help="only the fused out_proj leg (its JSON block), for profiling")
    ap.add_argument("--d-model", type=int, default=0,
                    help="with --outproj-only: one out_proj width instead of 3840 and 7680")
    ap.add_argument("--no-outproj", action="store_true",
                    help="skip timing the norm fused into the out_proj GEMM against the unfused pair")
    ap.add_argument("--no-per-config", action="store_true",
                    help="time only the headline workload (no per_config block)")
    ap.add_argument("--timeline", type=int, default=0,
                    help="N launches through the profiling build: per-CTA timeline summary "
                         "(not the benchmark line)")
    ap.add_argument("--profile-range", type=int, default=0,
                    help="N launches between profiler start/stop for an ncu range capture "
                         "(prints one short line; not the benchmark line)")
    ap.add_argument("--no-unfused", action="store_true",
                    help="skip timing the unfused PyTorch op chain (context)")
    ap.add_argument("--rows-sweep", default="",
                    help="comma-separated row counts: time per launch vs rows, and the fit "
                         "(fixed cost, steady-state GB/s); not the benchmark line")
    ap.add_argument("--sweep-path", type=int, default=0,
                    help="with --rows-sweep: also a forced kernel family (ggrn_path id)")
    args = ap.parse_args(argv)
    _, world, _ = dist_env()
    if world != args.gpus and args.gpus != 1:
        print(f"warning: --gpus {args.gpus} but WORLD_SIZE={world}", file=sys.stderr)
    if args.outproj_only:
        import gated_group_rmsnorm_gb300 as g
        torch.cuda.set_device(0)
        g.load(build_if_missing=True)
        dm = (args.d_model,) if args.d_model else (3840, 7680)
        print(json.dumps(_outproj_numbers(g, torch.device("cuda", 0), args.steps, dm)), flush=True)
    elif args.timeline:
        run_timeline(args)
    elif args.profile_range:
        run_profile_range(args)
    elif args.rows_sweep:
        if args.steps > 2000:
            args.steps = 1000
        run_rows_sweep(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
