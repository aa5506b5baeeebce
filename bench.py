"""Benchmark: achieved HBM bandwidth of the elementwise kernels on GB300.

Output: two JSON lines on stdout.  The first, ``{"aux_of": METRIC, ...}``,
holds every other measured workload; the LAST line is the compact headline
(well under 4 KB), so a reader that keeps only the tail of stdout still has it.

Headline: fp32 add C = A + B at N = 2^28 per GPU, A and B i.i.d.
uniform[-1, 1) from a seeded generator.  A step is one call of ``ew_add`` over
the whole array (dispatch, vector body, scalar head/tail).

* value       algorithmic bytes (12 per element: read A, read B, write C) of
              all steps on all ranks / max over ranks of the timed region.
              Withheld (null) when the output differs from the CPU oracle.
* roofline    the same bytes per launch / the mean kernel duration (CUDA events
              around every launch on the launching stream), against the measured
              copy bandwidth of this GPU model.
* e2e         the same metric through the public API with host buffers:
              ew_add is called on pinned host A, B and C, so every step moves
              A and B host->device and C device->host inside the kernel, over
              the CPU-GPU link.  Staged variants (cudaMemcpyAsync in, kernel on
              device copies, cudaMemcpyAsync out; serial, and chunked on three
              streams) are reported in the aux line.
* cpu_baseline  the CPU oracle, single-threaded, on the same inputs (rank 0,
              one GPU only); its output is also compared with the GPU's.  An
              all-cores figure (one slice per host core) is reported beside it.
* clocks      SM clock and clock-event reasons read through NVML while the
              timed launches execute (the nvidia-smi stream over the whole run
              as a fallback).
* aux line    the other workloads (bf16/fp16 add at 2^28 aligned, offset by one
              element and with pointers of different parity; bf16/fp16 SAXPY,
              ReLU and both fused chains at 2^28; SAXPY 32M, 2^26 and 2^28;
              ReLU 2^28 out of place and in place; fused add+ReLU and
              SAXPY+ReLU against the unfused pairs; copy and gathers at 2^26
              (fp32 strides 2 to 64 in each block order, bf16 strides 2, 3, 16
              and 64), each gather also against the contiguous copy of its
              dtype and n (frac_of_copy_same_n); the even/odd select;
              fp32 add at 2^20+3; the headline through the persistent schedule
              and the bulk-copy path; chains of short SAXPY calls; the library
              device-to-device copy).  Every entry's output is compared with
              the CPU oracle after its timed launches (in full up to 2^26
              elements, else its first and last 2^20 elements and four seeded
              2^20-element windows); an entry that differs reports
              "parity": "MISMATCH" and no speed.  Entries whose bytes fit in L2
              are labelled "l2_resident" and carry no fraction of HBM peak.

The CPU oracle is imported only by the cpu_baseline leg, the parity checks
beside it and the reference arm; nothing on the timed path calls it.

``--impl reference`` times the CPU oracle instead (the reference arm), on a
bounded sample of the same workload per step.
``--ab widths`` times 16-byte against 32-byte accesses (add, SAXPY, ReLU, copy
in fp32 and bf16 at 2^25 to 2^28), in alternating blocks of 50 launches.
Multi-GPU (torchrun): every rank runs its own 2^28-element slice of a
world x 2^28 problem (weak scaling, no collective on the data path).
"""
import argparse
import ctypes
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

METRIC = "achieved HBM GB/s (and % of GB300 peak) for fp32 add, N=2^28"
N_HEADLINE = 1 << 28
# The pages' own number for this metric and workload: fp32 add at 268.4M
# elements, 1576.5 GB/s for the scalar kernel (Version 1), the best of their
# table ("HyperAI elementwise add on RTX 5090", step 3: RTX 5090 results).
# Another machine (RTX 5090, GDDR7): context for vs_baseline, not a target.
PAGE_BASELINE = {"value": 1576.5, "unit": "GB/s", "hardware": "RTX 5090 (GDDR7)",
                 "kernel": "V1 FP32 scalar add, N = 268.4M"}
FALLBACK_HBM_GBS = 6800.0
HEADLINE_MAX_BYTES = 4096
# outputs up to this many elements are compared in full; larger ones on windows
PARITY_FULL_MAX = 1 << 26
PARITY_WINDOW = 1 << 20
ESIZE = {"f32": 4, "f16": 2, "bf16": 2, "i32": 4}
DT_CODE = {"f32": 0, "f16": 1, "bf16": 2, "i32": 3}


def parse(argv=None):
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--n", type=int, default=N_HEADLINE, help="elements per GPU (headline: 2^28)")
    p.add_argument("--no-aux", action="store_true", help="skip the other workloads")
    p.add_argument("--no-cpu", action="store_true",
                   help="skip the CPU oracle baseline (the headline is then checked on windows)")
    p.add_argument("--path", default="auto", help="kernel variant: auto, scalar, v128, v256, tma")
    p.add_argument("--schedule", default="auto", help="block schedule: auto, oneshot, persistent, laps, tiled")
    p.add_argument("--profile-case", default=None, choices=sorted(PROFILE_CASES),
                   help="run only warmup+steps launches of one workload at --n (for ncu captures)")
    p.add_argument("--stride", type=int, default=None, help="gather stride for the gather profile cases")
    p.add_argument("--ab-strides", default=None,
                   help="gather A/B: comma-separated strides, each on an aligned input and one element past it")
    p.add_argument("--ab-offsets", default="0,1",
                   help="gather A/B: comma-separated input offsets in elements (default 0,1)")
    p.add_argument("--ab", default=None, choices=["widths", "gather"],
                   help="A/B timing instead of the benchmark: access widths, or gather schedules by stride")
    return p.parse_args(argv)


# op, dtype, element offset of every pointer (or of A, B, C)
PROFILE_CASES = {
    "add_f32": ("add", "f32", 0),
    "add_bf16": ("add", "bf16", 0),
    "add_bf16_off1": ("add", "bf16", 1),
    "saxpy_f32": ("saxpy", "f32", 0),
    "relu_f32": ("relu", "f32", 0),
    "copy_f32": ("copy", "f32", 0),
    "gather2_f32": ("gather", "f32", 0),
    "add_relu_f32": ("add_relu", "f32", 0),
    "relu_inplace_f32": ("relu_inplace", "f32", 0),
    "select_i32": ("select", "f32", 0),
    "gather2_span_f32": ("gather_span", "f32", 0),
    "add_bf16_mixed": ("add", "bf16", (1, 0, 3)),
    "gather16_f32": ("gather16", "f32", 0),
    "gather16_f32_off1": ("gather16", "f32", 1),  # input one element past 16 bytes: the general tiled kernel
    "gather16_bf16": ("gather16", "bf16", 0),
    "gather2_bf16": ("gather", "bf16", 0),
    "saxpy_relu_f32": ("saxpy_relu", "f32", 0),
}


def run_profile_case(args):
    """Launch one workload warmup+steps times on the current stream (used under
    ncu: the launch list and the per-kernel counters come from this)."""
    import torch

    import memory_bound_elementwise_gb300 as ew
    from memory_bound_elementwise_gb300 import inputs
    op, dtype, off = PROFILE_CASES[args.profile_case]
    ew.set_path(args.path)
    ew.set_schedule(args.schedule)
    n = args.n
    e = ESIZE[dtype]
    dev = torch.device("cuda", 0)

    offs = off if isinstance(off, tuple) else (off, off, off)  # A (x), B (y), C (z)

    def buf(arr, o):
        raw = torch.empty(arr.size * e + 256, dtype=torch.uint8, device=dev)
        raw[o * e: o * e + arr.size * e].copy_(torch.from_numpy(np.ascontiguousarray(arr).view(np.uint8)))
        return raw, raw.data_ptr() + o * e

    x = inputs.as_dtype(inputs.normal(n, inputs.seed_for("add_f32")), dtype)
    rx, px = buf(x, offs[0])
    ry, py = buf(inputs.as_dtype(inputs.uniform(n, inputs.seed_for("add_f32", 1)), dtype), offs[1])
    rz, pz = buf(np.zeros_like(x), offs[2])
    L = ew.lib()
    s = torch.cuda.current_stream().cuda_stream
    code = DT_CODE[dtype]
    stride = args.stride if args.stride else (16 if op == "gather16" else 2)
    call = {"add": lambda: L.ew_add(code, px, py, pz, n, s),
            "saxpy": lambda: L.ew_saxpy(code, 2.5, px, py, n, s),
            "relu": lambda: L.ew_relu(code, px, pz, n, s),
            "copy": lambda: L.ew_copy(code, px, pz, n, s),
            "gather": lambda: L.ew_gather_stride(code, px, pz, n, stride, s),
            "add_relu": lambda: L.ew_add_relu(code, px, py, pz, n, s),
            "relu_inplace": lambda: L.ew_relu(code, px, px, n, s),
            "select": lambda: L.ew_select_even_odd(3, px, pz, n, s),
            "gather_span": lambda: L.ew_gather_stride(code, px, pz, n, stride, s),
            "gather16": lambda: L.ew_gather_stride(code, px, pz, n, stride, s),
            "saxpy_relu": lambda: L.ew_saxpy_relu(code, 2.5, px, py, n, s)}[op]
    if op == "gather_span":
        ew.set_path("v256")
    for _ in range(args.warmup + args.steps):
        st = call()
        if st != 0:
            raise ew.EwError(st, args.profile_case)
    torch.cuda.synchronize()
    print(json.dumps({"profile_case": args.profile_case, "n": n, "stride": stride if "gather" in op else None,
                      "launches": args.warmup + args.steps, "launch": ew.last_launch()}))


# ---------------------------------------------------------------- helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured hbm_gbs (copy, read+write bytes)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no measured peaks file)"


def profiled_entry(key):
    """An entry of the committed ncu summary (profiles/traffic.json) if it was
    taken on the current kernel sources; else (None, reason)."""
    from memory_bound_elementwise_gb300 import _build
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except Exception:
        return None, "no profiles/traffic.json"
    ent = d.get(key)
    if not ent:
        return None, "kernel not profiled"
    if ent.get("source_digest") != _build.source_digest():
        return None, "kernel sources changed since the ncu capture"
    return ent, ent.get("note", "")


def profiled_traffic(kernel_key):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources; else None."""
    ent, note = profiled_entry(kernel_key)
    if ent is None:
        return None, note
    return ent.get("dram_bytes_per_launch"), note


def profiled_sectors():
    """Global-load sectors per request of the stride-2 gather and of the
    contiguous copy, from the committed ncu summary; None when the kernel
    sources changed since it was taken."""
    ent, note = profiled_entry("sectors_per_request")
    if ent is None:
        return {"gather": None, "copy": None, "note": note}
    return {"gather": ent.get("gather2_f32"), "copy": ent.get("copy_f32"),
            "metric": ent.get("metric"), "note": note}


class ClockSampler:
    """nvidia-smi clock/throttle samples every 100 ms while running (the whole
    run; the timed region itself is sampled through NVML, see NvmlClocks)."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t_start = self.t_stop = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, "t_" + which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "note": "nvidia-smi unavailable"}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            rows.append((t, parts))
        inside = [r for t, r in rows if self.t_start and self.t_stop and
                  self.t_start - 0.1 <= t <= self.t_stop + 0.1]
        use = inside if inside else rows
        sm = [float(r[1]) for r in use if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in use if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[k] for r in use for k in range(4) if r[5 + k].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(use),
                "window": "timed region" if inside else "whole run (timed region shorter than the sampling interval)"}


# NVML clock-event reason bits (nvml.h, nvmlClocksEventReason*)
NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


def summarize_nvml_samples(samples, max_mhz):
    """samples: [(sm_mhz, reason_bits)] taken while the timed launches ran."""
    if not samples:
        return None
    reasons = sorted({name for _, bits in samples for bit, name in NVML_REASONS.items() if bits & bit})
    return {"sm_mhz": statistics.median(m for m, _ in samples), "sm_max_mhz": max_mhz,
            "sm_mhz_min": min(m for m, _ in samples), "reasons": reasons, "samples": len(samples),
            "window": "timed region", "source": "NVML, polled while the timed launches executed"}


class NvmlClocks:
    """SM clock and clock-event reasons through NVML (the driver's
    libnvidia-ml.so.1, by ctypes), read only.  Polled by the host while the
    GPU executes the timed launches, so every sample lies inside the timed
    region however short it is."""
    NVML_CLOCK_SM = 1

    def __init__(self, pci_bus_id=None, index=0, lib=None):
        self.ok = False
        self.samples = []
        self.max_mhz = None
        try:
            self.L = lib if lib is not None else ctypes.CDLL("libnvidia-ml.so.1")
            if self.L.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            rc = -1
            if pci_bus_id:
                rc = self.L.nvmlDeviceGetHandleByPciBusId_v2(pci_bus_id.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.L.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(index), ctypes.byref(self.h))
            if rc != 0:
                return
            self._reasons = getattr(self.L, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
                getattr(self.L, "nvmlDeviceGetCurrentClocksThrottleReasons")
            mx = ctypes.c_uint()
            if self.L.nvmlDeviceGetMaxClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(mx)) == 0:
                self.max_mhz = float(mx.value)
            self.ok = True
        except Exception:
            self.ok = False

    def sample(self):
        if not self.ok:
            return
        mhz, bits = ctypes.c_uint(), ctypes.c_ulonglong()
        if self.L.nvmlDeviceGetClockInfo(self.h, self.NVML_CLOCK_SM, ctypes.byref(mhz)) != 0:
            return
        if self._reasons(self.h, ctypes.byref(bits)) != 0:
            return
        self.samples.append((float(mhz.value), int(bits.value)))

    def summary(self):
        return summarize_nvml_samples(self.samples, self.max_mhz)


def host_cpu_model():
    """CPU model of the host (x86 /proc/cpuinfo, else lscpu, else the machine)."""
    import platform
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    try:
        out = subprocess.run(["lscpu"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                             text=True, timeout=20).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                return "%s %s" % (platform.machine(), line.split(":", 1)[1].strip())
    except Exception:
        pass
    return platform.machine()


def device_facts(torch, dev):
    """SM count, L2 size, driver and runtime versions of the measured GPU."""
    props = torch.cuda.get_device_properties(dev)
    facts = {"sms": props.multi_processor_count,
             "l2_bytes": getattr(props, "L2_cache_size", None),
             "cuda_runtime": torch.version.cuda}
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader",
                              "-i", str(dev.index or 0)], stdout=subprocess.PIPE,
                             stderr=subprocess.DEVNULL, text=True, timeout=20)
        facts["driver"] = out.stdout.strip() or None
    except Exception:
        facts["driver"] = None
    return facts


def pci_bus_id(torch, dev):
    props = torch.cuda.get_device_properties(dev)
    try:
        return "%08x:%02x:%02x.0" % (props.pci_domain_id, props.pci_bus_id, props.pci_device_id)
    except AttributeError:
        return None


# ---------------------------------------------------------------- reference arm

def run_reference(args):
    """The CPU oracle timed as the reference arm, on a bounded sample per step."""
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    from memory_bound_elementwise_gb300 import inputs, metrics
    # calibrate: choose a sample so that (warmup + steps) passes take <= ~120 s
    cal = 1 << 20
    a = inputs.uniform(cal, inputs.seed_for("add_f32"))
    b = inputs.uniform(cal, inputs.seed_for("add_f32", 1))
    t0 = time.perf_counter()
    oracle.add("f32", a, b)
    per_elem = max((time.perf_counter() - t0) / cal, 1e-10)
    budget = 120.0 / max(1, args.steps + args.warmup)
    sample = int(min(args.n, max(1 << 16, budget / per_elem)))
    sample = 1 << int(math.floor(math.log2(sample)))
    a = inputs.uniform(args.n, inputs.seed_for("add_f32"))[:sample]
    b = inputs.uniform(args.n, inputs.seed_for("add_f32", 1))[:sample]
    for _ in range(args.warmup):
        oracle.add("f32", a, b)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.add("f32", a, b)
    dt = time.perf_counter() - t0
    nbytes = metrics.algorithmic_bytes("add", "f32", sample) * args.steps
    value = metrics.gbps(nbytes, dt)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": value / PAGE_BASELINE["value"],
        "baseline": PAGE_BASELINE, "dtype": "f32",
        "data": "synthetic: A, B i.i.d. uniform[-1,1) binary32, seeded PCG64",
        "config": {"workload": "fp32 add C=A+B, N=2^28 per GPU", "n": args.n,
                   "l2": "CPU run (no GPU L2)"},
        "cpu_baseline": {"value": value, "unit": "GB/s", "cores": 1, "kind": "oracle",
                         "sample": "first %d of the %d elements per step (single-threaded C oracle)"
                                   % (sample, args.n), "cpu": host_cpu_model()},
        "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------- timing

class Timer:
    def __init__(self, torch, stream):
        self.torch, self.stream = torch, stream

    def event(self):
        e = self.torch.cuda.Event(enable_timing=True)
        e.record(self.stream)
        return e


def add_copy_fractions(out):
    """Each 2^26 gather entry gets its rate over that of the contiguous copy of
    the same dtype and n measured in the same run (copy_<dtype>_2p26)."""
    for name, ent in out.items():
        m = re.match(r"gather\d+_(f32|bf16)_2p26", name)
        copy = out.get("copy_%s_2p26" % m.group(1), {}) if m else {}
        if "gbps" in ent and "gbps" in copy:
            ent["frac_of_copy_same_n"] = ent["gbps"] / copy["gbps"]


def time_launches(torch, stream, fn, steps, warmup, poll=None):
    """Run fn() warmup times, then `steps` times with an event pair around each
    launch and one around all; returns (total_s, mean_kernel_s).  With `poll`,
    the host calls it repeatedly while the timed launches execute (after the
    first event has completed and until the last one has)."""
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    pairs = []
    t = Timer(torch, stream)
    start = t.event()
    for _ in range(steps):
        e0 = t.event()
        fn()
        e1 = t.event()
        pairs.append((e0, e1))
    end = t.event()
    if poll is not None:
        while not end.query():
            if start.query():
                poll()
            time.sleep(0.0005)
    torch.cuda.synchronize()
    total = start.elapsed_time(end) / 1e3
    per = [a.elapsed_time(b) / 1e3 for a, b in pairs]
    time_launches.last_per_launch = per
    return total, sum(per) / steps


# ---------------------------------------------------------------- parity (CPU oracle)

def parity_windows(n, seed, full_max=PARITY_FULL_MAX, w=PARITY_WINDOW):
    """Index ranges [lo, hi) compared with the oracle: everything up to
    full_max elements; else the first and last w elements and four seeded
    windows of w."""
    if n <= full_max:
        return [(0, n)]
    g = np.random.default_rng(seed)
    starts = {0, n - w} | {int(v) for v in g.integers(0, n - w, size=4)}
    return sorted((s, s + w) for s in starts)


def first_mismatch(got, want, dtype, nan_class):
    """Index of the first element whose bits differ (NaN matches NaN when
    nan_class), or None."""
    bits = np.uint32 if ESIZE[dtype] == 4 else np.uint16
    g = np.ascontiguousarray(got).view(bits)
    w = np.ascontiguousarray(want).view(bits)
    if g.shape != w.shape:
        return 0
    diff = g != w
    if nan_class and dtype != "i32":
        if dtype == "f32":
            gn, wn = (g & 0x7FFFFFFF) > 0x7F800000, (w & 0x7FFFFFFF) > 0x7F800000
        else:
            inf = 0x7C00 if dtype == "f16" else 0x7F80
            gn, wn = (g & 0x7FFF) > inf, (w & 0x7FFF) > inf
        diff &= ~(gn & wn)
    bad = np.nonzero(diff)[0]
    return int(bad[0]) if bad.size else None


class DevBuf:
    """n elements of `dtype` on the device, `offset` elements past a 256-byte
    boundary, filled from a host array."""

    def __init__(self, torch, dev, arr, dtype, offset=0):
        self.torch, self.dtype, self.e, self.off = torch, dtype, ESIZE[dtype], offset
        self.n = arr.size
        self.raw = torch.empty(self.n * self.e + 256, dtype=torch.uint8, device=dev)
        self.ptr = self.raw.data_ptr() + offset * self.e
        self.fill(arr)

    def fill(self, arr):
        b = np.ascontiguousarray(arr).view(np.uint8)
        self.raw[self.off * self.e: self.off * self.e + b.size].copy_(self.torch.from_numpy(b))

    def read(self, lo, hi):
        host = {"f32": np.float32, "i32": np.int32}.get(self.dtype, np.uint16)
        seg = self.raw[(self.off + lo) * self.e:(self.off + hi) * self.e]
        return seg.cpu().numpy().view(host)


class Parity:
    """Compares a workload's device output with the CPU oracle on the same
    inputs.  `want(lo, hi)` returns the oracle's result for outputs [lo, hi)."""

    def __init__(self, enabled):
        self.enabled = enabled
        self.oracle = None
        if enabled:
            import oracle
            self.oracle = oracle

    def check(self, name, out, want, n, nan_class=True, full_max=PARITY_FULL_MAX):
        if not self.enabled:
            return {"parity": "unchecked"}
        self.torch_sync(out)
        seed = sum(name.encode()) * 7919
        checked = 0
        for lo, hi in parity_windows(n, seed, full_max):
            bad = first_mismatch(out.read(lo, hi), want(lo, hi), out.dtype, nan_class)
            if bad is not None:
                return {"parity": "MISMATCH", "first_bad_index": lo + bad}
            checked += hi - lo
        return {"parity": True, "parity_elements": checked}

    @staticmethod
    def torch_sync(out):
        out.torch.cuda.synchronize()


# ---------------------------------------------------------------- aux workloads

class Aux:
    """The other workloads of the aux line: timing, then a parity check."""

    def __init__(self, torch, ew, inputs, metrics, stream, peak, dev, parity, l2_bytes):
        self.torch, self.ew, self.inputs, self.metrics = torch, ew, inputs, metrics
        self.stream, self.peak, self.dev, self.parity = stream, peak, dev, parity
        self.l2_bytes = l2_bytes or 0
        self.L = ew.lib()
        self.s = stream.cuda_stream
        self.out = {}

    def buf(self, arr, dtype, offset=0):
        return DevBuf(self.torch, self.dev, arr, dtype, offset)

    def _speed(self, nbytes, kern_s, footprint=None):
        g = self.metrics.gbps(nbytes, kern_s)
        ent = {"gbps": g, "kernel_ms": kern_s * 1e3, "bytes_per_launch": nbytes}
        if (footprint if footprint is not None else nbytes) <= self.l2_bytes:
            ent["l2_resident"] = True  # working set fits in L2: not an HBM figure
        else:
            ent["frac"] = g / self.peak
            ent["frac_of_nominal_8tbs"] = g / 8000.0
        return ent

    def _finish(self, name, ent, check):
        """check: (out DevBuf, want(lo, hi), n[, rerun][, kwargs]) or None.
        rerun: resets in-place operands and launches once more before reading."""
        if check is None:
            ent["parity"] = "not applicable"
        else:
            out_buf, want, n = check[0], check[1], check[2]
            rerun = check[3] if len(check) > 3 else None
            kw = check[4] if len(check) > 4 else {}
            if rerun is not None and self.parity.enabled:
                rerun()
            res = self.parity.check(name, out_buf, want, n, **kw)
            if res["parity"] == "MISMATCH":
                ent = {"parity": "MISMATCH", "first_bad_index": res["first_bad_index"],
                       "note": "output differs from the CPU oracle: no speed reported"}
            else:
                ent.update(res)
        self.out[name] = ent

    def _call_ok(self, call, name):
        st = call()
        if st != 0:
            raise self.ew.EwError(st, name)

    def record(self, name, op, dtype, n, call, check, steps=50, footprint=None):
        total, kern = time_launches(self.torch, self.stream, lambda: self._call_ok(call, name), steps, 3)
        per = sorted(time_launches.last_per_launch)
        nbytes = self.metrics.algorithmic_bytes(op, dtype, n)
        ent = self._speed(nbytes, kern, footprint)
        ent.update({"kernel_ms_median": per[len(per) // 2] * 1e3, "kernel_ms_min": per[0] * 1e3,
                    "step_ms": total / steps * 1e3, "gelem_per_s": n / kern / 1e9,
                    "launch": self.ew.last_launch()})
        self._finish(name, ent, check)

    def record_graph(self, name, op, dtype, n, call, check, k=50, reps=5):
        """K launches captured in one CUDA graph and replayed: the per-launch
        time without host launch gaps (median of `reps` replays).  The parity
        rerun replays the graph once more (k launches)."""
        torch, stream = self.torch, self.stream
        self._call_ok(call, name)  # fills the per-device caches outside the capture
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for _ in range(k):
                st = call()
        if st != 0:
            raise self.ew.EwError(st, name + " (captured)")
        times = []
        with torch.cuda.stream(stream):  # replay() launches on the current stream
            graph.replay()
            torch.cuda.synchronize()
            for _ in range(reps):
                e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                e0.record(stream)
                graph.replay()
                e1.record(stream)
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) / 1e3 / k)
        per = sorted(times)[len(times) // 2]
        ent = self._speed(self.metrics.algorithmic_bytes(op, dtype, n), per)
        ent.update({"launches_per_graph": k, "replays": reps,
                    "note": "%d launches in one CUDA graph; per-launch time of the median replay" % k})
        if check is not None:
            reset = check[3] if len(check) > 3 else None

            def rerun():
                if reset is not None:
                    reset()
                with torch.cuda.stream(stream):
                    graph.replay()
                torch.cuda.synchronize()
            check = (check[0], check[1], check[2], rerun) + tuple(check[4:])
        self._finish(name, ent, check)
        del graph

    def record_fn(self, name, nbytes, fn, check, steps=50, note=None, footprint=None):
        """A step of several calls (e.g. an unfused pair), timed as one."""
        total, kern = time_launches(self.torch, self.stream, fn, steps, 3)
        ent = self._speed(nbytes, kern, footprint)
        if note:
            ent["note"] = note
        self._finish(name, ent, check)

    # -------------------------------------------------------------- workloads

    def run(self):
        orc = self.parity.oracle
        L, s = self.L, self.s
        inputs = self.inputs
        ew = self.ew
        n28, n26 = 1 << 28, 1 << 26

        # -- 16-bit add, SAXPY, ReLU and fused chains at 2^28
        for dtype in ("bf16", "f16"):
            code = DT_CODE[dtype]
            xa = inputs.as_dtype(inputs.normal(n28, inputs.seed_for("add_16")), dtype)
            xb = inputs.as_dtype(inputs.normal(n28, inputs.seed_for("add_16", 1)), dtype)

            def want_add(lo, hi, xa=xa, xb=xb, dtype=dtype):
                return orc.add(dtype, xa[lo:hi], xb[lo:hi])
            for off in (0, 1):
                A, B, C = self.buf(xa, dtype, off), self.buf(xb, dtype, off), self.buf(np.zeros_like(xa), dtype, off)
                self.record("add_%s_2p28_off%d" % (dtype, off), "add", dtype, n28,
                            lambda: L.ew_add(code, A.ptr, B.ptr, C.ptr, n28, s), (C, want_add, n28))
                del A, B, C
            A, B, C = self.buf(xa, dtype), self.buf(xb, dtype), self.buf(np.zeros_like(xa), dtype)
            self.record("saxpy_%s_2p28_inplace" % dtype, "saxpy", dtype, n28,
                        lambda: L.ew_saxpy(code, 2.5, A.ptr, B.ptr, n28, s),
                        (B, lambda lo, hi: orc.saxpy(dtype, 2.5, xa[lo:hi], xb[lo:hi]), n28,
                         lambda: (B.fill(xb), self._call_ok(lambda: L.ew_saxpy(code, 2.5, A.ptr, B.ptr, n28, s),
                                                            "saxpy"))))
            B.fill(xb)
            self.record("relu_%s_2p28" % dtype, "relu", dtype, n28, lambda: L.ew_relu(code, A.ptr, C.ptr, n28, s),
                        (C, lambda lo, hi: orc.relu(dtype, xa[lo:hi]), n28), )
            self.record("add_relu_%s_2p28_fused" % dtype, "add_relu", dtype, n28,
                        lambda: L.ew_add_relu(code, A.ptr, B.ptr, C.ptr, n28, s),
                        (C, lambda lo, hi: orc.relu(dtype, orc.add(dtype, xa[lo:hi], xb[lo:hi])), n28))
            self.record("saxpy_relu_%s_2p28_fused" % dtype, "saxpy_relu", dtype, n28,
                        lambda: L.ew_saxpy_relu(code, 2.5, A.ptr, C.ptr, n28, s),
                        (C, lambda lo, hi: orc.relu(dtype, orc.saxpy(dtype, 2.5, xa[lo:hi], xb[lo:hi])), n28,
                         lambda: (C.fill(xb), self._call_ok(
                             lambda: L.ew_saxpy_relu(code, 2.5, A.ptr, C.ptr, n28, s), "saxpy_relu"))))
            del A, B, C
            if dtype == "bf16":
                # pointers of different parity (A +1, B +0, C +3 elements): the
                # realigning bulk-copy kernel (default) against 2-byte accesses
                A, B, C = self.buf(xa, dtype, 1), self.buf(xb, dtype, 0), self.buf(np.zeros_like(xa), dtype, 3)
                self.record("add_bf16_2p28_mixed_parity", "add", dtype, n28,
                            lambda: L.ew_add(code, A.ptr, B.ptr, C.ptr, n28, s), (C, want_add, n28))
                C.fill(np.zeros_like(xa))
                ew.set_path("v256")
                self.record("add_bf16_2p28_mixed_parity_2byte", "add", dtype, n28,
                            lambda: L.ew_add(code, A.ptr, B.ptr, C.ptr, n28, s), (C, want_add, n28))
                ew.set_path("auto")
                del A, B, C
            del xa, xb

        # -- fp32 SAXPY: 32M (the pages' size), then 2^26 and 2^28
        n32m = 32 << 20
        x = inputs.normal(n32m, inputs.seed_for("saxpy_f32"))
        y = inputs.normal(n32m, inputs.seed_for("saxpy_f32", 1))
        X, Y = self.buf(x, "f32"), self.buf(y, "f32")

        def saxpy32():
            return L.ew_saxpy(0, 2.5, X.ptr, Y.ptr, n32m, s)
        self.record("saxpy_f32_32M_inplace", "saxpy", "f32", n32m, saxpy32,
                    (Y, lambda lo, hi: orc.saxpy("f32", 2.5, x[lo:hi], y[lo:hi]), n32m,
                     lambda: (Y.fill(y), self._call_ok(saxpy32, "saxpy"))), steps=200)
        Y.fill(y)

        def want_saxpy_k(lo, hi, k=50):
            r = y[lo:hi]
            for _ in range(k):
                r = orc.saxpy("f32", 2.5, x[lo:hi], r)
            return r
        self.record_graph("saxpy_f32_32M_inplace_graph", "saxpy", "f32", n32m, saxpy32,
                          (Y, want_saxpy_k, n32m, lambda: Y.fill(y), {"full_max": 0}))
        del X, Y
        x = inputs.normal(n28, inputs.seed_for("saxpy_f32", 2))
        y = inputs.normal(n28, inputs.seed_for("saxpy_f32", 3))
        X, Y = self.buf(x, "f32"), self.buf(y, "f32")
        for lg in (26, 28):
            m = 1 << lg

            def call(m=m):
                return L.ew_saxpy(0, 2.5, X.ptr, Y.ptr, m, s)
            self.record("saxpy_f32_2p%d_inplace" % lg, "saxpy", "f32", m, call,
                        (Y, lambda lo, hi: orc.saxpy("f32", 2.5, x[lo:hi], y[lo:hi]), m,
                         lambda call=call: (Y.fill(y), self._call_ok(call, "saxpy"))),
                        steps=100 if lg == 26 else 50)
        del X, Y, x, y

        # -- fp32 ReLU at 2^28: out of place, in place on fresh data, in place again
        x = inputs.inject_signed_zeros(inputs.normal(n28, inputs.seed_for("relu_f32")))
        X, Y = self.buf(x, "f32"), self.buf(np.zeros_like(x), "f32")
        want_relu = lambda lo, hi: orc.relu("f32", x[lo:hi])  # noqa: E731
        self.record("relu_f32_2p28", "relu", "f32", n28, lambda: L.ew_relu(0, X.ptr, Y.ptr, n28, s),
                    (Y, want_relu, n28))
        # in place on fresh data: refill from the pristine copy before each
        # launch (outside the event pair), so every timed launch sees ~50% negatives
        kern_ms = []
        for _ in range(13):
            with self.torch.cuda.stream(self.stream):
                Y.raw.copy_(X.raw, non_blocking=True)
            e0, e1 = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            st = L.ew_relu(0, Y.ptr, Y.ptr, n28, s)
            e1.record(self.stream)
            if st != 0:
                raise ew.EwError(st, "relu in place")
            self.torch.cuda.synchronize()
            kern_ms.append(e0.elapsed_time(e1))
        kern = sum(kern_ms[3:]) / len(kern_ms[3:]) / 1e3
        ent = self._speed(self.metrics.algorithmic_bytes("relu", "f32", n28), kern)
        ent["launch"] = ew.last_launch()
        self._finish("relu_f32_2p28_inplace_fresh", ent, (Y, want_relu, n28))
        # in place again on the now non-negative data: nothing changes, so no
        # vector is stored (the page's case B: 4 bytes per element, read only)
        self.record_fn("relu_f32_2p28_inplace_nonnegative", 4 * n28,
                       lambda: self._call_ok(lambda: L.ew_relu(0, Y.ptr, Y.ptr, n28, s), "relu in place"),
                       (Y, want_relu, n28), note="read-only bytes: unchanged vectors are not stored")
        del X, Y, x

        # -- copy and gathers at 2^26
        x = inputs.uniform(n26, inputs.seed_for("copy_f32"), 0.0, 1.0)
        X, Y = self.buf(x, "f32"), self.buf(np.zeros_like(x), "f32")
        gathered = {}

        def want_gather(stride):
            if stride not in gathered:
                gathered[stride] = orc.gather_stride(x, stride)
            g = gathered[stride]
            return lambda lo, hi: g[lo:hi]
        want_copy = lambda lo, hi: x[lo:hi]  # noqa: E731

        def clear():
            Y.raw.zero_()
        copy_call = lambda: L.ew_copy(0, X.ptr, Y.ptr, n26, s)  # noqa: E731
        self.record("copy_f32_2p26", "copy", "f32", n26, copy_call, (Y, want_copy, n26), steps=200)
        clear()
        self.record_graph("copy_f32_2p26_graph", "copy", "f32", n26, copy_call, (Y, want_copy, n26, clear))
        clear()
        g2 = lambda: L.ew_gather_stride(0, X.ptr, Y.ptr, n26, 2, s)  # noqa: E731
        self.record_graph("gather2_f32_2p26_graph", "gather", "f32", n26, g2, (Y, want_gather(2), n26, clear))
        variants = [("gather2_f32_2p26", 2, "auto", "auto"), ("gather4_f32_2p26", 4, "auto", "auto"),
                    ("gather8_f32_2p26", 8, "auto", "auto"), ("gather12_f32_2p26", 12, "auto", "auto"),
                    ("gather16_f32_2p26", 16, "auto", "auto"),
                    ("gather64_f32_2p26", 64, "auto", "auto"),
                    ("gather16_f32_2p26_lap_order", 16, "auto", "laps"),
                    ("gather2_f32_2p26_index_order", 2, "auto", "oneshot"),
                    ("gather4_f32_2p26_index_order", 4, "auto", "oneshot"),
                    ("gather16_f32_2p26_index_order", 16, "auto", "oneshot"),
                    ("gather2_f32_2p26_span", 2, "v256", "auto")]
        for name, stride, path, sched in variants:
            ew.set_path(path)
            ew.set_schedule(sched)
            clear()
            self.record(name, "gather", "f32", n26,
                        lambda stride=stride: L.ew_gather_stride(0, X.ptr, Y.ptr, n26, stride, s),
                        (Y, want_gather(stride), n26), steps=100)
        ew.set_path("auto")
        ew.set_schedule("auto")
        del X, Y
        gathered.clear()
        # 16-bit gathers (the tiled kernels' 2-byte instantiations)
        xh = inputs.as_dtype(inputs.uniform(n26, inputs.seed_for("copy_f32", 3), 0.0, 1.0), "bf16")
        X, Y = self.buf(xh, "bf16"), self.buf(np.zeros_like(xh), "bf16")
        self.record("copy_bf16_2p26", "copy", "bf16", n26, lambda: L.ew_copy(2, X.ptr, Y.ptr, n26, s),
                    (Y, lambda lo, hi: xh[lo:hi], n26), steps=200)
        for stride in (2, 3, 16, 64):
            want = orc.gather_stride(xh, stride)
            Y.raw.zero_()
            self.record("gather%d_bf16_2p26" % stride, "gather", "bf16", n26,
                        lambda stride=stride: L.ew_gather_stride(2, X.ptr, Y.ptr, n26, stride, s),
                        (Y, lambda lo, hi, want=want: want[lo:hi], n26), steps=100)
        del X, Y, xh

        # -- the branch-free even/odd select on int32 (CUDA-MODE lecture notes §6)
        xi = inputs.rng(inputs.seed_for("copy_f32", 7)).integers(-2 ** 31, 2 ** 31, size=n28,
                                                                 dtype=np.int64).astype(np.int32)
        X, Y = self.buf(xi, "i32"), self.buf(np.zeros_like(xi), "i32")
        self.record("select_even_odd_i32_2p28", "select", "i32", n28,
                    lambda: L.ew_select_even_odd(3, X.ptr, Y.ptr, n28, s),
                    (Y, lambda lo, hi: orc.select_even_odd(xi[lo:hi]), n28))
        del X, Y, xi

        # -- fp32 add at 2^20 + 3 (L2-resident, launch-bound)
        n1 = (1 << 20) + 3
        a = inputs.uniform(n1, inputs.seed_for("add_f32_small"))
        b = inputs.uniform(n1, inputs.seed_for("add_f32_small", 1))
        A, B, C = self.buf(a, "f32"), self.buf(b, "f32"), self.buf(np.zeros_like(a), "f32")
        self.record("add_f32_2p20p3_l2_resident", "add", "f32", n1, lambda: L.ew_add(0, A.ptr, B.ptr, C.ptr, n1, s),
                    (C, lambda lo, hi: orc.add("f32", a[lo:hi], b[lo:hi]), n1), steps=500)
        del A, B, C

        # -- the headline workload through other variants, and the fused chains
        a = inputs.normal(n28, inputs.seed_for("add_f32"))
        b = inputs.normal(n28, inputs.seed_for("add_f32", 1))
        A, B, C = self.buf(a, "f32"), self.buf(b, "f32"), self.buf(np.zeros_like(a), "f32")
        want_add_relu = lambda lo, hi: orc.relu("f32", orc.add("f32", a[lo:hi], b[lo:hi]))  # noqa: E731
        self.record("add_relu_f32_2p28_fused", "add_relu", "f32", n28,
                    lambda: L.ew_add_relu(0, A.ptr, B.ptr, C.ptr, n28, s), (C, want_add_relu, n28))
        C.raw.zero_()

        def unfused():
            for st in (L.ew_add(0, A.ptr, B.ptr, C.ptr, n28, s), L.ew_relu(0, C.ptr, C.ptr, n28, s)):
                if st != 0:
                    raise ew.EwError(st, "add then relu")
        self.record_fn("add_then_relu_f32_2p28_unfused", self.metrics.algorithmic_bytes("add_relu", "f32", n28),
                       unfused, (C, want_add_relu, n28),
                       note="two launches per step (add, then ReLU in place); GB/s counts the fused "
                            "operation's 12 bytes per element")
        # SAXPY + ReLU fused in one pass (y = relu(2.5 x + y) in place, x = A, y = C)
        want_sr = lambda lo, hi: orc.relu("f32", orc.saxpy("f32", 2.5, a[lo:hi], b[lo:hi]))  # noqa: E731
        sr = lambda: L.ew_saxpy_relu(0, 2.5, A.ptr, C.ptr, n28, s)  # noqa: E731
        self.record("saxpy_relu_f32_2p28_fused", "saxpy_relu", "f32", n28, sr,
                    (C, want_sr, n28, lambda: (C.fill(b), self._call_ok(sr, "saxpy_relu"))))

        def saxpy_unfused():
            for st in (L.ew_saxpy(0, 2.5, A.ptr, C.ptr, n28, s), L.ew_relu(0, C.ptr, C.ptr, n28, s)):
                if st != 0:
                    raise ew.EwError(st, "saxpy then relu")
        self.record_fn("saxpy_then_relu_f32_2p28_unfused",
                       self.metrics.algorithmic_bytes("saxpy_relu", "f32", n28), saxpy_unfused,
                       (C, want_sr, n28, lambda: (C.fill(b), saxpy_unfused())),
                       note="two launches per step (SAXPY, then ReLU in place); GB/s counts the fused "
                            "operation's 12 bytes per element")
        want_a_plus_b = lambda lo, hi: orc.add("f32", a[lo:hi], b[lo:hi])  # noqa: E731
        for label, path, sched in (("persistent", "auto", "persistent"), ("tma", "tma", "auto")):
            ew.set_path(path)
            ew.set_schedule(sched)
            C.raw.zero_()
            self.record("add_f32_2p28_" + label, "add", "f32", n28,
                        lambda: L.ew_add(0, A.ptr, B.ptr, C.ptr, n28, s), (C, want_a_plus_b, n28))
        ew.set_path("tma")
        ew.set_schedule("auto")
        C.raw.zero_()
        self.record("copy_f32_2p26_tma", "copy", "f32", n26, lambda: L.ew_copy(0, A.ptr, C.ptr, n26, s),
                    (C, lambda lo, hi: a[lo:hi], n26), steps=200)
        ew.set_path("auto")
        del A, B, C, a, b

        # -- chains of short calls launched back to back without events in
        # between: programmatic dependent launch on (the default) against off
        for lg in (20, 23, 25):
            m = 1 << lg
            cx = inputs.normal(m, inputs.seed_for("saxpy_f32", 4))
            cy = inputs.normal(m, inputs.seed_for("saxpy_f32", 5))
            X, Y = self.buf(cx, "f32"), self.buf(cy, "f32")
            call = lambda m=m: L.ew_saxpy(0, 0.5, X.ptr, Y.ptr, m, s)  # noqa: E731
            for prog in (True, False):
                ew.set_programmatic_launch(prog)
                for _ in range(10):
                    call()
                self.torch.cuda.synchronize()
                e0, e1 = self.torch.cuda.Event(enable_timing=True), self.torch.cuda.Event(enable_timing=True)
                e0.record(self.stream)
                for _ in range(200):
                    self._call_ok(call, "saxpy chain")
                e1.record(self.stream)
                self.torch.cuda.synchronize()
                per = e0.elapsed_time(e1) / 1e3 / 200
                ent = self._speed(self.metrics.algorithmic_bytes("saxpy", "f32", m), per)
                ent["note"] = "200 launches back to back, time per launch from one event pair"
                self._finish("saxpy_chain_f32_2p%d_%s" % (lg, "pdl" if prog else "plain"), ent,
                             (Y, lambda lo, hi, cx=cx, cy=cy: orc.saxpy("f32", 0.5, cx[lo:hi], cy[lo:hi]), m,
                              lambda call=call, cy=cy: (Y.fill(cy), self._call_ok(call, "saxpy chain"))))
                Y.fill(cy)
            ew.set_programmatic_launch(True)
            del X, Y

        # -- device-to-device copy ceiling of this GPU (cudaMemcpyAsync via
        # torch copy_, 2 GiB, read + write bytes), timed on the same stream
        big = self.torch.empty(1 << 31, dtype=self.torch.uint8, device=self.dev)
        big2 = self.torch.empty_like(big)

        def d2d():
            with self.torch.cuda.stream(self.stream):
                big2.copy_(big, non_blocking=True)
        total, kern = time_launches(self.torch, self.stream, d2d, 20, 3)
        g = self.metrics.gbps(2 * big.numel(), kern)
        self.out["memcpy_d2d_2GiB"] = {"gbps": g, "frac": g / self.peak, "kernel_ms": kern * 1e3,
                                       "parity": "not applicable (library copy)",
                                       "note": "library device-to-device copy (torch copy_), read+write bytes"}
        del big, big2
        for ent in self.out.values():  # against the copy ceiling measured in this run
            if "frac" in ent:
                ent["frac_of_d2d"] = ent["gbps"] / g
        add_copy_fractions(self.out)
        if "gather2_f32_2p26" in self.out:
            self.out["gather2_f32_2p26"]["sectors_per_request"] = profiled_sectors()
        return self.out


# ---------------------------------------------------------------- access-width A/B

def run_ab_widths(args):
    """16-byte against 32-byte accesses: add, SAXPY, ReLU, copy in fp32 and
    bf16 at 2^25 to 2^28.  Each width runs in blocks of 50 launches of the
    same kernel (the way a caller repeats one operation), the blocks of the
    two widths alternating 4 times on the same buffers; the first 5 launches
    of every block are not counted.  Prints one JSON line per case with the
    median and minimum per launch."""
    import torch

    import memory_bound_elementwise_gb300 as ew
    from memory_bound_elementwise_gb300 import inputs, metrics
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    s = stream.cuda_stream
    L = ew.lib()
    parity = Parity(not args.no_cpu)
    block, blocks, skip = 50, 4, 5
    for dtype in ("f32", "bf16"):
        code = DT_CODE[dtype]
        for lg in (25, 26, 27, 28):
            n = 1 << lg
            a = inputs.as_dtype(inputs.normal(n, inputs.seed_for("add_f32")), dtype)
            b = inputs.as_dtype(inputs.normal(n, inputs.seed_for("add_f32", 1)), dtype)
            A, B = DevBuf(torch, dev, a, dtype), DevBuf(torch, dev, b, dtype)
            C = DevBuf(torch, dev, np.zeros_like(a), dtype)
            orc = parity.oracle
            cases = [("add", lambda: L.ew_add(code, A.ptr, B.ptr, C.ptr, n, s),
                      lambda lo, hi: orc.add(dtype, a[lo:hi], b[lo:hi])),
                     ("saxpy", lambda: L.ew_saxpy(code, 2.5, A.ptr, C.ptr, n, s), None),
                     ("relu", lambda: L.ew_relu(code, A.ptr, C.ptr, n, s),
                      lambda lo, hi: orc.relu(dtype, a[lo:hi])),
                     ("copy", lambda: L.ew_copy(code, A.ptr, C.ptr, n, s), lambda lo, hi: a[lo:hi])]
            for op, call, want in cases:
                if op == "saxpy":
                    C.fill(b)  # y = C: in place; values drift over the launches (timing only)
                per = {"v128": [], "v256": []}
                for _ in range(blocks):
                    for path in ("v128", "v256"):
                        ew.set_path(path)
                        evs = []
                        for k in range(block):
                            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
                            e0.record(stream)
                            st = call()
                            e1.record(stream)
                            if st != 0:
                                raise ew.EwError(st, op)
                            if k >= skip:
                                evs.append((e0, e1))
                        torch.cuda.synchronize()
                        per[path] += [e0.elapsed_time(e1) / 1e3 for e0, e1 in evs]
                nbytes = metrics.algorithmic_bytes(op, dtype, n)
                row = {"ab": "widths", "op": op, "dtype": dtype, "n": n,
                       "launches_each": blocks * (block - skip), "blocks": blocks}
                for path in ("v128", "v256"):
                    t = sorted(per[path])
                    row[path] = {"median_us": t[len(t) // 2] * 1e6, "min_us": t[0] * 1e6,
                                 "mean_us": sum(t) / len(t) * 1e6,
                                 "gbps_median": metrics.gbps(nbytes, t[len(t) // 2])}
                    ew.set_path(path)
                    if want is not None:
                        C.raw.zero_()
                        call()
                        row[path].update(parity.check("%s_%s_%s" % (op, dtype, path), C, want, n))
                    elif op == "saxpy" and parity.enabled:
                        C.fill(b)
                        call()
                        row[path].update(parity.check("saxpy_%s_%s" % (dtype, path), C,
                                                      lambda lo, hi: orc.saxpy(dtype, 2.5, a[lo:hi], b[lo:hi]), n))
                ew.set_path("auto")
                row["v256_over_v128"] = row["v128"]["median_us"] / row["v256"]["median_us"]
                print(json.dumps(row), flush=True)
            del A, B, C


def run_ab_gather(args):
    """Gather schedules (lap order, tiled) at strides 2 to 64, on 2^26 fp32 and
    bf16 elements, on a 16-byte aligned input and on one a single element past
    it: median and mean per launch and parity for each."""
    import torch

    import memory_bound_elementwise_gb300 as ew
    from memory_bound_elementwise_gb300 import inputs, metrics
    dev = torch.device("cuda", 0)
    stream = torch.cuda.Stream(dev)
    s = stream.cuda_stream
    L = ew.lib()
    parity = Parity(not args.no_cpu)
    n = args.n if args.n != N_HEADLINE else 1 << 26
    # aligned: the specialised strides and three that only the general tiled
    # kernel serves; one element past 16 bytes: the general kernel throughout
    plan = [(0, [2, 3, 4, 5, 6, 7, 8, 12, 16, 17, 24, 32, 40, 48, 63, 64]), (1, [2, 3, 4, 5, 12, 16, 40])]
    if args.ab_strides or args.stride:
        chosen = [int(v) for v in args.ab_strides.split(",")] if args.ab_strides else [args.stride]
        plan = [(int(o), chosen) for o in args.ab_offsets.split(",")]
    for dtype, (offset, strides) in ((d, p) for d in ("f32", "bf16") for p in plan):
        code = DT_CODE[dtype]
        x = inputs.as_dtype(inputs.uniform(n, inputs.seed_for("copy_f32"), 0.0, 1.0), dtype)
        X, Y = DevBuf(torch, dev, x, dtype, offset), DevBuf(torch, dev, np.zeros_like(x), dtype)
        for stride in strides:
            want = parity.oracle.gather_stride(x, stride) if parity.enabled else None
            row = {"ab": "gather", "dtype": dtype, "n": n, "stride": stride, "input_offset_elems": offset}
            for sched in ("auto", "laps", "tiled"):
                ew.set_schedule(sched)
                call = lambda: L.ew_gather_stride(code, X.ptr, Y.ptr, n, stride, s)  # noqa: E731
                Y.raw.zero_()
                total, kern = time_launches(torch, stream, call, 50, 3)
                t = sorted(time_launches.last_per_launch)
                rec = ew.last_launch()
                nbytes = metrics.algorithmic_bytes("gather", dtype, n)
                row[sched] = {"median_us": t[len(t) // 2] * 1e6, "mean_us": kern * 1e6,
                              "gbps_median": metrics.gbps(nbytes, t[len(t) // 2]),
                              "gbps_mean": metrics.gbps(nbytes, kern),
                              "schedule_ran": ew.SCHED_NAMES.get(rec["schedule"], rec["schedule"])}
                if want is not None:
                    row[sched].update(parity.check("g%d%s%s" % (stride, dtype, sched), Y,
                                                   lambda lo, hi: want[lo:hi], n))
            ew.set_schedule("auto")
            print(json.dumps(row), flush=True)
        del X, Y


# ---------------------------------------------------------------- our arm

def headline_line(*, value, parity, world, steps, warmup, total_s, n, lo, hi, step_bytes, rec, facts,
                  gpu_name, achieved, peak, peak_src, traffic, traffic_note, kern_s, per_launch,
                  e2e, clocks, cpu_baseline):
    """The compact headline dict (printed last, well under HEADLINE_MAX_BYTES)."""
    ok = parity is True or parity == "unchecked"
    line = {
        "metric": METRIC, "value": value if ok else None, "unit": "GB/s", "n_gpus": world,
        "steps": steps, "warmup": warmup, "ms_per_step": total_s / steps * 1e3,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / PAGE_BASELINE["value"]) if ok else None,
        "baseline": "%s GB/s, %s, %s" % (PAGE_BASELINE["value"], PAGE_BASELINE["kernel"],
                                         PAGE_BASELINE["hardware"]),
        "dtype": "f32",
        "data": "synthetic: A, B i.i.d. uniform[-1,1) binary32, seeded PCG64 per rank",
        "config": {"workload": "fp32 add C=A+B, N=2^28 per GPU", "n": n, "slice": [lo, hi],
                   "bytes_per_step_per_gpu": step_bytes,
                   "l2": "no flush: inputs larger than L2 (3.2 GB working set vs 129 MB L2)",
                   "path": rec.get("path"), "vec_bytes": rec.get("vec_bytes"),
                   "grid": rec.get("grid"), "block": rec.get("block"), "gpu": gpu_name,
                   "sms": facts.get("sms"), "l2_bytes": facts.get("l2_bytes"),
                   "driver": facts.get("driver")},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic, "peak_source": peak_src,
                     "traffic_note": traffic_note, "kernel_ms": kern_s * 1e3,
                     "kernel_ms_median": per_launch[len(per_launch) // 2] * 1e3,
                     "kernel_ms_min": per_launch[0] * 1e3, "frac_of_nominal_8tbs": achieved / 8000.0},
        "e2e": e2e,
        "gpu_launches": steps,
        "clocks": clocks,
        "parity": ("bit-exact vs the CPU oracle" if parity is True else parity),
    }
    if cpu_baseline is not None:
        line["cpu_baseline"] = cpu_baseline
    return line


def emit(aux_line, headline, out=None):
    """Print the aux line (if any), then the headline as the LAST line."""
    out = out or sys.stdout
    if aux_line is not None:
        out.write(json.dumps(aux_line) + "\n")
    text = json.dumps(headline, separators=(",", ":"))
    if len(text.encode()) > HEADLINE_MAX_BYTES:
        raise RuntimeError("headline line is %d bytes (limit %d)" % (len(text.encode()), HEADLINE_MAX_BYTES))
    out.write(text + "\n")
    out.flush()


def oracle_all_cores(oracle, metrics, a_h, b_h, want, min_s=5.0):
    """The same oracle add split into one contiguous slice per host core, run
    on that many threads (the oracle's C loop releases the GIL); a reported
    figure beside the single-core baseline."""
    from concurrent.futures import ThreadPoolExecutor
    n = a_h.size
    cores = os.cpu_count() or 1
    bounds = [(n * k // cores, n * (k + 1) // cores) for k in range(cores)]

    def part(b):
        return oracle.add("f32", a_h[b[0]:b[1]], b_h[b[0]:b[1]])

    with ThreadPoolExecutor(cores) as pool:
        t0 = time.perf_counter()
        reps = 0
        while True:
            parts = list(pool.map(part, bounds))
            reps += 1
            el = time.perf_counter() - t0
            if el >= min_s:
                break
    same = all(np.array_equal(p_.view(np.uint32), want[b[0]:b[1]].view(np.uint32))
               for p_, b in zip(parts, bounds))
    return {"value": metrics.gbps(12 * n * reps, el), "cores": cores, "matches_single_core": same}


def run_ours(args):
    import torch
    import torch.distributed as dist

    import memory_bound_elementwise_gb300 as ew
    from memory_bound_elementwise_gb300 import inputs, metrics
    from memory_bound_elementwise_gb300.shard import weak_scaling_range

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.Stream(dev)
    ew.set_path(args.path)
    ew.set_schedule(args.schedule)
    n = args.n
    lo, hi = weak_scaling_range(n, rank)

    # inputs: this rank's slice of a world*n problem, seeded per slice
    a_h = inputs.uniform(n, inputs.seed_for("add_f32", 2 * rank))
    b_h = inputs.uniform(n, inputs.seed_for("add_f32", 2 * rank + 1))
    a = torch.from_numpy(a_h).to(dev)
    b = torch.from_numpy(b_h).to(dev)
    c = torch.empty_like(a)
    L = ew.lib()
    pa, pb, pc, s = a.data_ptr(), b.data_ptr(), c.data_ptr(), stream.cuda_stream

    def step():
        st = L.ew_add(0, pa, pb, pc, n, s)
        if st != 0:
            raise ew.EwError(st, "ew_add")

    peak, peak_src = measured_peak()
    clocks = ClockSampler(local)
    clocks.start()
    nvml = NvmlClocks(pci_bus_id(torch, dev), local)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    clocks.mark("start")
    total, kern = time_launches(torch, stream, step, args.steps, 0, poll=nvml.sample)
    per_launch = sorted(time_launches.last_per_launch)
    clocks.mark("stop")
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    rec = ew.last_launch()
    rec["path"] = ew.PATH_NAMES.get(rec["path"], rec["path"])
    clk_run = clocks.stop()
    clk = nvml.summary() or clk_run
    if world > 1:
        t = torch.tensor([total, kern], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total, kern = float(t[0]), float(t[1])
    step_bytes = metrics.algorithmic_bytes("add", "f32", n)
    value = metrics.gbps(step_bytes * args.steps * world, total)
    achieved = metrics.gbps(step_bytes, kern)
    traffic, traffic_note = profiled_traffic("add_f32_v256")

    # end to end through the public API with host buffers
    e2e_steps = max(3, min(args.steps, 10))
    a_pin = torch.from_numpy(a_h).pin_memory()
    b_pin = torch.from_numpy(b_h).pin_memory()
    c_pin = torch.empty(n, dtype=torch.float32).pin_memory()
    a_d, b_d, c_d = torch.empty_like(a), torch.empty_like(b), torch.empty_like(c)

    def e2e_serial_step():
        with torch.cuda.stream(stream):
            a_d.copy_(a_pin, non_blocking=True)
            b_d.copy_(b_pin, non_blocking=True)
            ew.ew_add(a_d, b_d, c_d, stream=stream)
            c_pin.copy_(c_d, non_blocking=True)

    # pipelined: chunks of 2^24 elements; host->device copies on one stream,
    # ew_add on the timed stream, device->host copies on a third, so the two
    # copy directions and the kernels overlap
    h2d, d2h = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    chunk = min(n, 1 << 24)
    spans = [(o, min(n, o + chunk)) for o in range(0, n, chunk)]

    def e2e_step():
        start = torch.cuda.Event()
        start.record(stream)
        h2d.wait_event(start)
        d2h.wait_event(start)
        for lo_, hi_ in spans:
            with torch.cuda.stream(h2d):
                a_d[lo_:hi_].copy_(a_pin[lo_:hi_], non_blocking=True)
                b_d[lo_:hi_].copy_(b_pin[lo_:hi_], non_blocking=True)
            loaded = torch.cuda.Event()
            loaded.record(h2d)
            stream.wait_event(loaded)
            ew.ew_add(a_d[lo_:hi_], b_d[lo_:hi_], c_d[lo_:hi_], stream=stream)
            done = torch.cuda.Event()
            done.record(stream)
            d2h.wait_event(done)
            with torch.cuda.stream(d2h):
                c_pin[lo_:hi_].copy_(c_d[lo_:hi_], non_blocking=True)
        back = torch.cuda.Event()
        back.record(d2h)
        stream.wait_event(back)

    # direct: ew_add on the pinned host buffers themselves; the kernel reads A
    # and B and writes C over the CPU-GPU link (no staging copies at all)
    def e2e_direct_step():
        st = L.ew_add(0, a_pin.data_ptr(), b_pin.data_ptr(), c_pin.data_ptr(), n, s)
        if st != 0:
            raise ew.EwError(st, "ew_add (host buffers)")

    e2e_serial_total, _ = time_launches(torch, stream, e2e_serial_step, e2e_steps, 2)
    c_pin.zero_()
    e2e_piped_total, _ = time_launches(torch, stream, e2e_step, e2e_steps, 2)
    piped_ok = bool(torch.equal(c_pin, c.cpu()))
    c_pin.zero_()
    e2e_total, _ = time_launches(torch, stream, e2e_direct_step, e2e_steps, 2)
    if world > 1:
        t = torch.tensor([e2e_total, e2e_serial_total, e2e_piped_total], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_total, e2e_serial_total, e2e_piped_total = float(t[0]), float(t[1]), float(t[2])
    e2e_value = metrics.gbps(step_bytes * e2e_steps * world, e2e_total)
    e2e_ok = bool(torch.equal(c_pin, c.cpu())) and piped_ok

    # the CPU-GPU link's own ceiling in this run: copy-engine transfers of the
    # same pinned buffers host to device, device to host, and both at once
    def link_step(up, down):
        start = torch.cuda.Event()
        start.record(stream)
        for side, go, dst, src in ((h2d, up, a_d, a_pin), (d2h, down, c_pin, c_d)):
            if go:
                side.wait_event(start)
                with torch.cuda.stream(side):
                    dst.copy_(src, non_blocking=True)
                joined = torch.cuda.Event()
                joined.record(side)
                stream.wait_event(joined)
    link = {}
    for name, up, down, per in (("h2d", True, False, 4 * n), ("d2h", False, True, 4 * n), ("both", True, True, 8 * n)):
        tot, _ = time_launches(torch, stream, lambda up=up, down=down: link_step(up, down), 5, 1)
        link[name + "_gbps"] = metrics.gbps(per * 5, tot)
    e2e = {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": 8 * n, "d2h_bytes_per_step": 4 * n,
           "steps": e2e_steps, "result_matches_device": e2e_ok,
           "how": "ew_add on pinned host A, B, C: the kernel reads 8N bytes from and writes 4N bytes "
                  "to host memory over the CPU-GPU link every step",
           "link": dict(link, how="cudaMemcpyAsync of the same pinned 1 GiB buffers, one direction and "
                                  "both at once on two streams, in this run"),
           "frac_of_link_both": e2e_value / link["both_gbps"]}
    e2e_staged = {"staged_pipelined_gbps": metrics.gbps(step_bytes * e2e_steps * world, e2e_piped_total),
                  "staged_pipelined_how": "cudaMemcpyAsync H2D of A, B, ew_add on device copies, D2H of C, "
                                          "in %d chunks overlapped on three streams" % len(spans),
                  "staged_serial_gbps": metrics.gbps(step_bytes * e2e_steps * world, e2e_serial_total)}

    # parity of the headline output, then the CPU baseline (rank 0, one GPU)
    torch.cuda.synchronize()
    c_host = c.cpu().numpy()
    cpu_baseline, all_cores, parity = None, None, "unchecked"
    if rank == 0 and world == 1 and not args.no_cpu:
        import oracle
        t0 = time.perf_counter()
        reps = 0
        want = None
        while True:
            want = oracle.add("f32", a_h, b_h)
            reps += 1
            el = time.perf_counter() - t0
            if el >= 10.0 or el / reps * (reps + 1) > 30.0:
                break
        cpu_gbps = metrics.gbps(step_bytes * reps, el)
        parity = True if np.array_equal(want.view(np.uint32), c_host.view(np.uint32)) else "MISMATCH"
        all_cores = oracle_all_cores(oracle, metrics, a_h, b_h, want)
        cpu_baseline = {"value": cpu_gbps, "unit": "GB/s", "cores": 1, "kind": "oracle",
                        "sample": "%d full passes over the N=2^28 inputs (%.1f s)" % (reps, el),
                        "cpu": host_cpu_model(), "all_cores_value": all_cores["value"],
                        "all_cores_cores": all_cores["cores"]}
        del want
    elif not args.no_cpu:  # other ranks and multi-GPU runs: seeded windows of the output
        chk = Parity(True)
        pr = True
        for w0, w1 in parity_windows(n, 1234 + rank):
            if first_mismatch(c_host[w0:w1], chk.oracle.add("f32", a_h[w0:w1], b_h[w0:w1]), "f32", True) is not None:
                pr = "MISMATCH"
                break
        parity = pr
    if world > 1:
        t = torch.tensor([1.0 if parity is True else 0.0], dtype=torch.float64, device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MIN)
        if parity is True and float(t[0]) < 1.0:
            parity = "MISMATCH on another rank"

    aux_line = None
    if rank == 0:
        aux_line = {"aux_of": METRIC, "e2e_staged": e2e_staged, "clocks_whole_run": clk_run,
                    "peak_source": peak_src, "baseline": PAGE_BASELINE,
                    "device": {"gpu": torch.cuda.get_device_name(dev), **device_facts(torch, dev)}}
        if all_cores is not None:
            aux_line["cpu_all_cores"] = all_cores
    if not args.no_aux and world == 1:
        del a_pin, b_pin, c_pin, a_d, b_d, c_d
        facts = device_facts(torch, dev)
        aux = Aux(torch, ew, inputs, metrics, stream, peak, dev, Parity(not args.no_cpu), facts.get("l2_bytes"))
        aux_line["aux"] = aux.run()
    if rank == 0:
        facts = device_facts(torch, dev)
        line = headline_line(
            value=value, parity=parity, world=world, steps=args.steps, warmup=args.warmup, total_s=total,
            n=n, lo=lo, hi=hi, step_bytes=step_bytes, rec=rec, facts=facts,
            gpu_name=torch.cuda.get_device_name(dev), achieved=achieved, peak=peak, peak_src=peak_src,
            traffic=traffic, traffic_note=traffic_note, kern_s=kern, per_launch=per_launch, e2e=e2e,
            clocks=clk, cpu_baseline=cpu_baseline)
        emit(aux_line, line)
    if world > 1:
        dist.destroy_process_group()


def main():
    args = parse()
    if args.profile_case:
        run_profile_case(args)
    elif args.impl == "reference":
        run_reference(args)
    elif args.ab == "widths":
        run_ab_widths(args)
    elif args.ab == "gather":
        run_ab_gather(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
