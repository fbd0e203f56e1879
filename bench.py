#!/usr/bin/env python
"""Benchmark: selective-scan forward (and the decode step) on B300.

One "step" is one pass of the whole hot path over one batch of synthetic input
already resident in HBM: a single ``ssm_scan_fwd`` call over the workload
(softplus step size, discretisation, recurrence, readout, gate, last state),
or, for the decode workload, the 1024 sequential ``ssm_state_update`` calls (captured once in
a CUDA graph and replayed; plain launches are reported beside).
Prints one JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload KEY] [--impl ours|reference]

Under torchrun (N > 1) every rank runs the same per-GPU workload on its own
GPU (weak scaling: the channels of a model shard independently, with no
exchange) and the slowest rank's time is reported.  ``--impl reference`` times
the float64 CPU oracle on a bounded sample of the same workload instead.
"""
from __future__ import annotations

import argparse
import json
import os
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from inputgen import workloads as W  # noqa: E402

PEAKS_FILE = os.path.join(ROOT, "MEASURED_PEAKS.json")
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "dram_traffic.json")
# The kernel sources each workload kind runs; DRAM counters taken under another version of them
# are stale.
KERNEL_SOURCES = {"scan": ("ssm_scan_fwd.cu", "ssm_device.cuh"),
                  "decode": ("ssm_decode.cu", "ssm_device.cuh"),
                  "ssd": ("ssm_ssd.cu", "ssm_ssd_gram.cu", "ssm_device.cuh")}
FALLBACK_HBM_GBS = 6400.0
NOMINAL_HBM_GBS = 7700.0  # B300 HBM3e nominal, reported beside the measured-copy fraction
SM_MAX_MHZ_NOMINAL = 2032.0
# Per-SM rates of the pipes the scan uses (operations per clock), measured on B300 with a
# throughput probe: FP32 FFMA/FMUL/FADD 128; MUFU ex2 32, lg2 and rcp 16.  The MUFU
# operations share one pipe (a 1:1 mix of ex2 and rcp runs at 19.9 per clock, what one shared
# pipe gives, not the 32 of two separate ones), so the bound counts MUFU "slots": an ex2 takes
# one, a lg2 or rcp two, at 32 slots per clock.
FP32_PER_CLK, MUFU_SLOTS_PER_CLK = 128.0, 32.0
L2_FLUSH_BYTES = 512 << 20


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default="long", choices=sorted(W.WORKLOADS),
                    help="default: the long-context scan (1 x 1,048,576 x 2048 x 16, bf16 I/O), the "
                         "largest single-GPU workload")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=8)
    ap.add_argument("--pass", dest="which", default="forward", choices=["forward", "backward", "conv"],
                    help="forward: ssm_scan_fwd (default); backward: ssm_scan_bwd (gradients); "
                         "conv: ssm_scan_fwd_conv (causal conv1d + SiLU fused in front)")
    ap.add_argument("--no-graph", action="store_true",
                    help="decode: report plain launches only (default: the step's launches "
                         "replayed as a CUDA graph, plain launches beside)")
    ap.add_argument("--decode-steps", type=int, default=None,
                    help="decode steps per bench step (default: the workload's 1024); "
                         "only for small profiling captures")
    return ap.parse_args()


# ---------------------------------------------------------------------------------------------
# Algorithmic work per workload (the roofline numerators).

def algorithmic_bytes(w: W.Workload) -> float:
    """HBM bytes a perfect implementation must move for one step."""
    s = 2 if w.bf16 else 4
    N = w.d_state
    params = w.d_inner * (N + 2) * 4                      # A, D, delta_bias (fp32)
    if w.decode:
        per_tok = w.batch * w.d_inner * (4 * s + 2 * N * 4)   # u, delta, z, y + state read/write
        per_tok += w.batch * 2 * N * s                       # B, C rows
        return float(w.L * (per_tok + params))
    acts = w.batch * w.L * w.d_inner * 4 * s             # u, delta, z read; y write
    bc = w.batch * w.L * 2 * N * s                       # B, C rows
    last = w.batch * w.d_inner * N * 4                   # last_state write
    return float(acts + bc + params + last)


def ssd_algorithmic_bytes(w: W.Workload) -> float:
    """Chunked SSD: read x, z (bf16, per channel), dt (bf16, per head), B, C (bf16, shared by
    the heads); write y (bf16) and the last state (fp32); A_head, dt_bias, D once."""
    acts = w.batch * w.L * w.d_inner * 3 * 2
    dt = w.batch * w.L * w.heads * 2
    bc = w.batch * w.L * 2 * w.d_state * 2
    last = w.batch * w.d_inner * w.d_state * 4
    return float(acts + dt + bc + last + (2 * w.heads + w.d_inner) * 4)


SSD_Q = 64  # chunk length of the tensor-core form


def ssd_flops(w: W.Workload) -> float:
    """Tensor-core FLOPs of the chunked form, each product counted once (Q = 64, P = 64):
    per (batch, chunk) the Gram matrix C B^T (2 Q^2 N; the same for every head, since B and C
    are shared), and per (batch, head, chunk) the local state X^T (w B) (2 Q P N), the
    carried-state readout C H^T (2 Q N P) and the masked mix M X (2 Q^2 P)."""
    P, N, Q = w.d_inner // w.heads, w.d_state, SSD_Q
    chunks = -(-w.L // Q)
    per_head = 2 * Q * P * N + 2 * Q * N * P + 2 * Q * Q * P
    return float(w.batch * chunks * (2 * Q * Q * N + w.heads * per_head))


def bwd_algorithmic_bytes(w: W.Workload) -> float:
    """Backward: read u, delta, z, dy, B, C (io dtype), write du, ddelta, dz (io dtype) and
    dB, dC (fp32); A, D, bias and their gradients once."""
    s = 2 if w.bf16 else 4
    N = w.d_state
    acts = w.batch * w.L * w.d_inner * 7 * s
    bc = w.batch * w.L * N * (2 * s + 2 * 4)
    params = w.d_inner * (N + 2) * 4 * 2
    return float(acts + bc + params)


def bwd_alu_clocks_per_element(N: int) -> float:
    """Backward lower bound per element: recomputing the state (4 FP32 + 1 ex2 per state) and
    the reverse step (per state: the adjoint FMA, dA's product and ex2, the two terms of the
    step-size gradient, the A-gradient FMA, the u-gradient FMA, the B and C partials and the
    carry: 11 FP32 + 1 ex2), plus ~16 FP32, 4 ex2 and 4 lg2/rcp (two MUFU slots each) per
    element."""
    fp32 = 15 * N + 16
    mufu = 2 * N + 4 + 2 * 4
    return max(fp32 / FP32_PER_CLK, mufu / MUFU_SLOTS_PER_CLK)


def alu_clocks_per_element(N: int, conv: bool = False) -> float:
    """Lower bound on SM clocks per (b, t, d) element from the arithmetic the method needs:
    per state n: delta*A, exp, (delta u)*B_n, the FMA of the recurrence and the FMA of the
    readout (4 FP32 + 1 ex2); per element: delta*u, bias add, D*u, gate multiply, the sigmoid's
    1 + e^-z and z * (.) (6 FP32), the exps of softplus and sigmoid (2 ex2), the sigmoid's
    reciprocal (2 MUFU slots), and softplus's log1p, which costs either a MUFU lg2 (2 slots) or
    about 10 FP32 operations of a polynomial: the bound takes the cheaper assignment.  With the
    conv1d + SiLU in front: 4 more FMA, 3 more FP32 and one more exp and reciprocal.  FP32 and
    MUFU are separate pipes; the slower one binds."""
    fp32 = 4 * N + 6 + (7 if conv else 0)
    mufu = N + 2 + 2 + (3 if conv else 0)
    log_on_mufu = max(fp32 / FP32_PER_CLK, (mufu + 2) / MUFU_SLOTS_PER_CLK)
    log_on_fma = max((fp32 + 10) / FP32_PER_CLK, mufu / MUFU_SLOTS_PER_CLK)
    return min(log_on_mufu, log_on_fma)


def workload_kind(w: W.Workload) -> str:
    return "ssd" if w.heads else "decode" if w.decode else "scan"


def kernel_source_hash(kind: str) -> str:
    """Hash of the kernel sources of one workload kind."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kind]:
        with open(os.path.join(ROOT, "selective_state_space_161_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def measured_traffic(w: W.Workload):
    """DRAM bytes (read + write) per step from the committed ncu capture of this workload,
    or None if there is none or the kernels changed since it was taken."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f).get(w.key)
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_hash") != kernel_source_hash(workload_kind(w)):
        return None
    return float(rec["dram_bytes_per_step"])


def load_peaks():
    try:
        with open(PEAKS_FILE) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p.get("sm_max_mhz", SM_MAX_MHZ_NOMINAL)), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, SM_MAX_MHZ_NOMINAL, "fallback"


# ---------------------------------------------------------------------------------------------
# Clock sampling (NVML, read-only) during the timed region.

class _Nvml:
    """Read-only NVML queries through ctypes (libnvidia-ml ships with the driver)."""

    def __init__(self, index: int):
        import ctypes
        self.ct = ctypes
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise RuntimeError("nvmlInit failed")
        self.h = ctypes.c_void_p()
        if self.lib.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
            raise RuntimeError("nvmlDeviceGetHandleByIndex failed")
        self._reasons = (getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
                         or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons)

    def _uint(self, fn, *args):
        v = self.ct.c_uint()
        if fn(self.h, *args, self.ct.byref(v)) != 0:
            raise RuntimeError(f"{fn.__name__} failed")
        return v.value

    def sm_clock(self):
        return self._uint(self.lib.nvmlDeviceGetClockInfo, 1)  # NVML_CLOCK_SM

    def sm_max_clock(self):
        return self._uint(self.lib.nvmlDeviceGetMaxClockInfo, 1)

    def power_w(self):
        return self._uint(self.lib.nvmlDeviceGetPowerUsage) / 1000.0

    def reasons(self):
        v = self.ct.c_ulonglong()
        if self._reasons(self.h, self.ct.byref(v)) != 0:
            return 0
        return v.value


class ClockSampler:
    """Samples SM clock, power and clock-event reasons in a thread during the timed region."""
    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown", 0x100: "display_clock_setting",
    }

    def __init__(self, index: int, period_s: float = 0.002):
        self.samples, self.power, self.reasons, self.max_mhz = [], [], 0, None
        self.period, self.error = period_s, None
        self._stop = threading.Event()
        self._thread = None
        try:
            self._nv = _Nvml(index)
            self.max_mhz = self._nv.sm_max_clock()
        except Exception as e:  # noqa: BLE001 - clocks are then reported as unavailable
            self.error = f"{type(e).__name__}: {e}"
            self._nv = None

    def _sample(self):
        self.samples.append(self._nv.sm_clock())
        self.power.append(self._nv.power_w())
        self.reasons |= self._nv.reasons()

    def _loop(self):
        while not self._stop.is_set():
            try:
                self._sample()
            except Exception as e:  # noqa: BLE001
                self.error = f"{type(e).__name__}: {e}"
                return
            time.sleep(self.period)

    def start(self):
        if self._nv is not None:
            self._thread = threading.Thread(target=self._loop, daemon=True)
            self._thread.start()

    def stop(self):
        if self._thread is not None:
            self._stop.set()
            self._thread.join()

    def summary(self):
        if self._nv is None or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"],
                    "error": self.error}
        names = [n for bit, n in self.REASONS.items() if self.reasons & bit and n != "gpu_idle"]
        return {"sm_mhz": float(np.median(self.samples)), "sm_max_mhz": self.max_mhz,
                "sm_mhz_min": float(min(self.samples)), "power_w_max": float(max(self.power)),
                "samples": len(self.samples), "reasons": names}


# ---------------------------------------------------------------------------------------------
# Our implementation.

class ScanStep:
    """One step = one ssm_scan_fwd call over the whole workload."""

    input_names = ("u", "delta", "z", "B", "C", "A", "D", "delta_bias")

    def __init__(self, w, dev, ssm, torch):
        self.w, self.dev, self.ssm, self.torch = w, dev, ssm, torch
        self.y = torch.empty_like(dev["u"])
        self.last = torch.empty((w.batch, w.d_inner, w.d_state), dtype=torch.float32, device="cuda")
        io = ssm.SSM_BF16 if w.bf16 else ssm.SSM_F32
        nbytes = ssm.ssm_scan_fwd_workspace_size(w.batch, w.L, w.d_inner, w.d_state, io)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
        self.launches = 1  # one launch per call (time chunks joined by the look-back inside it)

    def workspace(self):
        return self.ws

    def call(self, d, y, last, ws, stream=None):
        self.ssm.ssm_scan_fwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                              d["delta_bias"], True, y, last, ws, stream)

    def __call__(self, stream=None):
        self.call(self.dev, self.y, self.last, self.ws, stream)


class SsdStep(ScanStep):
    """One step = one ssm_ssd_fwd call: the chunked tensor-core form over the whole workload
    (one A and one step size per head of 64 channels)."""

    input_names = ("x", "z", "dt", "B", "C", "A_head", "dt_bias", "D")

    def __init__(self, w, dev, ssm, torch):
        self.w, self.dev, self.ssm = w, dev, ssm
        self.y = torch.empty_like(dev["x"])
        self.last = torch.empty((w.batch, w.d_inner, w.d_state), dtype=torch.float32, device="cuda")
        nbytes = ssm.ssm_ssd_fwd_workspace_size(w.batch, w.L, w.d_inner, w.heads, w.d_state)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda") if nbytes else None
        self.launches = 2  # the chunk Gram matrices (tensor cores), then the heads

    def workspace(self):
        return self.ws

    def call(self, d, y, last, ws, stream=None):
        self.ssm.ssm_ssd_fwd(d["x"], d["dt"], d["A_head"], d["B"], d["C"], d["D"], d["z"],
                             d["dt_bias"], True, y, last, ws, stream)


class ConvScanStep(ScanStep):
    """One step = one ssm_scan_fwd_conv call: u = silu(conv1d(x)) fused in front of the scan
    (x: the workload's u tensor; d_conv = 4 taps ~ N(0, 0.5), bias ~ N(0, 0.2), seeded)."""

    def __init__(self, w, dev, ssm, torch):
        super().__init__(w, dev, ssm, torch)
        import inputgen
        self.cw = torch.from_numpy(inputgen.normal(w.seed, 10, 0.0, 0.5, 0, w.d_inner * 4, False)
                                   .reshape(w.d_inner, 4)).cuda()
        self.cb = torch.from_numpy(inputgen.normal(w.seed, 11, 0.0, 0.2, 0, w.d_inner, False)).cuda()

    def __call__(self, stream=None):
        d = self.dev
        self.ssm.ssm_scan_fwd_conv(d["u"], self.cw, self.cb, d["delta"], d["A"], d["B"], d["C"], d["D"],
                                   d["z"], d["delta_bias"], True, None, self.y, self.last, None,
                                   self.ws, stream)


class BackwardStep:
    """One step = one ssm_scan_bwd call (all gradients) for dy ~ N(0, 1) (seeded)."""

    def __init__(self, w, dev, ssm, torch):
        import inputgen
        self.dev, self.ssm = dev, ssm
        self.dy = torch.empty_like(dev["u"])
        inputgen.dev_fill_normal(w.seed, 9, 0.0, 1.0, 0, self.dy.numel(), w.bf16, self.dy.data_ptr(),
                                 torch.cuda.current_stream().cuda_stream)
        f32 = dict(dtype=torch.float32, device="cuda")
        N = w.d_state
        self.g = dict(du=torch.empty_like(dev["u"]), ddelta=torch.empty_like(dev["u"]),
                      dz=torch.empty_like(dev["u"]), dA=torch.empty((w.d_inner, N), **f32),
                      dB=torch.empty((w.batch, w.L, N), **f32), dC=torch.empty((w.batch, w.L, N), **f32),
                      dD=torch.empty(w.d_inner, **f32), ddelta_bias=torch.empty(w.d_inner, **f32))
        io = ssm.SSM_BF16 if w.bf16 else ssm.SSM_F32
        nbytes = ssm.ssm_scan_bwd_workspace_size(w.batch, w.L, w.d_inner, N, io)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        # the forward recompute, the gradients, and the reverse summaries if the plan needs them
        self.launches = ssm.ssm_scan_bwd_launches(w.batch, w.L, w.d_inner, N, io)

    def __call__(self, stream=None):
        d, g = self.dev, self.g
        self.ssm.ssm_scan_bwd(d["u"], d["delta"], d["A"], d["B"], d["C"], d["D"], d["z"],
                              d["delta_bias"], True, None, self.dy, None, g["du"], g["ddelta"],
                              g["dA"], g["dB"], g["dC"], g["dD"], g["dz"], g["ddelta_bias"], None,
                              self.ws, stream)


class DecodeStep:
    """One step = the workload's sequential single-token decode steps.  With layers > 1 the
    steps rotate over that many state buffers (launch s updates buffer s % layers), as in a
    model whose layers take turns: between two updates of a buffer the other layers' states
    (84 MB each at 256 x 5120 x 16) pass through L2, so no state is still cached."""

    def __init__(self, w, dev, ssm, torch, layers=1):
        self.w, self.dev, self.ssm = w, dev, ssm
        self.states = [dev["state0"].clone() for _ in range(layers)]
        self.y = torch.empty((w.batch, w.d_inner), dtype=dev["u"].dtype, device="cuda")
        self.steps = dev["u"].shape[0]
        self.launches = self.steps

    def __call__(self, stream=None):
        d = self.dev
        for s in range(self.steps):
            self.ssm.ssm_state_update(self.states[s % len(self.states)], d["u"][s], d["delta"][s],
                                      d["A"], d["B"][s], d["C"][s], d["D"], d["z"][s], self.y,
                                      d["delta_bias"], True, stream)


def time_decode_graph(step, flush, torch, steps):
    """The same decode step (all its sequential launches) captured once in a CUDA graph and
    replayed: launch overhead off the host, timed like the plain launches (L2 flushed between
    timed replays, CUDA events on the replay stream).  The state keeps evolving across
    replays, as it does across plain steps."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # one eager step on the side stream before capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        step()
    for _ in range(2):
        g.replay()
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for e0, e1 in ev:
        flush.zero_()
        e0.record(cur)
        g.replay()
        e1.record(cur)
    torch.cuda.synchronize()
    t = [e0.elapsed_time(e1) for e0, e1 in ev]
    return {"ms_per_step": float(np.mean(t)), "ms_per_step_median": float(np.median(t))}


def run_e2e(w, step, torch, steps):
    """Same metric through the public call with pinned host buffers: every step copies its
    inputs host->device, runs the step's entry point and copies y and last_state back.  Two
    streams, each with its own device buffers and workspace, alternate steps, so step k+1's
    input copy overlaps step k's kernel and output copy (PCIe is full duplex); every step
    still carries its own copies."""
    if w.decode:
        return None
    names = step.input_names
    host = {k: step.dev[k].cpu().pin_memory() for k in names}
    slots = []
    for _ in range(2):
        ws = step.workspace()
        slots.append(dict(stream=torch.cuda.Stream(),
                          d={k: torch.empty_like(step.dev[k]) for k in names},
                          y=torch.empty_like(step.y), last=torch.empty_like(step.last),
                          ws=torch.empty_like(ws) if ws is not None else None,
                          y_h=torch.empty(step.y.shape, dtype=step.y.dtype, pin_memory=True),
                          last_h=torch.empty(step.last.shape, dtype=step.last.dtype, pin_memory=True)))
    h2d = sum(t.numel() * t.element_size() for t in host.values())
    d2h = step.y.numel() * step.y.element_size() + step.last.numel() * 4
    cur = torch.cuda.current_stream()

    def one(k):
        sl = slots[k % 2]
        with torch.cuda.stream(sl["stream"]):
            for n in names:
                sl["d"][n].copy_(host[n], non_blocking=True)
            step.call(sl["d"], sl["y"], sl["last"], sl["ws"], sl["stream"].cuda_stream)
            sl["y_h"].copy_(sl["y"], non_blocking=True)
            sl["last_h"].copy_(sl["last"], non_blocking=True)

    def run(n_steps):
        for sl in slots:
            sl["stream"].wait_stream(cur)
        for k in range(n_steps):
            one(k)
        for sl in slots:
            cur.wait_stream(sl["stream"])

    run(2)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(cur)
    run(steps)
    e1.record(cur)
    torch.cuda.synchronize()
    ms = e0.elapsed_time(e1) / steps
    return {"value": w.elements / (ms * 1e-3), "unit": "elements/s", "ms_per_step": ms,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "pipelining": "2 streams: a step's host-to-device copies overlap the previous step's "
                          "kernel and device-to-host copies"}


def oracle_sample_rate(w, budget_s: float, threads: int | None = None):
    """Elements/s of the float64 oracle on a bounded sample of the workload: a subset of
    channels over the full sequence (all batches), sized to roughly budget_s of work."""
    import oracle
    oracle.build()
    threads = threads or oracle.max_threads()
    if w.decode:
        steps = 8
        probe = W.host_decode_inputs(w, steps, d_sel=np.arange(64))
        t0 = time.perf_counter()
        st = probe["state0"]
        for s in range(steps):
            _, st = oracle.state_update(st, probe["u"][s], probe["delta"][s], probe["A"],
                                        probe["B"][s], probe["C"][s], D=probe["D"], z=probe["z"][s],
                                        delta_bias=probe["delta_bias"], nthreads=threads)
        el = steps * w.batch * 64
        return el / (time.perf_counter() - t0), threads, \
            f"{steps} decode steps x {w.batch} batch x 64 of {w.d_inner} channels"
    T = min(w.L, 1 << 16)
    d_try = max(1, min(w.d_inner, threads))
    if w.heads:  # the chunked form's oracle is the per-channel scan with head-broadcast operands
        def inputs(d_cnt):
            return W.host_ssd_inputs(w, d_sel=np.arange(d_cnt))
    else:
        def inputs(d_cnt):
            return W.host_scan_inputs(w, d_sel=np.arange(d_cnt), t_count=T)
    x = inputs(d_try)
    t0 = time.perf_counter()
    oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                    delta_bias=x["delta_bias"], nthreads=threads)
    rate = w.batch * T * d_try / (time.perf_counter() - t0)
    d_cnt = int(min(w.d_inner, max(d_try, rate * budget_s / (w.batch * T))))
    x = inputs(d_cnt)
    t0 = time.perf_counter()
    oracle.scan_fwd(x["u"], x["delta"], x["A"], x["B"], x["C"], D=x["D"], z=x["z"],
                    delta_bias=x["delta_bias"], nthreads=threads)
    dt = time.perf_counter() - t0
    return w.batch * T * d_cnt / dt, threads, \
        f"{w.batch} batch x {T} steps x {d_cnt} of {w.d_inner} channels (float64, {dt:.1f} s)"


def max_over_ranks(value: float, world: int, device=None) -> float:
    """The largest value across ranks (barrier included); the value itself on one rank."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_rate(elements_per_rank: int, world: int, ms_max: float) -> float:
    """Weak scaling: every rank processed its own workload; the slowest rank sets the time."""
    return world * elements_per_rank / (ms_max * 1e-3)


def roofline(w, ms_per_step, hbm_gbs, sm_mhz, sms, peak_src, traffic=None, which="forward"):
    el_rate = w.elements / (ms_per_step * 1e-3)
    nbytes = bwd_algorithmic_bytes(w) if which == "backward" else algorithmic_bytes(w)
    clocks = (bwd_alu_clocks_per_element(w.d_state) if which == "backward"
              else alu_clocks_per_element(w.d_state, conv=which == "conv"))
    if which == "ssd":
        nbytes = ssd_algorithmic_bytes(w)
        achieved = nbytes / (ms_per_step * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": traffic, "algorithmic_bytes": nbytes,
                "peak_source": f"{peak_src} copy bandwidth",
                "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
                "tensor_tflops": ssd_flops(w) / (ms_per_step * 1e-3) / 1e12}
    t_hbm = nbytes / (hbm_gbs * 1e9)
    t_alu = w.elements * clocks / (sms * sm_mhz * 1e6)
    if t_hbm >= t_alu:
        achieved = nbytes / (ms_per_step * 1e-3) / 1e9
        return {"bound": "hbm", "achieved": achieved, "peak": hbm_gbs, "unit": "GB/s",
                "frac": achieved / hbm_gbs, "traffic": traffic,
                "algorithmic_bytes": algorithmic_bytes(w),
                "peak_source": f"{peak_src} copy bandwidth",
                "frac_of_nominal_hbm": achieved / NOMINAL_HBM_GBS,
                "alu_frac": el_rate * t_alu / w.elements}
    peak = w.elements / t_alu / 1e9
    return {"bound": "alu", "achieved": el_rate / 1e9, "peak": peak, "unit": "Gelem/s",
            "frac": el_rate / 1e9 / peak, "traffic": traffic,
            "algorithmic_bytes": algorithmic_bytes(w),
            "peak_source": (f"{sms} SMs x {sm_mhz:.0f} MHz, per-element FP32 and MUFU op counts at the "
                            f"measured rates {FP32_PER_CLK:.0f} FP32 and {MUFU_SLOTS_PER_CLK:.0f} MUFU "
                            f"slots per clock per SM (ex2 one slot, lg2/rcp two, one shared pipe)"),
            "hbm_frac": algorithmic_bytes(w) / (ms_per_step * 1e-3) / 1e9 / hbm_gbs,
            "hbm_frac_of_nominal": algorithmic_bytes(w) / (ms_per_step * 1e-3) / 1e9 / NOMINAL_HBM_GBS}


def bench_config(w, which, world):
    """The config dict of a bench line (identical for our arm and the reference arm)."""
    return {"workload": w.desc, "batch": w.batch,
            ("steps" if w.decode else "seq_len"): w.L, "d_inner": w.d_inner,
            "d_state": w.d_state, "io_dtype": "bf16" if w.bf16 else "f32",
            **({"heads": w.heads, "chunk": SSD_Q} if w.heads else {}),
            "pass": which,
            "parallelism": f"replica per GPU x{world}" if world > 1 else "single GPU",
            "l2": f"flushed between timed steps ({L2_FLUSH_BYTES >> 20} MiB write)"}


def main_ours(args, rank, world, local_rank):
    import torch
    import selective_state_space_161_b300 as ssm

    torch.cuda.set_device(local_rank)
    ssm.load_library()
    w = W.WORKLOADS[args.workload]
    if w.decode and args.decode_steps:
        import dataclasses
        w = dataclasses.replace(w, L=args.decode_steps)
    if w.heads:
        args.which = "ssd"
        dev = W.device_ssd_inputs(w)
    else:
        dev = W.device_inputs(w)
    if w.heads:
        step = SsdStep(w, dev, ssm, torch)
    elif w.decode:
        step = DecodeStep(w, dev, ssm, torch)
    elif args.which == "backward":
        step = BackwardStep(w, dev, ssm, torch)
    elif args.which == "conv":
        step = ConvScanStep(w, dev, ssm, torch)
    else:
        step = ScanStep(w, dev, ssm, torch)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    sms = torch.cuda.get_device_properties(local_rank).multi_processor_count

    for _ in range(max(args.warmup, 0)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = ClockSampler(local_rank)
    events = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
    torch.cuda.synchronize()
    clocks.start()
    for e0, e1 in events:
        flush.zero_()            # evict the previous step's data from L2 (untimed)
        e0.record(stream)
        step()
        e1.record(stream)
    torch.cuda.synchronize()
    clocks.stop()
    times = [e0.elapsed_time(e1) for e0, e1 in events]
    ms = max_over_ranks(float(np.mean(times)), world, "cuda")
    ms_median = max_over_ranks(float(np.median(times)), world, "cuda")

    plain = None
    if w.decode and not args.no_graph:
        # decode: the step's launches replayed as one CUDA graph are the reported figure; the
        # plain launches just timed are kept beside it
        graph = time_decode_graph(step, flush, torch, args.steps)
        plain = {"ms_per_step": ms, "ms_per_step_median": ms_median,
                 "value": whole_job_rate(w.elements, world, ms), "how": "plain launches"}
        ms = max_over_ranks(graph["ms_per_step"], world, "cuda")
        ms_median = max_over_ranks(graph["ms_per_step_median"], world, "cuda")
        # the same launches over 4 rotating state buffers: every state comes from HBM
        cold_step = DecodeStep(w, dev, ssm, torch, layers=4)
        cold = time_decode_graph(cold_step, flush, torch, args.steps)
        cold_ms = max_over_ranks(cold["ms_per_step"], world, "cuda")
        del cold_step

    e2e = None
    if not args.no_e2e and not w.decode and args.which in ("forward", "ssd"):
        e2e = run_e2e(w, step, torch, args.e2e_steps)
        if e2e is not None and world > 1:
            e2e["ms_per_step"] = max_over_ranks(e2e["ms_per_step"], world, "cuda")
            e2e["value"] = whole_job_rate(w.elements, world, e2e["ms_per_step"])

    if rank != 0:
        return
    hbm_gbs, _, peak_src = load_peaks()
    clk = clocks.summary()
    sm_mhz_peak = float(clk["sm_max_mhz"] or SM_MAX_MHZ_NOMINAL)
    out = {
        "metric": metric_name(w, args.which),
        "value": whole_job_rate(w.elements, world, ms),
        "unit": "elements/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "ms_per_step_median": ms_median,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16" if w.heads else "f32",
        "dtype_note": ("bf16 tensor-core products (hi+lo split operands), f32 accumulation"
                       if w.heads else "f32 state and arithmetic, " + ("bf16" if w.bf16 else "f32") + " I/O"),
        "data": "synthetic (seeded; recipe in inputgen/workloads.py)",
        "config": bench_config(w, args.which, world),
        "roofline": roofline(w, ms, hbm_gbs, sm_mhz_peak, sms, peak_src,
                             measured_traffic(w) if args.which in ("forward", "ssd") else None,
                             args.which),
        "gpu_launches": step.launches * args.steps,
        "clocks": clk,
    }
    if e2e is not None:
        out["e2e"] = e2e
    if plain is not None:
        out["config"]["launch"] = "CUDA graph of the step's launches, replayed"
        out["plain_launches"] = plain
        hbm_gbs_cold = algorithmic_bytes(w) / (cold_ms * 1e-3) / 1e9
        out["l2_cold"] = {"ms_per_step": cold_ms, "value": whole_job_rate(w.elements, world, cold_ms),
                          "unit": "elements/s", "achieved_gbs": hbm_gbs_cold,
                          "frac": hbm_gbs_cold / hbm_gbs,
                          "how": "launch s updates state buffer s % 4 (4 layers' states, 336 MB, "
                                 "rotate through L2), CUDA graph replayed like the main figure"}
    if not args.no_cpu_baseline:
        rate, cores, sample = oracle_sample_rate(w, budget_s=12.0)
        rate1, _, sample1 = oracle_sample_rate(w, budget_s=3.0, threads=1)
        out["cpu_baseline"] = {"value": rate, "unit": "elements/s", "cores": cores,
                               "kind": "oracle", "sample": sample,
                               "single_thread": {"value": rate1, "sample": sample1}}
    print(json.dumps(out), flush=True)


def metric_name(w, which):
    if w.decode:
        return "decode elements/s (B*d_inner*steps)"
    if which == "backward":
        return "scan backward elements/s (B*L*d_inner)"
    if w.heads:
        return "chunked SSD scan elements/s (B*L*d_inner)"
    return "scan elements/s (B*L*d_inner)"


def main_reference(args, rank, world):
    """The float64 oracle on the host cores: each step is a bounded sample of the workload."""
    if rank != 0:
        return
    w = W.WORKLOADS[args.workload]
    rates = []
    info = None
    for i in range(args.warmup + args.steps):
        rate, cores, sample = oracle_sample_rate(w, budget_s=1.5)
        if i >= args.warmup:
            rates.append(rate)
            info = (cores, sample)
    value = float(np.median(rates))
    out = {
        "impl": "reference",
        "metric": metric_name(w, "ssd" if w.heads else "forward"),
        "value": value, "unit": "elements/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": w.elements / value * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded; recipe in inputgen/workloads.py)",
        "config": bench_config(w, "ssd" if w.heads else args.which, world),
        "cpu_baseline": {"value": value, "unit": "elements/s", "cores": info[0], "kind": "oracle",
                         "sample": info[1]},
        "e2e": {"value": value, "unit": "elements/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out), flush=True)


def main():
    args = parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        main_reference(args, rank, world)
        return
    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    try:
        main_ours(args, rank, world, local_rank)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
