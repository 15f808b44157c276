#!/usr/bin/env python
"""Throughput of the chunked SSD scan (fwd + bwd) on one or more GPUs.

A step is one forward and one backward pass (ssd_fwd then ssd_bwd: the whole
hot path, the backward recomputing what it needs from the inputs, so nothing
is kept between the two, as in the pages' chunked records; --saved-states
times ssd_fwd_save then ssd_bwd_saved instead, the backward reading the
forward's segment states) over the g2h8_d128 L=8192 long-memory workload: B=4, G=2, H=8,
L=8192, dk=dv=128, chunk 64, fp32 storage, seeded synthetic inputs.  The
metric is tokens/s with tokens = B*L*H per step.  Prints ONE JSON line
(rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--path tc|simt]
  python bench.py --impl reference ...   # the float64 CPU oracle, timed on host cores

Under torchrun each rank runs the full workload on its own GPU (the units --
batch entries and groups -- are independent, so there is no collective on the
data path); value is the tokens of all ranks over the slowest rank's time.
"""
import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "SSD fwd / fwd_bwd tokens/s (B·L·H) at 1 GB300 and % of roofline vs oracle"
WORKLOAD = "g2h8_d128_L8192_long"
# chunked fwd_bwd, g2h8_d128, seq 8192 on the "kernel_ssd_gpu.json" benchmark
# page (RTX 3090): 11.883 ms per call -> B*L*H / t tokens/s
PAGE_FWD_BWD_MS = {"g2h8_d128_L8192_long": 11.883, "g2h8_d128_L2048": 3.210,
                   "g1h24_dk128_dv64_L8192": 10.695, "g1h1_d128_L512": 0.2519,
                   "g2h4_dk48_dv40_L2048": 0.9683}
PAGE_FWD_MS = {"g2h8_d128_L8192_long": 4.182, "g2h8_d128_L2048": 1.170,
               "g1h24_dk128_dv64_L8192": 3.461, "g1h1_d128_L512": 0.08903,
               "g2h4_dk48_dv40_L2048": 0.3709}
# the same page's memory records for impl "chunked", g2h8_d128 (RTX 3090, 24 GB):
# peak MB of fwd / fwd_bwd at seq 8192, and the largest seq (doubling) that ran
PAGE_PEAK_MB = {"fwd": 1128.0, "fwd_bwd": 1323.007568359375}
PAGE_MAX_LEN = 65536
MiB = 1 << 20


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        d = json.load(open(p))
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"])),
                "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
                "source": "fallback"}


# DRAM bytes (read + write) per launch of each kernel at the g2h8_d128 L=8192
# long-memory workload, from one ncu capture of the launch list
# (gpu__time_duration.sum, dram__bytes_read.sum, dram__bytes_write.sum) of the
# kernels as they stood then.  Each group names the commit of the capture and
# the SHA-256 (first 16 hex digits) of the kernel source it measured: when the
# file in the tree no longer hashes to that, the group's figures no longer
# describe the kernels and the bench line reports traffic null, saying why.
TRAFFIC_GROUPS = {
    "tc.": {"source": "ssd_chunked_scan_gb300/csrc/tc.cu", "sha16": "c7871499ec73c5ad", "commit": "0112b14",
            "bytes": {
                "tc.seg_state": 172355072,
                "tc.seg_state_dq": 169376768,
                "tc.seg_state_dk": 169300736,
                "tc.seg_scan": (10550272 + 8458752 + 10553088) // 3,  # mean of the three passes' scans
                "tc.walk_out": 303517696,
                "tc.walk_dq": 403231232,
                "tc.walk_dk": 401504256,
                "tc.walk_dv": 304301056,
                "tc.dla_intra": 338004480,
                "tc.dla_carry": 12590336,
                "tc.dla": 3171328,
            }},
    "simt.": {"source": "ssd_chunked_scan_gb300/csrc/simt.cu", "sha16": "5682068978fc8373", "commit": "02155b1",
              "bytes": {}},
    "mamba.": {"source": "ssd_chunked_scan_gb300/csrc/mamba.cu", "sha16": "46a5b2d4c8f2dcb9", "commit": "c617278",
               "bytes": {}},
}
_SIMT_TRAFFIC = {
    # kernels that run twice per step: the mean of their launches
    "simt.chunk_state": (381861888 + 379118080) // 2,
    "simt.state_scan_fwd": (475357696 + 475306752) // 2,
    "simt.chunk_out": 582941184,
    "simt.query_state": 377939968,
    "simt.state_scan_rev": 475440384,
    "simt.chunk_grad": 1518565888,
    "simt.dla_carry": 1090048,
}
# the same for the Mamba kernels at d1024 L8192; seg_state and seg_scan run more
# than once per step: the mean of their launches
_MAMBA_TRAFFIC = {
    "mamba.seg_state": (270622976 + 3436800 + 270637056 + 328448) // 2,
    "mamba.seg_scan": (6209280 + 6209024 + 6209024) // 3,
    "mamba.out": 278507776 + 99099904,
    "mamba.seg_grad_state": 270713856 + 371456,
    "mamba.bwd": 427659520 + 242076672,
}
TRAFFIC_GROUPS["simt."]["bytes"] = _SIMT_TRAFFIC
TRAFFIC_GROUPS["mamba."]["bytes"] = _MAMBA_TRAFFIC


def _sha16(rel):
    import hashlib
    try:
        with open(os.path.join(ROOT, rel), "rb") as f:
            return hashlib.sha256(f.read()).hexdigest()[:16]
    except OSError:
        return None


def traffic_of(kernel):
    """(DRAM bytes per launch or None, a note on where the figure comes from)."""
    for prefix, grp in TRAFFIC_GROUPS.items():
        if not kernel.startswith(prefix):
            continue
        if kernel not in grp["bytes"] or grp["sha16"] is None:
            return None, f"no ncu capture of {kernel} in its current form"
        if _sha16(grp["source"]) != grp["sha16"]:
            return None, (f"{grp['source']} changed since the ncu capture at commit {grp['commit']}; "
                          "its figure no longer applies")
        return grp["bytes"][kernel], (f"ncu capture at commit {grp['commit']}, "
                                      f"{grp['source']} unchanged since (sha256 {grp['sha16']}...)")
    return None, f"no ncu capture of {kernel}"

# nominal dense tensor rates: tf32 1.1 PF vs bf16 2.25 PF per GPU
TF32_OVER_BF16 = 1.1 / 2.25
# FP32 FFMA: 152 SMs x 128 lanes x 2 flop x 2070 MHz (maximum SM clock)
FP32_TFLOPS = 152 * 128 * 2 * 2.070e9 / 1e12


def kernel_costs(w, sms=152):
    """Algorithmic bytes and flops per launch of each kernel, and its bound.

    Bytes count each tensor a kernel must read or write once (a group's q / k
    once, not once per head); flops count multiply-adds as 2, the causal half
    of each chunk's C x C block, per (b, l) token: QK^T G*C*dk, PV / dP etc.
    H*C*d, each dk x dv contraction 2*H*dk*dv."""
    B, L, G, H, dk, dv, C = w.B, w.L, w.G, w.H, w.dk, w.dv, w.chunk
    N = -(-L // C)
    f = 4
    qk = B * L * G * dk * f
    vv = B * L * H * dv * f
    la = B * L * H * f
    st = B * H * N * dk * dv * f
    h0 = B * H * dk * dv * f
    BL = B * L
    c = {}
    c["simt.chunk_state"] = (qk + vv + la + st, BL * 2 * H * dk * dv, "alu")
    c["simt.query_state"] = (qk + vv + la + st, BL * 2 * H * dk * dv, "alu")
    c["simt.state_scan_fwd"] = (2 * st + h0, 2 * B * H * N * dk * dv, "hbm")
    c["simt.state_scan_rev"] = (2 * st + h0, 2 * B * H * N * dk * dv, "hbm")
    c["simt.chunk_out"] = (2 * qk + 2 * vv + la + st, BL * (G * C * dk + H * C * dv + 2 * H * dk * dv), "alu")
    c["simt.chunk_grad"] = (2 * qk + 2 * vv + la + 2 * st + 2 * qk + vv + la,
                            BL * (G * C * dk + 2 * H * C * (dk + dv) + 6 * H * dk * dv), "alu")
    c["simt.dla_carry"] = (2 * la, BL * H, "hbm")
    # tensor-core path: per-segment states [B,H,nseg,dk,dv]; every kernel is
    # bound by HBM traffic at these shapes (arithmetic intensity < 60 FLOP/B)
    nseg = tc_nseg(w, sms)
    sst = B * H * nseg * dk * dv * f
    fw = BL * (G * C * dk + H * C * dv + 4 * H * dk * dv)      # forward pass
    st2 = BL * 2 * H * dk * dv                                 # one state contraction
    for n in ("tc.seg_state", "tc.seg_state_dq", "tc.seg_state_dk", "tc.seg_state_dv"):
        c[n] = (qk + vv + la + sst, st2, "hbm")
    c["tc.seg_scan"] = (2 * sst + h0, 2 * B * H * nseg * dk * dv, "hbm")
    c["tc.walk_out"] = (2 * qk + 2 * vv + la + sst, fw, "hbm")
    c["tc.walk_dv"] = (2 * qk + 2 * vv + la + sst, fw, "hbm")
    for n in ("tc.walk_dq", "tc.walk_dk"):
        c[n] = (3 * qk + 2 * vv + 2 * la + sst, fw + BL * H * dk * 2, "hbm")
    c["tc.dla_intra"] = (2 * qk + 2 * vv + 2 * la, BL * (G * C * dk + H * C * dv + H * C), "hbm")
    # dla: the in-segment suffix sums (B_t, rq, rk in, dla out); dla_carry: the
    # segment carries, a dot of the two passes' states per segment
    c["tc.dla"] = (4 * la + B * H * nseg * 8, BL * H * 4, "hbm")
    c["tc.dla_carry"] = (2 * sst + B * H * nseg * 8, 2 * B * H * nseg * dk * dv, "hbm")
    # deterministic group sums (opt-in): read every head's share, write the group's
    c["tc.group_sum"] = (BL * H * dk * f + qk, BL * H * dk, "hbm")
    # sequential kernels (chunk = 1): fp32 state updates and reductions, one
    # token at a time; E arrays hold one float per token, head and column block
    nblk = -(-dv // 32)
    e = B * L * H * nblk * f
    c["seq.sweep_out"] = (2 * qk + 2 * vv + la + 2 * h0, BL * H * 4 * dk * dv, "alu")
    c["seq.sweep_dq"] = (3 * qk + 2 * vv + la + h0 + e, BL * H * 6 * dk * dv, "alu")
    c["seq.sweep_dkdv"] = (3 * qk + 3 * vv + la + 2 * h0 + e, BL * H * 6 * dk * dv, "alu")
    c["seq.dla"] = (2 * e + la, BL * H * 2 * nblk, "hbm")
    return c


def tc_nseg(w, sms=152):
    """Segments per sequence chosen by the tensor-core path (same rule as tc.cu:
    one wave of walk CTAs at one CTA per SM)."""
    bh = w.B * w.H
    want = max(1, sms // bh)
    Ls = -(-(-(-w.L // want)) // 64) * 64
    Ls = max(Ls, 64)
    return -(-w.L // Ls)


# Kernels that, with the backward's passes overlapped, run on the SMs the
# one-CTA-per-SM walks leave idle, beside them for most of the backward: their
# live launch time is long by design and is not the step's critical path.
SIDE_KERNELS = ("tc.dla_intra",)


def kernel_roofline(trace, costs, peaks, traffic_ok, exclude=(), rank=None):
    """Roofline entry of one kernel of `trace` ({name: (launches, total ms)}):
    algorithmic bytes (or flops) per launch over its mean launch time in
    `trace`, against the measured peak.  The kernel is the one with the most
    device time in `rank` (default: `trace` itself) among those not in
    `exclude`.  (With the backward's passes overlapped, a short kernel's live
    span also holds the time it queues behind the other stream's kernels, so
    the ranking uses the serialised timing when there is one.)"""
    rank = rank if rank else trace
    cand = {k: v for k, v in rank.items() if k not in exclude and k in trace} or trace
    top_name = max(cand.items(), key=lambda kv: kv[1][1])[0]
    top_n, top_ms = trace[top_name]
    per_launch_ms = top_ms / top_n
    if top_name not in costs:
        raise KeyError(f"no algorithmic cost entry for kernel {top_name}")
    kb, kf, kbound = costs[top_name]
    if kbound == "tensor":
        peak = peaks["bf16_tflops"] * TF32_OVER_BF16
        ach = kf / (per_launch_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": ach, "peak": peak, "unit": "TFLOP/s",
                "peak_note": f"tf32 = {peaks['source']} bf16 burst x nominal tf32/bf16 ratio"}
    elif kbound == "alu":
        ach = kf / (per_launch_ms / 1e3) / 1e12
        roof = {"bound": "alu", "achieved": ach, "peak": FP32_TFLOPS, "unit": "TFLOP/s",
                "peak_note": "fp32 FFMA: 152 SMs x 128 lanes x 2 flop x 2070 MHz"}
    else:
        ach = kb / (per_launch_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": ach, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "peak_note": f"{peaks['source']} copy bandwidth"}
    roof["frac"] = roof["achieved"] / roof["peak"]
    if traffic_ok:
        roof["traffic"], roof["traffic_source"] = traffic_of(top_name)
    else:
        roof["traffic"], roof["traffic_source"] = None, "captured at the default workload only"
    roof["kernel"] = top_name
    roof["kernel_ms_per_launch"] = per_launch_ms
    roof["alg_bytes_per_launch"] = kb
    roof["alg_flops_per_launch"] = kf
    return roof


def kernel_table(trace):
    tot = sum(x[1] for x in trace.values())
    return {n: {"launches": c, "ms_total": t, "share": t / tot}
            for n, (c, t) in sorted(trace.items(), key=lambda kv: -kv[1][1])}


def step_totals(w):
    """Minimal bytes and flops of one fwd + bwd step (two calls)."""
    B, L, G, H, dk, dv, C = w.B, w.L, w.G, w.H, w.dk, w.dv, w.chunk
    f = 4
    args = (2 * B * L * G * dk + B * L * H * dv + B * L * H + B * H * dk * dv) * f
    out = B * L * H * dv * f
    bytes_fb = 3 * args + 2 * out  # fwd reads args writes out; bwd reads args + dout, writes grads
    fl_f = B * L * (G * C * dk + H * C * dv + 4 * H * dk * dv)
    fl_b = B * L * (G * C * dk + 2 * H * C * (dk + dv) + 10 * H * dk * dv)
    return bytes_fb, fl_f + fl_b, args + out, fl_f


class ClockSampler:
    """SM clock, power and clock-event (throttle) reasons of one GPU, sampled in
    the background every 5 ms through NVML's read-only queries (ctypes on
    libnvidia-ml), so that even a timed region of a few tens of milliseconds
    holds samples; `nvidia-smi -lms 100` when NVML cannot be loaded.  The GPU
    is found by the CUDA device's UUID."""

    PERIOD_S = 0.005
    # clock-event reason bits (nvml.h) reported by name
    BITS = {"sw_power_cap": 0x4, "hw_slowdown": 0x8 | 0x80, "sw_thermal_slowdown": 0x20,
            "hw_thermal_slowdown": 0x40}
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.samples = []  # (time, sm_mhz, max_mhz, power_w, [reason names])
        self.index = index
        self.proc = None
        self.source = None
        self._stop = threading.Event()
        self.t = None

    def _uuid(self):
        try:
            import torch
            u = str(torch.cuda.get_device_properties(self.index).uuid)
            return u if u.startswith("GPU-") else "GPU-" + u
        except Exception:
            return None

    def _nvml(self):
        import ctypes
        lib = ctypes.CDLL("libnvidia-ml.so.1")
        if lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit failed")
        h = ctypes.c_void_p()
        uuid = self._uuid()
        if uuid is None or lib.nvmlDeviceGetHandleByUUID(uuid.encode(), ctypes.byref(h)) != 0:
            n = ctypes.c_uint(0)
            if lib.nvmlDeviceGetCount_v2(ctypes.byref(n)) != 0 or n.value != 1:
                raise OSError("cannot tell which NVML device is this CUDA device")
            if lib.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(h)) != 0:
                raise OSError("nvmlDeviceGetHandleByIndex failed")
        reasons_fn = getattr(lib, "nvmlDeviceGetCurrentClocksEventReasons", None) or \
            lib.nvmlDeviceGetCurrentClocksThrottleReasons
        return lib, h, reasons_fn

    def start(self):
        try:
            lib, h, reasons_fn = self._nvml()
        except Exception:
            return self._start_smi()
        import ctypes
        self.source = "nvml, 5 ms"

        def run():
            sm, mx, pw, rs = ctypes.c_uint(), ctypes.c_uint(), ctypes.c_uint(), ctypes.c_ulonglong()
            while not self._stop.is_set():
                t = time.time()
                ok = (lib.nvmlDeviceGetClockInfo(h, 1, ctypes.byref(sm)) == 0 and
                      lib.nvmlDeviceGetMaxClockInfo(h, 1, ctypes.byref(mx)) == 0 and
                      reasons_fn(h, ctypes.byref(rs)) == 0)
                p = float(pw.value) / 1e3 if lib.nvmlDeviceGetPowerUsage(h, ctypes.byref(pw)) == 0 else None
                if ok:
                    names = sorted(n for n, b in self.BITS.items() if rs.value & b)
                    self.samples.append((t, float(sm.value), float(mx.value), p, names))
                self._stop.wait(self.PERIOD_S)
        self.t = threading.Thread(target=run, daemon=True)
        self.t.start()

    def _start_smi(self):
        dev = self._uuid() or str(self.index)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", dev, f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.source = "nvidia-smi, 100 ms"
        self.t = threading.Thread(target=self._read_smi, daemon=True)
        self.t.start()

    def _read_smi(self):
        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8 and num(parts[0]) is not None:
                rs = sorted(names[i] for i in range(4) if parts[4 + i].lower() == "active")
                self.samples.append((time.time(), num(parts[0]), num(parts[1]), num(parts[2]), rs))

    def wait_first(self, timeout=5.0):
        """Block until the sampler has produced a sample (nvidia-smi's start-up
        stalls the GPU briefly; it must not fall inside a timed region)."""
        t0 = time.time()
        while self.t is not None and not self.samples and time.time() - t0 < timeout:
            time.sleep(0.01)

    def stop(self):
        self._stop.set()
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
        if self.t is not None:
            self.t.join(timeout=5)

    def summary(self, t0, t1):
        inwin = [x for x in self.samples if t0 <= x[0] <= t1]
        window = "timed"
        if not inwin:
            inwin = list(self.samples)
            window = "whole run (no sample fell inside the timed region)"
        if not inwin:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"], "samples": 0,
                    "source": self.source}
        sm = [x[1] for x in inwin if x[1] is not None]
        mx = [x[2] for x in inwin if x[2] is not None]
        pw = [x[3] for x in inwin if x[3] is not None]
        reasons = sorted({r for x in inwin for r in x[4]})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "power_w_max": max(pw) if pw else None, "samples": len(inwin), "window": window,
                "source": self.source}


def oracle_sample(w, threads):
    """The oracle's bounded sample of workload w: the first nb batch entries
    (every group and head, full sequence), nb the fewest whose nb*H
    independent (batch, head) sequences keep `threads` threads busy.
    Returns (arrays, nb, threads actually used)."""
    import numpy as np
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    nb = max(1, min(w.B, -(-threads // w.H)))
    arrs = tuple(np.ascontiguousarray(x[:nb]) for x in workload_inputs(w))
    return arrs, nb, min(threads, nb * w.H)


def cpu_oracle_sample(w, min_seconds=10.0, max_reps=60):
    """Time the float64 oracle (fwd + bwd) on a sample of the workload,
    repeated until min_seconds have passed; returns tokens/s and details,
    with the fwd and fwd+bwd time of one rep and a single-thread figure (the
    oracle on one (batch, head) sequence, which one thread runs)."""
    import numpy as np
    from oracle import oracle_threads, ssd_bwd_ref, ssd_fwd_ref
    (q, k, v, la, h0, dout), nb, used = oracle_sample(w, oracle_threads())
    toks, t0, reps, t_fwd = 0, time.perf_counter(), 0, 0.0
    first = None
    while True:
        ta = time.perf_counter()
        r_out = ssd_fwd_ref(q, k, v, la, h0)
        t_fwd += time.perf_counter() - ta
        r_g = ssd_bwd_ref(q, k, v, la, h0, dout)
        if first is None:
            first = (r_out, r_g)
        reps += 1
        toks += nb * w.L * w.H
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    one = (q[:1, :, :1], k[:1, :, :1], v[:1, :, :1], la[:1, :, :1], h0[:1, :1], dout[:1, :, :1])
    one = tuple(np.ascontiguousarray(x) for x in one)
    ta = time.perf_counter()
    ssd_fwd_ref(*one[:5])
    tb = time.perf_counter()
    ssd_bwd_ref(*one)
    tc_ = time.perf_counter()
    return {"value": toks / el, "unit": "tokens/s", "cores": used, "kind": "oracle",
            "sample": f"batch entries 0..{nb - 1} of {w.name} ({nb} x {w.L} x {w.H} heads, "
                      f"all groups), float64 fwd+bwd, {reps} rep(s), {el:.1f} s",
            "fwd_ms_per_rep": t_fwd / reps * 1e3, "fwd_bwd_ms_per_rep": el / reps * 1e3,
            "single_thread": {"sample": f"one (batch, head) sequence of {w.name}, {w.L} tokens",
                              "fwd_ms": (tb - ta) * 1e3, "fwd_bwd_ms": (tc_ - ta) * 1e3,
                              "tokens_per_s": w.L / (tc_ - ta)},
            "_ref": first, "_nb": nb}


GRAD_KEYS = {"q": "dq", "k": "dk", "v": "dv", "log_alpha": "dlog_alpha", "h0": "dh0"}


def _rel(x, ref):
    import numpy as np
    x = np.asarray(x, np.float64)
    ref = np.asarray(ref, np.float64)
    den = float(np.max(np.abs(ref))) if ref.size else 0.0
    num = float(np.max(np.abs(x - ref))) if ref.size else 0.0
    return num / den if den > 0 else num


def oracle_accuracy(w, out, grads, ref=None, nb=None, residual_mb=0.0):
    """The accuracy fields of a bench record, as the benchmark pages keep them
    beside each timing: rel_err = max|x - ref| / max|ref| of the output and of
    each gradient against the float64 oracle, on a sample of the workload,
    computed outside the timed region; residual_mb: what is kept between the
    forward and the backward besides the inputs (the segment states and the
    final state, or 0 when the backward recomputes them).  out / grads: the GPU results for the whole workload (host numpy
    arrays; grads None for a forward alone).  ref: the oracle's (out, grads)
    on batch entries 0..nb-1, when the CPU baseline has computed them; else
    the oracle runs here on one (batch 0, group 0) unit."""
    import numpy as np
    from oracle import ssd_bwd_ref, ssd_fwd_ref
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    hpg = w.H // w.G
    if ref is not None:
        sel = lambda x, kind: x[:nb]
        sample = f"batch entries 0..{nb - 1} of {w.name}, every head"
        r_out, r_g = ref
    else:
        gs, hs = slice(0, 1), slice(0, hpg)

        def sel(x, kind):
            if kind == "qk":
                return np.ascontiguousarray(x[:1, :, gs])
            if kind == "h":
                return np.ascontiguousarray(x[:1, hs])
            return np.ascontiguousarray(x[:1, :, hs])
        q, k, v, la, h0, dout = workload_inputs(w)
        uq, uk, uv, ula, uh0, udo = (sel(q, "qk"), sel(k, "qk"), sel(v, "v"), sel(la, "v"),
                                     sel(h0, "h"), sel(dout, "v"))
        r_out = ssd_fwd_ref(uq, uk, uv, ula, uh0)
        r_g = ssd_bwd_ref(uq, uk, uv, ula, uh0, udo) if grads is not None else None
        sample = f"batch entry 0, group 0 of {w.name} ({hpg} heads x {w.L} tokens)"
    kinds = {"dq": "qk", "dk": "qk", "dv": "v", "dlog_alpha": "v", "dh0": "h"}
    acc = {"rel_err": _rel(sel(out, "v"), r_out),
           "rel_err_grads": None if grads is None else
           {a: _rel(sel(grads[g], kinds[g]), r_g[g]) for a, g in GRAD_KEYS.items()},
           "residual_mb": residual_mb,
           "accuracy_sample": sample + ", float64 oracle, max|x - ref| / max|ref| per tensor"}
    return acc


def max_over_ranks(x, device=None):
    """The largest x over all ranks (x itself when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_tokens_per_s(tokens_per_rank, world, ms):
    """Whole-job throughput of `world` replicas that each processed
    tokens_per_rank tokens, over the slowest rank's ms."""
    return tokens_per_rank * world / (ms / 1e3)


def run_reference(args, w):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from oracle import oracle_threads, ssd_bwd_ref, ssd_fwd_ref
    (q, k, v, la, h0, dout), nb, used = oracle_sample(w, oracle_threads())

    def step():
        ssd_fwd_ref(q, k, v, la, h0)
        ssd_bwd_ref(q, k, v, la, h0, dout)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    toks = nb * w.L * w.H
    val = toks * args.steps / el
    sample = (f"batch entries 0..{nb - 1} ({nb * w.H} heads, all groups) of {w.name}, "
              f"full L={w.L}, float64 fwd+bwd per step")
    line = {"impl": "reference", "metric": METRIC, "value": val, "unit": "tokens/s",
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": w.name, "mode": "fwd_bwd", "B": w.B, "G": w.G, "H": w.H,
                       "L": w.L, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                       "sample_tokens_per_step": toks},
            "cpu_baseline": {"value": val, "unit": "tokens/s", "cores": used,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": val, "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


L2_BYTES = 126 * 2 ** 20  # GB300 L2


def l2_note(step_bytes):
    """How L2 stands between timed steps (no flush is made)."""
    mib = step_bytes / 2 ** 20
    if step_bytes > L2_BYTES:
        return f"no flush: each step's inputs and outputs ({mib:.0f} MiB) exceed L2"
    return (f"no flush: each step's inputs and outputs ({mib:.0f} MiB) fit in L2, so this "
            f"small workload's steps read them from L2")


def resident_bytes(B, L, G, H, dk, dv, mode):
    """Bytes of the caller's tensors one step touches: the five arguments and
    out, plus dout and the five gradients for fwd_bwd."""
    args = 4 * (2 * B * L * G * dk + B * L * H * dv + B * L * H + B * H * dk * dv)
    out = 4 * B * L * H * dv
    if mode == "fwd":
        return args + out
    return 2 * args + out + 4 * B * L * H * dv


def measure_peak(ssd, torch, dev, fn, resident):
    """Peak device bytes of one call of fn: the caller's resident tensors plus
    the high-water mark of the library's workspace pool during the call."""
    torch.cuda.synchronize(dev)
    ssd.ssd_pool_high_water(reset=True)
    fn()
    torch.cuda.synchronize(dev)
    return resident + ssd.ssd_pool_high_water()


def run_max_len(args, w):
    """Largest sequence length (doubling from the workload's L) whose fwd_bwd
    runs on one GPU, with the peak memory of each length that ran.  The next
    length is not attempted once its predicted footprint (caller tensors plus
    the reported workspace) exceeds 90% of the free device memory."""
    import torch
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    from ssd_chunked_scan_gb300 import ssd
    from ssd_chunked_scan_gb300.inputs import make_inputs_on_device
    ssd.ssd_set_path(ssd.SSD_PATH_TC if args.path == "tc" else ssd.SSD_PATH_SIMT)
    B, G, H, dk, dv, C = w.B, w.G, w.H, w.dk, w.dv, w.chunk

    def need(L):
        ws = max(ssd.ssd_fwd_workspace_bytes(B, L, G, H, dk, dv, C),
                 ssd.ssd_bwd_workspace_bytes(B, L, G, H, dk, dv, C))
        return resident_bytes(B, L, G, H, dk, dv, "fwd_bwd") + ws

    runs, L, stop = [], w.L, None
    P = 512  # prefix / suffix tokens compared with separate short runs
    while True:
        free, total = torch.cuda.mem_get_info(dev)
        try:
            ok_shape = need(L)
        except ssd.SSDError as e:  # beyond what the path's index types take
            stop = {"seq": L, "reason": str(e)}
            break
        if ok_shape > 0.9 * free:
            stop = {"seq": L, "needed_mb": ok_shape / MiB, "free_mb": free / MiB,
                    "reason": "predicted footprint above 90% of free device memory"}
            break
        q, k, v, la, h0, dout = make_inputs_on_device(dev, B, L, G, H, dk, dv, w.seed, w.la_mu)
        out = torch.empty((B, L, H, dv), device=dev)
        grads = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
                 "dlog_alpha": torch.empty_like(la), "dh0": torch.empty_like(h0)}

        def step():
            ssd.ssd_fwd(q, k, v, la, h0, chunk=C, out=out)
            ssd.ssd_bwd(q, k, v, la, h0, dout, chunk=C, grads=grads)
        t0 = time.perf_counter()
        peak = measure_peak(ssd, torch, dev, step, resident_bytes(B, L, G, H, dk, dv, "fwd_bwd"))
        sec = time.perf_counter() - t0
        if ssd.ssd_last_device_error() != 0:
            raise RuntimeError(f"device error word set at L={L}")
        finite = all(bool(torch.isfinite(t).all()) for t in [out] + list(grads.values()))
        # self-consistency: the first P outputs depend only on the first P
        # inputs; dk, dv of the last P tokens only on the last P inputs
        pre = [x[:, :P].contiguous() for x in (q, k, v, la, dout)]
        suf = [x[:, L - P:].contiguous() for x in (q, k, v, la, dout)]
        o_pre = ssd.ssd_fwd(pre[0], pre[1], pre[2], pre[3], h0, chunk=C)
        g_suf = ssd.ssd_bwd(suf[0], suf[1], suf[2], suf[3], None, suf[4], chunk=C)
        torch.cuda.synchronize(dev)
        rel = lambda a, b: float((a - b).abs().max() / b.abs().max().clamp_min(1e-30))
        cons = {"out_prefix": rel(out[:, :P], o_pre), "dk_suffix": rel(grads["dk"][:, L - P:], g_suf["dk"]),
                "dv_suffix": rel(grads["dv"][:, L - P:], g_suf["dv"])}
        runs.append({"seq": L, "peak_mb": peak / MiB, "predicted_mb": ok_shape / MiB,
                     "fwd_bwd_s": sec, "finite": finite, "consistency_rel_err": cons})
        del q, k, v, la, h0, dout, out, grads, pre, suf, o_pre, g_suf
        torch.cuda.empty_cache()
        L *= 2
    best = runs[-1] if runs else None
    line = {"metric": "largest sequence length for fwd_bwd on one GPU (doubling)",
            "value": best["seq"] if best else 0, "unit": "tokens", "n_gpus": 1,
            "higher_is_better": True, "dtype": "tf32" if args.path == "tc" else "f32",
            "data": "synthetic (seeded, generated on the device)",
            "config": {"workload": w.name, "path": args.path, "B": B, "G": G, "H": H,
                       "dk": dk, "dv": dv, "chunk": C, "start_seq": w.L},
            "largest_ok": best, "runs": runs, "first_not_run": stop,
            "device_total_mb": torch.cuda.mem_get_info(dev)[1] / MiB,
            "page_context": {"rtx3090_24gb_chunked_largest_seq": PAGE_MAX_LEN}}
    print(json.dumps(line), flush=True)
    return 0


# ---- Mamba-1 selective scan (--op mamba) -----------------------------------

MAMBA_WORKLOAD = "mamba_d1024_L8192"
MAMBA_METRIC = "Mamba-1 selective scan fwd / fwd_bwd channel-tokens/s (B·L·D) at 1 GB300"
# "kernel_mamba_cpu.json" records, impl chunked (CPU backend): ms per call
PAGE_MAMBA_CPU_MS = {"mamba_d1024_L8192": {"fwd": 298.87558800692204, "fwd_bwd": 1867.5783030048478},
                     "mamba_d256_L8192": {"fwd": 107.37162199802697, "fwd_bwd": 644.8948080069385},
                     "mamba_d512_L8192": {"fwd": 205.45388301252387, "fwd_bwd": 1037.0018319954397}}
# MUFU (ex2) rate: 16 results per clock per SM x 152 SMs x 2070 MHz
MUFU_GEXP = 152 * 16 * 2.070


def mamba_nseg(w, sms=152):
    """Segments per sequence chosen by the Mamba kernels (same rule as mamba.cu)."""
    base = w.B * w.D
    want = max(1, (640 * sms) // base)
    ls = -(-w.L // want)
    ls = min(max(-(-ls // 32) * 32, 32), 1024)
    return -(-w.L // ls)


def mamba_costs(w, sms=152):
    """Algorithmic bytes and exponentials per launch of each Mamba kernel."""
    f = 4
    BLD, BLN = w.B * w.L * w.D * f, w.B * w.L * w.N * f
    nseg = mamba_nseg(w, sms)
    st = w.B * nseg * w.D * w.N * f
    ds = w.B * nseg * w.D * f
    ex = w.B * w.L * w.D * w.N
    return {
        "mamba.seg_state": (2 * BLD + BLN + st + ds, ex),
        "mamba.seg_scan": (2 * st + ds, w.B * nseg * w.D * w.N),
        "mamba.out": (3 * BLD + 2 * BLN + st + ds, ex),
        "mamba.seg_grad_state": (2 * BLD + BLN + st + ds, ex),
        "mamba.bwd": (5 * BLD + 4 * BLN + 2 * st, 2 * ex),
    }


def run_mamba(args):
    """One JSON line for the Mamba selective scan: fwd + bwd per step."""
    import torch
    from ssd_chunked_scan_gb300 import ssd
    from ssd_chunked_scan_gb300.inputs import MAMBA_BY_NAME, mamba_workload_inputs
    name = args.workload if args.workload in MAMBA_BY_NAME else MAMBA_WORKLOAD
    w = MAMBA_BY_NAME[name]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    host = [torch.from_numpy(x).pin_memory() for x in mamba_workload_inputs(w)]
    x, dt, A, Bm, Cm, Dk, dy = [t.to(dev) for t in host]
    y = torch.empty_like(x)
    grads = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x), "dA": torch.empty_like(A),
             "dB": torch.empty_like(Bm), "dC": torch.empty_like(Cm), "dD": torch.empty_like(Dk)}
    stream = torch.cuda.current_stream(dev)
    fb = args.mode != "fwd"

    def step():
        ssd.ssd_mamba_fwd(x, dt, A, Bm, Cm, Dk, y=y)
        if fb:
            ssd.ssd_mamba_bwd(x, dt, A, Bm, Cm, Dk, dy, grads=grads)

    def timed(fn, n):
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(n):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) / n

    clocks = ClockSampler(0)
    clocks.start()
    clocks.wait_first()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    n0 = ssd.ssd_launch_count()
    th0 = time.time()
    ms = timed(step, args.steps)
    th1 = time.time()
    launches = ssd.ssd_launch_count() - n0
    ssd.ssd_trace_reset()
    ssd.ssd_trace_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    ssd.ssd_trace_enable(False)
    trace = ssd.ssd_trace_collect()
    ssd.ssd_trace_reset()
    clocks.stop()
    fwd_ms = timed(lambda: ssd.ssd_mamba_fwd(x, dt, A, Bm, Cm, Dk, y=y), args.steps)

    e2e = None
    if not args.no_e2e:
        dbuf = [torch.empty_like(t) for t in (x, dt, A, Bm, Cm, Dk, dy)]
        h_y = torch.empty(y.shape, pin_memory=True)
        h_g = {n: torch.empty(t.shape, pin_memory=True) for n, t in grads.items()}

        def e2e_step():
            for d, hsrc in zip(dbuf, host):
                d.copy_(hsrc, non_blocking=True)
            ssd.ssd_mamba_fwd(*dbuf[:6], y=y)
            h_y.copy_(y, non_blocking=True)
            if fb:
                ssd.ssd_mamba_bwd(*dbuf, grads=grads)
                for n in h_g:
                    h_g[n].copy_(grads[n], non_blocking=True)
        e2e_step()
        e2e_ms = timed(e2e_step, args.steps)
        h2d = sum(t.numel() * 4 for t in (host if fb else host[:6]))
        d2h = y.numel() * 4 + (sum(t.numel() * 4 for t in grads.values()) if fb else 0)
        e2e = {"value": w.tokens / (e2e_ms / 1e3), "unit": "channel-tokens/s", "ms_per_step": e2e_ms,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    peaks = load_peaks()
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    costs = mamba_costs(w, sms)
    top_name, (top_n, top_ms) = max(trace.items(), key=lambda kv: kv[1][1])
    per = top_ms / top_n
    kb, kx = costs[top_name]
    t_hbm = kb / (peaks["hbm_gbs"] * 1e9)
    t_mufu = kx / (MUFU_GEXP * 1e9)
    if t_mufu >= t_hbm:
        roof = {"bound": "alu", "achieved": kx / (per / 1e3) / 1e9, "peak": MUFU_GEXP,
                "unit": "Gexp/s", "peak_note": "MUFU ex2: 152 SMs x 16 per clock x 2070 MHz"}
    else:
        roof = {"bound": "hbm", "achieved": kb / (per / 1e3) / 1e9, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "peak_note": f"{peaks['source']} copy bandwidth"}
    traffic, traffic_src = (traffic_of(top_name) if w.name == MAMBA_WORKLOAD
                            else (None, "captured at the default workload only"))
    roof.update({"frac": roof["achieved"] / roof["peak"],
                 "traffic": traffic, "traffic_source": traffic_src,
                 "kernel": top_name,
                 "kernel_ms_per_launch": per, "alg_bytes_per_launch": kb,
                 "alg_exp_per_launch": kx})
    page = PAGE_MAMBA_CPU_MS.get(w.name, {})
    line = {
        "metric": MAMBA_METRIC, "value": w.tokens / (ms / 1e3), "unit": "channel-tokens/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": w.name, "op": "mamba", "mode": "fwd_bwd" if fb else "fwd",
                   "B": w.B, "L": w.L, "D": w.D, "N": w.N, "segments": mamba_nseg(w, sms),
                   "l2": "no flush: each step's inputs and outputs exceed L2"},
        "roofline": roof,
        "fwd": {"ms": fwd_ms, "tokens_per_s": w.tokens / (fwd_ms / 1e3)},
        "kernels": {n: {"launches": c, "ms_total": t, "share": t / sum(v[1] for v in trace.values())}
                    for n, (c, t) in sorted(trace.items(), key=lambda kv: -kv[1][1])},
        "gpu_launches": launches, "clocks": clocks.summary(th0, th1), "e2e": e2e,
        "page_context": {"cpu_chunked_ms": page or None},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = mamba_cpu_sample(w, fb)
    print(json.dumps(line), flush=True)
    return 0


def run_mamba_reference(args):
    """The float64 Mamba oracle as the reference arm: one fwd + bwd of batch
    entry 0 of the workload per step, on the host cores (rank 0 only)."""
    if int(os.environ.get("RANK", "0")) != 0:
        return 0
    import numpy as np
    from oracle import mamba_bwd_ref, mamba_fwd_ref, oracle_threads
    from ssd_chunked_scan_gb300.inputs import MAMBA_BY_NAME, mamba_workload_inputs
    w = MAMBA_BY_NAME.get(args.workload, MAMBA_BY_NAME[MAMBA_WORKLOAD])
    x, dt, A, Bm, Cm, Dk, dy = mamba_workload_inputs(w)
    sl = lambda a: np.ascontiguousarray(a[:1])
    x, dt, Bm, Cm, dy = map(sl, (x, dt, Bm, Cm, dy))
    fb = args.mode != "fwd"

    def step():
        mamba_fwd_ref(x, dt, A, Bm, Cm, Dk)
        if fb:
            mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
    for _ in range(args.warmup):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    val = w.L * w.D * args.steps / el
    sample = f"batch entry 0 of {w.name} ({w.L} x {w.D} channels), float64 {'fwd+bwd' if fb else 'fwd'} per step"
    cores = min(oracle_threads(), w.D)
    print(json.dumps({
        "impl": "reference", "metric": MAMBA_METRIC, "value": val, "unit": "channel-tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "op": "mamba", "mode": "fwd_bwd" if fb else "fwd",
                   "B": w.B, "L": w.L, "D": w.D, "N": w.N, "sample_tokens_per_step": w.L * w.D},
        "cpu_baseline": {"value": val, "unit": "channel-tokens/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": val, "unit": "channel-tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0}}), flush=True)
    return 0


def mamba_cpu_sample(w, fb, min_seconds=10.0, max_reps=80):
    """The float64 Mamba oracle on batch entry 0 of the workload, repeated for
    about min_seconds."""
    import numpy as np
    from oracle import mamba_bwd_ref, mamba_fwd_ref, oracle_threads
    from ssd_chunked_scan_gb300.inputs import mamba_workload_inputs
    x, dt, A, Bm, Cm, Dk, dy = mamba_workload_inputs(w)
    sl = lambda a: np.ascontiguousarray(a[:1])
    x, dt, Bm, Cm, dy = map(sl, (x, dt, Bm, Cm, dy))
    toks, reps, t0 = 0, 0, time.perf_counter()
    while True:
        mamba_fwd_ref(x, dt, A, Bm, Cm, Dk)
        if fb:
            mamba_bwd_ref(x, dt, A, Bm, Cm, Dk, dy)
        reps += 1
        toks += w.L * w.D
        el = time.perf_counter() - t0
        if el >= min_seconds or reps >= max_reps:
            break
    return {"value": toks / el, "unit": "channel-tokens/s", "cores": min(oracle_threads(), w.D),
            "kind": "oracle", "sample": f"batch entry 0 of {w.name} (1 x {w.L} x {w.D} channels), "
                                        f"float64 {'fwd+bwd' if fb else 'fwd'}, {reps} rep(s), {el:.1f} s"}


def sweep_records(workloads, paths=("tc", "simt"), modes=("fwd", "fwd_bwd")):
    """The records of a sweep: every (workload, path, mode) a path supports,
    as the key dicts that identify a record."""
    recs = []
    for w in workloads:
        for path in paths:
            if path == "tc" and (w.dk % 8 or w.dv % 8 or w.dk > 128 or w.dv > 128 or w.chunk != 64):
                continue
            for mode in modes:
                recs.append({"workload": w.name, "path": path, "mode": mode, "chunk": w.chunk})
    return recs


def sweep_key(rec):
    return (rec["workload"], rec["path"], rec["mode"], rec["chunk"])


def sweep_todo(out_path, records):
    """Records not yet in the JSON-lines file out_path (a line counts once it
    holds a record key, whether it measured a value or recorded an error), so
    an interrupted sweep resumes where it stopped."""
    done = set()
    if os.path.exists(out_path):
        with open(out_path) as f:
            for line in f:
                line = line.strip()
                if not line:
                    continue
                try:
                    r = json.loads(line)
                except ValueError:
                    continue  # a line cut short by an interruption
                if isinstance(r, dict) and isinstance(r.get("record"), dict):
                    done.add(sweep_key(r["record"]))
    return [r for r in records if sweep_key(r) not in done]


def run_sweep(args):
    """Measure every record of the sweep not yet in args.sweep, one bench
    process per record, appending one JSON line each: the record's bench line,
    or the error that stopped it (the sweep goes on)."""
    from ssd_chunked_scan_gb300.inputs import WORKLOADS
    todo = sweep_todo(args.sweep, sweep_records(WORKLOADS))
    if os.path.exists(args.sweep) and os.path.getsize(args.sweep) > 0:
        with open(args.sweep, "rb") as f:
            f.seek(-1, os.SEEK_END)
            cut = f.read(1) != b"\n"
        if cut:  # close a line an interruption left unfinished
            with open(args.sweep, "a") as f:
                f.write("\n")
    for rec in todo:
        cmd = [sys.executable, os.path.abspath(__file__), "--workload", rec["workload"],
               "--path", rec["path"], "--mode", rec["mode"], "--steps", str(args.steps),
               "--warmup", str(args.warmup), "--no-cpu-baseline", "--no-e2e"]
        try:
            r = subprocess.run(cmd, capture_output=True, text=True, timeout=600)
            lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
            if r.returncode == 0 and lines:
                out = {"record": rec, "result": json.loads(lines[-1])}
            else:
                tail = (r.stderr or r.stdout).strip().splitlines()[-1:] or ["no output"]
                out = {"record": rec, "error": f"exit {r.returncode}: {tail[0][:300]}"}
        except subprocess.TimeoutExpired:
            out = {"record": rec, "error": "timed out after 600 s"}
        with open(args.sweep, "a") as f:
            f.write(json.dumps(out) + "\n")
        print(json.dumps({"record": rec, "ok": "result" in out}), flush=True)
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--path", default=os.environ.get("SSD_BENCH_PATH", "tc"), choices=["tc", "simt"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--op", default="ssd", choices=["ssd", "mamba"],
                    help="mamba times the Mamba-1 selective scan instead (its own JSON line)")
    ap.add_argument("--chunk", type=int, default=None,
                    help="override the workload's chunk length (1: the sequential kernels)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--deterministic", action="store_true",
                    help="tensor-core backward with deterministic group sums (ssd_set_deterministic)")
    ap.add_argument("--no-accuracy", action="store_true",
                    help="skip the rel_err fields (the float64 oracle on a sample of the workload)")
    ap.add_argument("--saved-states", action="store_true",
                    help="fwd_bwd step as ssd_fwd_save + ssd_bwd_saved (the forward keeps its "
                         "segment states for the backward: residual memory) instead of "
                         "ssd_fwd + ssd_bwd (recompute, no residual)")
    ap.add_argument("--mode", default="fwd_bwd", choices=["fwd_bwd", "fwd", "max_len"],
                    help="fwd times ssd_fwd alone (a step is then one forward pass); "
                         "max_len finds the largest sequence length fwd_bwd runs at")
    ap.add_argument("--sweep", default=None, metavar="OUT.jsonl",
                    help="measure every (workload, path, mode) record not yet in OUT.jsonl "
                         "(fwd and fwd_bwd, both paths), appending one line per record")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.sweep:
        if args.steps == 200:
            args.steps = 20  # a record is a short measurement
        return run_sweep(args)

    if args.op == "mamba":
        if args.impl == "reference":
            return run_mamba_reference(args)
        return run_mamba(args)
    from ssd_chunked_scan_gb300.inputs import BY_NAME
    w = BY_NAME[args.workload]
    if args.chunk:
        import dataclasses
        w = dataclasses.replace(w, chunk=args.chunk)
    if args.impl == "reference":
        return run_reference(args, w)
    if args.mode == "max_len":
        return run_max_len(args, w)

    import torch
    import torch.distributed as dist
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        dist.init_process_group("nccl", device_id=dev)

    from ssd_chunked_scan_gb300 import ssd
    from ssd_chunked_scan_gb300.inputs import workload_inputs
    ssd.ssd_set_deterministic(bool(args.deterministic))
    ssd.ssd_set_path(ssd.SSD_PATH_TC if args.path == "tc" else ssd.SSD_PATH_SIMT)

    host = [torch.from_numpy(x).pin_memory() for x in workload_inputs(w)]
    q, k, v, la, h0, dout = [x.to(dev) for x in host]
    out = torch.empty((w.B, w.L, w.H, w.dv), device=dev)
    grads = {"dq": torch.empty_like(q), "dk": torch.empty_like(k), "dv": torch.empty_like(v),
             "dlog_alpha": torch.empty_like(la), "dh0": torch.empty_like(h0)}
    stream = torch.cuda.current_stream(dev)
    # the forward's segment states (and final state) kept for the backward
    save = args.mode == "fwd_bwd" and args.saved_states
    n_saved = ssd.ssd_saved_bytes(w.B, w.L, w.G, w.H, w.dk, w.dv, w.chunk) // 4 if save else 0
    saved = torch.empty((n_saved,), device=dev) if n_saved else None
    hT = torch.empty_like(h0) if save else None
    residual_mb = ((n_saved + hT.numel()) * 4 / MiB) if save else 0.0

    def step():
        if not save:
            ssd.ssd_fwd(q, k, v, la, h0, chunk=w.chunk, out=out)
            if args.mode == "fwd_bwd":
                ssd.ssd_bwd(q, k, v, la, h0, dout, chunk=w.chunk, grads=grads)
            return
        ssd.ssd_fwd_save(q, k, v, la, h0, chunk=w.chunk, out=out, hT=hT, saved=saved)
        ssd.ssd_bwd_saved(q, k, v, la, h0, dout, None, hT, saved, chunk=w.chunk, grads=grads)

    def barrier():
        if world > 1:
            dist.barrier()

    clocks = ClockSampler(local)
    clocks.start()
    clocks.wait_first()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if ssd.ssd_last_device_error() != 0:
        raise RuntimeError("device error word set during warm-up")

    # timed region: exactly K steps, inputs (323 MiB + dout 128 MiB) larger than L2
    barrier()
    torch.cuda.synchronize(dev)
    n0 = ssd.ssd_launch_count()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    # events at the ends of up to five equal runs of steps inside the region:
    # the per-run ms per step give the median and quartiles
    nrep = min(5, args.steps)
    ends = {round(args.steps * (j + 1) / nrep) - 1: torch.cuda.Event(enable_timing=True)
            for j in range(nrep)}
    th0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step()
        if i in ends:
            ends[i].record(stream)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    th1 = time.time()
    barrier()
    launches = ssd.ssd_launch_count() - n0
    ms = max_over_ranks(e0.elapsed_time(e1) / args.steps, dev)
    runs, prev_ev, prev_i = [], e0, -1
    for i in sorted(ends):
        runs.append(prev_ev.elapsed_time(ends[i]) / (i - prev_i))
        prev_ev, prev_i = ends[i], i
    qs = statistics.quantiles(runs, n=4, method="inclusive") if len(runs) > 1 else runs * 3
    repeats = {"runs": len(runs), "ms_per_step_median": statistics.median(runs),
               "ms_per_step_q1": qs[0], "ms_per_step_q3": qs[2]}
    if ssd.ssd_last_device_error() != 0:
        raise RuntimeError("device error word set during the timed region")

    # per-kernel device time: the same K steps again with every launch bracketed by events
    ssd.ssd_trace_reset()
    ssd.ssd_trace_enable(True)
    for _ in range(args.steps):
        step()
    torch.cuda.synchronize(dev)
    ssd.ssd_trace_enable(False)
    trace = ssd.ssd_trace_collect()
    ssd.ssd_trace_reset()
    # and once more with the backward's passes serialised, so that each
    # kernel's time is its own (the ncu launch list is serialised too)
    overlap_on = (ssd.ssd_get_overlap() and args.path == "tc" and args.mode == "fwd_bwd"
                  and w.chunk != 1)
    trace_iso = None
    if overlap_on:
        prev = ssd.ssd_set_overlap(False)
        ssd.ssd_trace_enable(True)
        for _ in range(args.steps):
            step()
        torch.cuda.synchronize(dev)
        ssd.ssd_trace_enable(False)
        ssd.ssd_set_overlap(prev)
        trace_iso = ssd.ssd_trace_collect()
        ssd.ssd_trace_reset()
    clocks.stop()
    clk = clocks.summary(th0, th1)
    # the results of these steps, for the accuracy fields (compared with the
    # oracle after everything timed has run)
    want_acc = rank == 0 and not args.no_accuracy
    res_out = out.cpu().numpy() if want_acc else None
    res_grads = ({n: t.cpu().numpy() for n, t in grads.items()}
                 if want_acc and args.mode == "fwd_bwd" else None)

    # fwd alone (context line)
    torch.cuda.synchronize(dev)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    for _ in range(args.steps):
        ssd.ssd_fwd(q, k, v, la, h0, chunk=w.chunk, out=out)
    f1.record(stream)
    torch.cuda.synchronize(dev)
    fwd_ms = f0.elapsed_time(f1) / args.steps

    # peak device memory of one step (caller tensors + workspace high-water)
    dims = (w.B, w.L, w.G, w.H, w.dk, w.dv)
    memory = {
        "peak_mb_fwd": measure_peak(ssd, torch, dev,
                                    lambda: ssd.ssd_fwd(q, k, v, la, h0, chunk=w.chunk, out=out),
                                    resident_bytes(*dims, "fwd")) / MiB,
        "peak_mb_fwd_bwd": measure_peak(ssd, torch, dev, step,
                                        resident_bytes(*dims, args.mode) + residual_mb * MiB) / MiB,
        "residual_mb": residual_mb,
        "resident_mb_fwd_bwd": resident_bytes(*dims, "fwd_bwd") / MiB,
        "workspace_mb_fwd": ssd.ssd_fwd_workspace_bytes(*dims, w.chunk) / MiB,
        "workspace_mb_bwd": ssd.ssd_bwd_workspace_bytes(*dims, w.chunk) / MiB,
        "definition": "caller tensors the call touches + high-water of the library's "
                      "workspace pool during the call",
    }

    # end to end through the public API: every step copies its inputs from
    # pinned host memory to the device and its output and every gradient back
    # to pinned host memory.  Two sets of device buffers alternate between
    # steps, and the copies run on two copy streams (one per direction), so
    # that step i + 1's inputs arrive and step i - 1's results leave while
    # step i computes; events order each buffer's reuse.
    e2e = None
    if not args.no_e2e:
        fb = args.mode == "fwd_bwd"
        h_out = torch.empty(out.shape, pin_memory=True)
        h_grads = {n: torch.empty(t.shape, pin_memory=True) for n, t in grads.items()}
        ins = [[torch.empty_like(t) for t in (q, k, v, la, h0, dout)] for _ in range(2)]
        outs = [torch.empty_like(out) for _ in range(2)]
        gsets = [{n: torch.empty_like(t) for n, t in grads.items()} for _ in range(2)]
        # (the residual never leaves the device: one set per buffer set)
        res = [(torch.empty_like(saved) if saved is not None else None,
                torch.empty_like(hT) if hT is not None else None) for _ in range(2)]
        s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()
        in_ready, in_free = [ev(), ev()], [ev(), ev()]      # inputs landed / consumed
        res_ready, res_free = [ev(), ev()], [ev(), ev()]    # results written / copied out
        for e_ in in_free + res_free:
            e_.record(stream)

        def e2e_step(i):
            b = i & 1
            with torch.cuda.stream(s_in):
                s_in.wait_event(in_free[b])
                for d, hsrc in zip(ins[b], host if fb else host[:5]):
                    d.copy_(hsrc, non_blocking=True)
                in_ready[b].record(s_in)
            stream.wait_event(in_ready[b])
            stream.wait_event(res_free[b])
            if save:
                ssd.ssd_fwd_save(*ins[b][:5], chunk=w.chunk, out=outs[b], hT=res[b][1], saved=res[b][0])
                ssd.ssd_bwd_saved(*ins[b][:5], ins[b][5], None, res[b][1], res[b][0], chunk=w.chunk,
                                  grads=gsets[b])
            else:
                ssd.ssd_fwd(*ins[b][:5], chunk=w.chunk, out=outs[b])
                if fb:
                    ssd.ssd_bwd(*ins[b], chunk=w.chunk, grads=gsets[b])
            in_free[b].record(stream)
            res_ready[b].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(res_ready[b])
                h_out.copy_(outs[b], non_blocking=True)
                if fb:
                    for n in h_grads:
                        h_grads[n].copy_(gsets[b][n], non_blocking=True)
                res_free[b].record(s_out)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize(dev)
        barrier()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        s_in.wait_stream(stream)
        for i in range(args.steps):
            e2e_step(i)
        stream.wait_stream(s_out)
        g1.record(stream)
        torch.cuda.synchronize(dev)
        barrier()
        e2e_ms = max_over_ranks(g0.elapsed_time(g1) / args.steps, dev)
        h2d = sum(x.numel() * x.element_size() for x in (host if fb else host[:5]))
        d2h = h_out.numel() * 4 + (sum(x.numel() * x.element_size() for x in h_grads.values()) if fb else 0)
        e2e = {"value": job_tokens_per_s(w.tokens, world, e2e_ms), "unit": "tokens/s",
               "ms_per_step": e2e_ms, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "staging": "two device buffer sets; host-to-device and device-to-host copies "
                          "on their own streams, overlapping the neighbouring steps' compute"}

    if rank != 0:
        if world > 1:
            dist.destroy_process_group()
        return 0

    peaks = load_peaks()
    costs = kernel_costs(w, torch.cuda.get_device_properties(dev).multi_processor_count)
    side = tuple(k for k in SIDE_KERNELS if k in trace) if overlap_on else ()
    roof = kernel_roofline(trace, costs, peaks, w.name == WORKLOAD, exclude=side, rank=trace_iso)
    roof["timing"] = ("live, in the timed configuration" + (
        ": the backward runs its dk / dv passes on a second stream beside the dq pass, so a "
        "kernel's time includes the periods it shares the GPU with the other pass's kernels"
        if overlap_on else ""))
    roof["dominance"] = ("the most device time with the backward's passes serialised" if trace_iso
                         else "the most device time")
    if side:
        roof["dominance"] += ("; " + ", ".join(side) + " runs on the SMs the walks leave idle, beside "
                              "them (roofline_side)")
    roof_side = kernel_roofline({k: trace[k] for k in side}, costs, peaks, w.name == WORKLOAD) if side else None
    if roof_side is not None:
        roof_side["timing"] = "live: its launch spans most of the backward, on the SMs the walks leave idle"
    roof_iso = kernel_roofline(trace_iso, costs, peaks, w.name == WORKLOAD) if trace_iso else None
    if roof_iso is not None:
        roof_iso["timing"] = "the same steps with the backward's passes serialised (one kernel at a time)"

    bytes_fb, fl_fb, bytes_f, fl_f = step_totals(w)
    # the step's own algorithmic totals: a forward alone with --mode fwd
    step_bytes, step_flops = (bytes_f, fl_f) if args.mode == "fwd" else (bytes_fb, fl_fb)
    t_hbm = step_bytes / (peaks["hbm_gbs"] * 1e9)
    t_tc = step_flops / (peaks["bf16_tflops"] * TF32_OVER_BF16 * 1e12)
    step_roof_s = max(t_hbm, t_tc)
    value = job_tokens_per_s(w.tokens, world, ms)
    page_ms = (PAGE_FWD_MS if args.mode == "fwd" else PAGE_FWD_BWD_MS).get(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / (w.tokens / (page_ms / 1e3))) if page_ms else None,
        "dtype": "tf32" if (args.path == "tc" and w.chunk != 1) else "f32", "data": "synthetic",
        "config": {"workload": w.name, "mode": args.mode, "path": args.path, "B": w.B, "G": w.G,
                   "H": w.H, "L": w.L, "dk": w.dk, "dv": w.dv, "chunk": w.chunk,
                   "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                   "deterministic_group_sums": bool(args.deterministic),
                   "saved_states": bool(save),
                   "l2": l2_note(resident_bytes(w.B, w.L, w.G, w.H, w.dk, w.dv, args.mode))},
        "roofline": roof,
        "step_roofline": {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                          "alg_bytes": step_bytes, "alg_flops": step_flops,
                          "roofline_ms": step_roof_s * 1e3, "frac": step_roof_s * 1e3 / ms},
        "fwd": {"ms": fwd_ms, "tokens_per_s": w.tokens / (fwd_ms / 1e3),
                "frac_of_roofline": max(bytes_f / (peaks["hbm_gbs"] * 1e9),
                                        fl_f / (peaks["bf16_tflops"] * TF32_OVER_BF16 * 1e12)) / (fwd_ms / 1e3)},
        "repeats": repeats,
        "kernels": kernel_table(trace),
        "roofline_isolated": roof_iso,
        "roofline_side": roof_side,
        "kernels_isolated": kernel_table(trace_iso) if trace_iso else None,
        "gpu_launches": launches,
        "clocks": clk,
        "e2e": e2e,
        "memory": memory,
        "page_context": {"rtx3090_fwd_bwd_ms": PAGE_FWD_BWD_MS.get(w.name),
                         "rtx3090_fwd_ms": PAGE_FWD_MS.get(w.name),
                         "rtx3090_chunked_peak_mb": PAGE_PEAK_MB if w.name == WORKLOAD else None},
    }
    ref = None
    if world == 1 and not args.no_cpu_baseline:
        cb = cpu_oracle_sample(w)
        ref, ref_nb = cb.pop("_ref"), cb.pop("_nb")
        line["cpu_baseline"] = cb
    if want_acc:
        if ref is not None:
            acc = oracle_accuracy(w, res_out, res_grads, ref=(ref[0], ref[1] if res_grads else None),
                                  nb=ref_nb, residual_mb=residual_mb)
        else:
            acc = oracle_accuracy(w, res_out, res_grads, residual_mb=residual_mb)
        line.update(acc)
    print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
