#!/usr/bin/env python
"""Benchmark of the selective scan (Mamba S6) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one ssm_selective_scan_fwd call over one batch of the workload
(default: bf16, batch 4, L 2048, d_inner 1536, d_state 16, softplus(delta +
bias), gate), i.e. every step of the scan path. Rank 0 prints one JSON line.

* value: elements (batch * L * dim) per second over the K timed steps, inputs
  resident in HBM; the K steps rotate over several input sets whose total is
  larger than twice the L2 cache, so every step reads its inputs from HBM.
* e2e: the same metric through the same C-ABI call with host buffers:
  pinned host -> device copies of the step's inputs and a device -> host copy
  of its output inside the timed region, every step; the copies of one step
  overlap the compute of its neighbours (three streams, two buffer sets).
* roofline: the binding unit of the scan, the SFU: the SFU operations the
  method needs per call / average call time, against the measured ex2 rate;
  hbm_roofline: algorithmic bytes per call / call time against the measured
  HBM copy bandwidth; floors_us: the per-call floor of each unit.
* decode: the recurrent step ssm_state_update on the decode workload (batch
  256, dim 5120, N 16), rotating over several cached states.
* input_stage: the causal conv1d + SiLU (width 4) alone, fused in front of
  the scan, and as two calls (conv, then the scan on its output).
* train: training through the scan on the same workload, the checkpointing
  forward and the backward (every gradient), per call.
* bc_per_channel: the scan with per-channel B, C on the same shapes (bound by
  HBM: its roofline is the copy bandwidth).
* zoh: the scan with the exact zero-order-hold Bbar on the same workload,
  against the same SFU roofline.
  A side leg that fails reports {"error": ...} in its place; the headline
  line is still printed.
* cpu_baseline: the float64 CPU oracle timed on this host (rank 0, N = 1);
  check: its last pass compared with the last timed GPU output, every element.

N > 1 (torchrun): every rank runs its own replica of the workload on its own
GPU (the scan has no cross-channel exchange: weak scaling, no collective on
the data path); the timed region is bracketed by a barrier and the time is
the maximum over ranks. ``--impl reference`` times the float64 CPU oracle on
the same workload instead (rank 0 only).
"""
from __future__ import annotations

import argparse
import ctypes
import json
import math
import os
import statistics
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "selective-scan elems/s (B·L·D) and achieved HBM GB/s vs B300 peak, 1 GPU"
DEFAULT_WORKLOAD = "scan_bf16_b4_L2048_d1536_softplus"
DECODE_WORKLOAD = "decode_bf16_b256_d5120_x64"
L2_BYTES = 126 * 1024 * 1024
FALLBACK_HBM_GBS = 6400.0
NOMINAL_HBM_GBS = 7700.0      # B300 HBM3e datasheet bandwidth, for context beside the measured peak


def nominal(achieved_gbs):
    """The same achieved bandwidth as a fraction of the nominal HBM3e figure."""
    return {"nominal_peak": NOMINAL_HBM_GBS, "frac_of_nominal": achieved_gbs / NOMINAL_HBM_GBS}


# ---------------------------------------------------------------------------
# small utilities (host side)
# ---------------------------------------------------------------------------
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def reduce_max(value: float, group=None) -> float:
    """Maximum of a per-rank float over the process group (identity at N = 1)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX, group=group)
    return float(t.item())


def reduce_sum(value: float, group=None) -> float:
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return value
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM, group=group)
    return float(t.item())


def aggregate(units_this_rank: float, seconds_this_rank: float, group=None):
    """Whole-job throughput: units of all ranks / slowest rank's time."""
    total_units = reduce_sum(units_this_rank, group)
    slowest = reduce_max(seconds_this_rank, group)
    return total_units / slowest, slowest


class ClockSampler:
    """Samples the SM clock and the clock-event reasons during the timed region:
    through NVML when it initialises, else by running nvidia-smi in a loop."""

    REASONS = {
        0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
        0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
        0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
        0x100: "display_clock_setting",
    }

    def __init__(self, index: int, period_s: float = 0.02):
        self.index, self.period = index, period_s
        self.samples = []
        self.sm_max = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self.source = None

    def start(self):
        try:
            import pynvml
            pynvml.nvmlInit()
            self._nv = pynvml
            self._h = pynvml.nvmlDeviceGetHandleByIndex(self.index)
            self.sm_max = pynvml.nvmlDeviceGetMaxClockInfo(self._h, pynvml.NVML_CLOCK_SM)
            self.source = "nvml"
            self._thread = threading.Thread(target=self._run_nvml, daemon=True)
            self._thread.start()
            return self
        except Exception:
            pass
        try:
            import subprocess
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 "--query-gpu=clocks.sm,clocks.max.sm,clocks_event_reasons.active",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            self._thread = threading.Thread(target=self._run_smi, daemon=True)
            self._thread.start()
        except Exception:
            self.source = None
        return self

    def _run_nvml(self):
        nv = self._nv
        while not self._stop.is_set():
            try:
                sm = nv.nvmlDeviceGetClockInfo(self._h, nv.NVML_CLOCK_SM)
                r = nv.nvmlDeviceGetCurrentClocksEventReasons(self._h)
                self.samples.append((time.time(), sm, r))
            except Exception:
                pass
            time.sleep(self.period)

    def _run_smi(self):
        for line in self._proc.stdout:
            try:
                sm, smax, reasons = [x.strip() for x in line.split(",")]
                self.sm_max = int(float(smax))
                self.samples.append((time.time(), int(float(sm)), int(reasons, 16)))
            except Exception:
                pass
            if self._stop.is_set():
                break

    def stop(self):
        self._stop.set()
        if self._proc is not None:
            self._proc.terminate()
            try:
                self._proc.wait(timeout=2)
            except Exception:
                self._proc.kill()
        if self._thread:
            self._thread.join(timeout=2)

    def summary(self, t0=None, t1=None):
        if self.source is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["clock sampling unavailable"]}
        s = [x for x in self.samples if (t0 is None or x[0] >= t0) and (t1 is None or x[0] <= t1)]
        window = "timed"
        if len(s) < 3:
            s, window = self.samples, "warmup+timed"
        reasons = set()
        for _, _, r in s:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": statistics.median([x[1] for x in s]) if s else None,
                "sm_max_mhz": self.sm_max, "reasons": sorted(reasons), "samples": len(s),
                "window": window, "source": self.source}


# ---------------------------------------------------------------------------
# the GPU arm
# ---------------------------------------------------------------------------
def _upload(arr, dev):
    import numpy as np
    import torch
    if arr is None:
        return None
    if arr.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(dev).view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(arr)).to(dev)


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def bench_scan(args, rank, world, local):
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    spec = I.WORKLOADS[args.workload]
    inp = I.make_scan_inputs(spec)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    elems = spec.elements
    alg_bytes = I.algorithmic_bytes_scan(spec)

    # input sets, rotated so that no step finds its inputs in L2
    per_set = alg_bytes
    nsets = max(2, min(16, math.ceil(2 * L2_BYTES / per_set) + 1))
    base = {k: _upload(v, dev) for k, v in inp.items()}
    sets = []
    for i in range(nsets):
        s = {k: (None if base[k] is None else (base[k] if k in ("A", "D", "delta_bias")
                                                else base[k].clone()))
             for k in base}
        s["out"] = torch.empty_like(base["x"])
        s["fs"] = (torch.empty((spec.batch, spec.dim, spec.N), dtype=torch.float32, device=dev)
                   if spec.final_state else None)
        sets.append(s)
    plan = libssm.ssm_scan_plan(spec.batch, spec.L, spec.dim, spec.N, io)
    ws = libssm.alloc_workspace(spec.batch, spec.L, spec.dim, spec.N, io, dev)
    dims = libssm.make_dims(spec.batch, spec.L, spec.dim, spec.N, io,
                            None if ws is None else ws.data_ptr(),
                            0 if ws is None else ws.numel())
    stream = torch.cuda.current_stream(dev)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    fn = libssm.lib.ssm_selective_scan_fwd
    call_args = [(_vp(s["x"]), _vp(s["delta"]), _vp(s["A"]), _vp(s["B"]), _vp(s["C"]),
                  _vp(s["D"]), _vp(s["z"]), _vp(s["delta_bias"]), 1 if spec.delta_softplus else 0,
                  _vp(s["out"]), _vp(s["fs"]), ctypes.byref(dims), sptr) for s in sets]

    def step(i):
        rc = fn(*call_args[i % nsets])
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd")

    clocks = ClockSampler(local).start()
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()

    import torch.distributed as dist
    if dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(args.steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist.is_initialized():
        dist.barrier()
    clocks.stop()
    sec = e0.elapsed_time(e1) / 1e3
    value, slowest = aggregate(elems * args.steps, sec)
    status = libssm.ssm_get_device_status(spec.batch, spec.L, spec.dim, spec.N, io, ws)
    if status != 0:
        raise libssm.SSMError(status, "device status")

    per_call = sec / args.steps
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / per_call / 1e9
    res = {
        "value": value, "ms_per_step": slowest / args.steps * 1e3,
        "gbps": achieved,
        "roofline": dict(alu_roofline(spec, per_call, plan),
                         traffic=scan_traffic(args.workload)),
        "hbm_roofline": dict({"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                              "frac": achieved / peak, "traffic": scan_traffic(args.workload),
                              "peak_kind": peak_kind, "algorithmic_bytes_per_call": alg_bytes},
                             **nominal(achieved)),
        "floors_us": time_floors(spec, alg_bytes, peak),
        "gpu_launches": args.steps * plan["kernels"],
        "clocks": clocks.summary(t_wall0, t_wall1),
        "plan": plan,
        "input_sets": nsets,
    }

    # end to end: pinned host buffers; every step copies its inputs in and its
    # output out inside the timed region. The copies of one step overlap the
    # compute of its neighbours: three streams (in, compute, out), two device
    # buffer sets, ordered by events (a set's inputs are overwritten only after
    # the compute two steps back has read them, its output only after the copy
    # out two steps back has read it).
    host = {k: (None if base[k] is None else base[k].cpu().pin_memory())
            for k in ("x", "delta", "z", "B", "C")}
    e2e_sets = sets[:2]
    h_outs = [torch.empty(e2e_sets[0]["out"].shape, dtype=e2e_sets[0]["out"].dtype).pin_memory()
              for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    k_e2e = max(3, min(args.steps, 50))
    s_in, s_cmp, s_out = (torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev))
    cmp_ptr = ctypes.c_void_p(s_cmp.cuda_stream)
    cmp_args = [(_vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
                 _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]),
                 1 if spec.delta_softplus else 0, _vp(st["out"]), _vp(st["fs"]),
                 ctypes.byref(dims), cmp_ptr) for st in e2e_sets]
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_cmp = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def e2e_step(i):
        k = i % 2
        st = e2e_sets[k]
        if i >= 2:
            s_in.wait_event(ev_cmp[k])
        with torch.cuda.stream(s_in):
            for name, t in host.items():
                if t is not None:
                    st[name].copy_(t, non_blocking=True)
            ev_in[k].record(s_in)
        s_cmp.wait_event(ev_in[k])
        if i >= 2:
            s_cmp.wait_event(ev_out[k])
        rc = fn(*cmp_args[k])
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd")
        ev_cmp[k].record(s_cmp)
        s_out.wait_event(ev_cmp[k])
        with torch.cuda.stream(s_out):
            h_outs[k].copy_(st["out"], non_blocking=True)
            ev_out[k].record(s_out)

    for i in range(4):
        e2e_step(i)
    torch.cuda.synchronize()
    if dist.is_initialized():
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s_in)
    for i in range(k_e2e):
        e2e_step(i)
    e1.record(s_out)           # after the last copy out, which follows every other step
    torch.cuda.synchronize()
    e2e_sec = e0.elapsed_time(e1) / 1e3
    e2e_value, _ = aggregate(elems * k_e2e, e2e_sec)
    res["e2e"] = {"value": e2e_value, "unit": "elems/s", "h2d_bytes_per_step": h2d,
                  "d2h_bytes_per_step": d2h, "steps": k_e2e,
                  "pipelined": "copies in, compute and copies out of neighbouring steps "
                               "overlap (3 streams, 2 device buffer sets)"}

    # the last timed output (every set holds the same input values), for the
    # CPU-baseline leg to compare with the oracle's output on the host
    res["out_host"] = (sets[0]["out"].float().cpu().numpy().astype("float64")
                       if rank == 0 and world == 1 else None)
    del sets
    torch.cuda.empty_cache()
    legs = (("decode", not args.no_decode, lambda: bench_decode(args, dev, stream)),
            ("input_stage", not args.no_input_stage,
             lambda: bench_input_stage(args, spec, dev, stream)),
            ("train", not args.no_train and spec.N == 16,
             lambda: bench_train(args, spec, dev, stream)),
            ("bc_per_channel", not args.no_bcd and spec.N == 16,
             lambda: bench_bcd(args, spec, dev, stream)),
            ("zoh", not args.no_zoh and spec.N == 16,
             lambda: bench_zoh(args, spec, dev, stream)))
    for name, wanted, run in legs:
        if not wanted:
            continue
        try:
            res[name] = run()
        except Exception as e:   # a failed side leg is reported, not fatal to the headline
            res[name] = {"error": "%s: %s" % (type(e).__name__, e)}
    return res, spec


# SFU (MUFU) exponential rate of one B300 SM per clock, measured with a probe of
# back-to-back independent ex2.approx.ftz.f32 at full occupancy: 29.1 per SM per
# clock (the nominal 2 x 16 of Blackwell Ultra's doubled SFU), 148 SMs, at the
# 2032 MHz maximum SM clock. FP32 lanes per SM per clock: 128 (nominal).
EX2_PER_SM_CLK = 29.1
FP32_PER_SM_CLK = 128.0
SMS = 148
SM_MAX_MHZ = 2032.0


def exps_per_element(spec):
    """SFU operations the method needs per element: N exponentials for
    exp(dt A), two for softplus (e^v and the log) and two for the silu gate
    (e^-z and the reciprocal)."""
    return spec.N + (2 if spec.delta_softplus else 0) + (2 if spec.gate else 0)


def fp32_ops_per_element(spec):
    """FP32 operations the method needs per element: per state dt*A, (dt x)*B,
    the h update and the C.h readout (4N), plus dt*x, the D skip and the gate."""
    return 4 * spec.N + 3


def time_floors(spec, alg_bytes, hbm_gbs):
    """Lower bounds on one call (us) from each unit: HBM bytes, SFU exps, FP32 ops."""
    sfu = spec.elements * exps_per_element(spec) / (EX2_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6)
    fp32 = spec.elements * fp32_ops_per_element(spec) / (FP32_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6)
    return {"hbm": alg_bytes / (hbm_gbs * 1e9) * 1e6, "sfu": sfu * 1e6, "fp32": fp32 * 1e6}


# DRAM traffic of one scan call of the benchmark workload (both launches:
# chunk-state pass + output pass), dram__bytes_read.sum + dram__bytes_write.sum
# from the ncu capture summarised in profiles/scan_launches_b4_L2048_d1536.md.
# It holds only for the kernel source it was taken on: the sha256 below covers
# the scan kernel and the headers it includes; any change there reports null.
SCAN_TRAFFIC = {"workload": "scan_bf16_b4_L2048_d1536_softplus",
                "bytes_per_call": 43607808 + 5632 + 78255360 + 759552,
                "sha256": "a19f03079bff8d8bde37b0b179a0213db41b0d2c25bbae62266af8777d03099b"}
SCAN_SOURCES = ("scan_fwd.cu", "ssm_device.cuh", "ssm_tma.cuh", "ssm_tmap.h", "ssm_internal.h")


def scan_source_sha256():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_119_b300", "csrc")
    for name in SCAN_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def scan_traffic(spec_name):
    if (SCAN_TRAFFIC["bytes_per_call"] is None or spec_name != SCAN_TRAFFIC["workload"]
            or scan_source_sha256() != SCAN_TRAFFIC["sha256"]):
        return None
    return SCAN_TRAFFIC["bytes_per_call"]


def alu_roofline(spec, per_call_s, plan):
    """The binding roofline of the scan: the SFU operations the method needs
    per second against the SFU peak (the largest of the three floors)."""
    per_elem = exps_per_element(spec)
    achieved = spec.elements * per_elem / per_call_s / 1e12
    peak = EX2_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6 / 1e12
    return {"bound": "alu", "unit": "T SFU op/s", "achieved": achieved, "peak": peak,
            "frac": achieved / peak, "traffic": None, "sfu_ops_per_element": per_elem,
            "kernel": "scan_kernel, one ssm_selective_scan_fwd call (%d launch%s)"
                      % (plan["kernels"], "es" if plan["kernels"] > 1 else ""),
            "peak_basis": "measured ex2 rate 29.1 per SM per clock x 148 SMs x 2032 MHz"}


def output_check(got, ref):
    """Error statistics of the timed output against a reference output (both
    float64 host arrays): relative L2 and max |err| / (1 + |ref|)."""
    import numpy as np
    rel = float(np.linalg.norm(got - ref) / np.linalg.norm(ref))
    mx = float(np.max(np.abs(got - ref) / (1 + np.abs(ref))))
    return {"elements": int(got.size), "rel_l2": rel, "max_scaled_err": mx}


def bench_decode(args, dev, stream):
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    spec = I.WORKLOADS[DECODE_WORKLOAD]
    small = I.DecodeSpec(spec.batch, spec.dim, steps=4, seed=spec.seed)
    inp = I.make_decode_inputs(small)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    state_bytes = spec.batch * spec.dim * spec.N * 4
    nstates = max(2, min(8, math.ceil(2 * L2_BYTES / state_bytes) + 1))
    st0 = _upload(inp["state0"], dev)
    states = [st0.clone() for _ in range(nstates)]
    tok = [{k: _upload(inp[k][t], dev) for k in ("x", "delta", "z", "B", "C")} for t in range(4)]
    A, D = _upload(inp["A"], dev), _upload(inp["D"], dev)
    outs = [torch.empty_like(tok[0]["x"]) for _ in range(4)]
    dims = libssm.make_dims(spec.batch, 1, spec.dim, spec.N, io)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    fn = libssm.lib.ssm_state_update

    def step(i):
        t = tok[i % 4]
        rc = fn(_vp(states[i % nstates]), _vp(t["x"]), _vp(t["delta"]), _vp(A), _vp(t["B"]),
                _vp(t["C"]), _vp(D), _vp(t["z"]), None, 0, _vp(outs[i % 4]), ctypes.byref(dims),
                sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_state_update")

    n = max(64, min(args.steps, 2000))
    for i in range(max(args.warmup, 3)):
        step(i)
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / n
    alg = I.algorithmic_bytes_decode_step(spec)
    peak, kind = measured_peaks()
    gbs = alg / sec / 1e9
    return {"workload": DECODE_WORKLOAD, "metric": "decode elems/s (B*D per step)",
            "value": spec.batch * spec.dim / sec, "unit": "elems/s", "us_per_step": sec * 1e6,
            "us_per_64_steps": sec * 64 * 1e6, "states_rotated": nstates, "timed_steps": n,
            "roofline": dict({"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                              "frac": gbs / peak, "traffic": None, "peak_kind": kind,
                              "algorithmic_bytes_per_call": alg}, **nominal(gbs))}


def bench_input_stage(args, spec, dev, stream):
    """The Mamba block's input stage on the scan workload: the standalone
    causal conv1d + SiLU (width 4, with bias), the scan with that stage fused
    in front, and the two-call path (conv, then scan on its output), each over
    rotating input sets larger than twice the L2 cache."""
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    K = 4
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(spec.dim, K, True, seed=spec.seed + 7)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    conv_bytes = I.algorithmic_bytes_conv(spec.batch, spec.L, spec.dim, K, spec.io)
    scan_bytes = I.algorithmic_bytes_scan(spec)
    nsets = max(2, min(16, math.ceil(2 * L2_BYTES / scan_bytes) + 1))
    base = {k: _upload(v, dev) for k, v in inp.items()}
    wt, bt = _upload(w, dev), _upload(b, dev)
    sets = []
    for _ in range(nsets):
        st = {k: (None if base[k] is None else (base[k] if k in ("A", "D", "delta_bias")
                                                 else base[k].clone())) for k in base}
        st["u"] = torch.empty_like(base["x"])
        st["out"] = torch.empty_like(base["x"])
        sets.append(st)
    ws = libssm.alloc_workspace(spec.batch, spec.L, spec.dim, spec.N, io, dev)
    dims = libssm.make_dims(spec.batch, spec.L, spec.dim, spec.N, io,
                            None if ws is None else ws.data_ptr(),
                            0 if ws is None else ws.numel())
    plan = libssm.ssm_scan_plan(spec.batch, spec.L, spec.dim, spec.N, io)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    sp = 1 if spec.delta_softplus else 0

    def conv(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_causal_conv1d_silu(_vp(st["x"]), _vp(wt), _vp(bt), K, _vp(st["u"]),
                                               ctypes.byref(dims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_causal_conv1d_silu")

    def scan_args(st, xkey):
        return (_vp(st[xkey]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
                _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, _vp(st["out"]), None,
                ctypes.byref(dims), sptr)

    def fused(i):
        a = scan_args(sets[i % nsets], "x")
        rc = libssm.lib.ssm_selective_scan_fwd_conv(a[0], _vp(wt), _vp(bt), K, *a[1:])
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd_conv")

    def two_calls(i):
        conv(i)
        rc = libssm.lib.ssm_selective_scan_fwd(*scan_args(sets[i % nsets], "u"))
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd")

    def timed(fn, n):
        for i in range(max(args.warmup, 3)):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    n = max(64, min(args.steps, 2000))
    t_conv = timed(conv, n)
    t_fused = timed(fused, n)
    t_two = timed(two_calls, n)
    status = libssm.ssm_get_device_status(spec.batch, spec.L, spec.dim, spec.N, io, ws)
    if status != 0:
        raise libssm.SSMError(status, "device status")
    peak, kind = measured_peaks()
    gbs = conv_bytes / t_conv / 1e9
    elems = spec.elements
    return {"conv_width": K, "timed_calls": n, "input_sets": nsets,
            "conv": {"us_per_call": t_conv * 1e6, "value": elems / t_conv, "unit": "elems/s",
                     "roofline": dict({"bound": "hbm", "achieved": gbs, "peak": peak,
                                       "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                                       "peak_kind": kind,
                                       "algorithmic_bytes_per_call": conv_bytes},
                                      **nominal(gbs))},
            "fused_scan": {"us_per_call": t_fused * 1e6, "value": elems / t_fused,
                           "unit": "elems/s", "kernels_per_call": plan["kernels"]},
            "conv_then_scan": {"us_per_call": t_two * 1e6, "value": elems / t_two,
                               "unit": "elems/s", "kernels_per_call": plan["kernels"] + 1}}


def bench_train(args, spec, dev, stream):
    """Training through the scan on the scan workload: the checkpointing
    forward and the backward (every gradient), each over rotating input sets
    larger than twice the L2 cache; dout ~ N(0, 1) in the I/O dtype."""
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    inp = I.make_scan_inputs(spec)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    scan_bytes = I.algorithmic_bytes_scan(spec)
    nsets = max(2, min(8, math.ceil(2 * L2_BYTES / scan_bytes) + 1))
    base = {k: _upload(v, dev) for k, v in inp.items()}
    gen = torch.Generator(device=dev).manual_seed(spec.seed + 11)
    sets = []
    for _ in range(nsets):
        st = {k: (None if base[k] is None else (base[k] if k in ("A", "D", "delta_bias")
                                                 else base[k].clone())) for k in base}
        st["dout"] = torch.randn(base["x"].shape, generator=gen, device=dev).to(base["x"].dtype)
        st["ckpt"] = torch.empty((spec.batch, (spec.L + 7) // 8, spec.dim, spec.N),
                                 dtype=torch.float32, device=dev)
        sets.append(st)
    B_, L_, D_, N_ = spec.batch, spec.L, spec.dim, spec.N
    ws = libssm.alloc_workspace(B_, L_, D_, N_, io, dev)
    fdims = libssm.make_dims(B_, L_, D_, N_, io, None if ws is None else ws.data_ptr(),
                             0 if ws is None else ws.numel())
    nb = libssm.ssm_scan_bwd_workspace_bytes(B_, L_, D_, N_, io)
    bws = torch.empty(nb, dtype=torch.uint8, device=dev)
    bdims = libssm.make_dims(B_, L_, D_, N_, io, bws.data_ptr(), nb)
    out = torch.empty_like(base["x"])
    fs = torch.empty((B_, D_, N_), dtype=torch.float32, device=dev)
    g = {"dx": torch.empty_like(base["x"]), "ddelta": torch.empty_like(base["x"]),
         "dz": torch.empty_like(base["x"]) if base["z"] is not None else None,
         "dA": torch.empty((D_, N_), dtype=torch.float32, device=dev),
         "dB": torch.empty((B_, L_, N_), dtype=base["x"].dtype, device=dev),
         "dC": torch.empty((B_, L_, N_), dtype=base["x"].dtype, device=dev),
         "dD": torch.empty(D_, dtype=torch.float32, device=dev),
         "dbias": torch.empty(D_, dtype=torch.float32, device=dev)}
    sptr = ctypes.c_void_p(stream.cuda_stream)
    sp = 1 if spec.delta_softplus else 0

    def fwd(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_selective_scan_fwd_ckpt(
            _vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
            _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, None, _vp(out), _vp(fs),
            _vp(st["ckpt"]), ctypes.byref(fdims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd_ckpt")

    def bwd(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_selective_scan_bwd(
            _vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
            _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, _vp(st["ckpt"]),
            _vp(st["dout"]), None, _vp(g["dx"]), _vp(g["ddelta"]), _vp(g["dA"]), _vp(g["dB"]),
            _vp(g["dC"]), _vp(g["dD"]), _vp(g["dz"]), _vp(g["dbias"]), None,
            ctypes.byref(bdims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_bwd")

    def timed(fn, n):
        for i in range(max(args.warmup, 3)):
            fn(i)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for i in range(n):
            fn(i)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3 / n

    for i in range(nsets):          # every set's checkpoints exist before the first backward
        fwd(i)
    n = max(16, min(args.steps, 400))
    t_f = timed(fwd, n)
    t_b = timed(bwd, n)
    plan = libssm.ssm_scan_plan(B_, L_, D_, N_, io)
    elems = spec.elements
    return {"timed_calls": n, "input_sets": nsets, "dout": "N(0,1)",
            "fwd_ckpt": {"us_per_call": t_f * 1e6, "value": elems / t_f, "unit": "elems/s",
                         "kernels_per_call": plan["kernels"]},
            "bwd": {"us_per_call": t_b * 1e6, "value": elems / t_b, "unit": "elems/s",
                    "kernels_per_call": (2 if plan["nchunks"] > 1 else 1) + 1,
                    "workspace_bytes": nb},
            "step": {"us_per_call": (t_f + t_b) * 1e6, "value": elems / (t_f + t_b),
                     "unit": "elems/s"}}


def bench_bcd(args, spec, dev, stream):
    """The scan with per-channel B, C ([batch, L, dim, N], SSM_FLAG_BC_PER_CHANNEL)
    on the scan workload's shapes: bound by HBM (each channel reads its own
    2 N values per token), so its roofline is the measured copy bandwidth."""
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    inp = I.make_scan_inputs(spec)
    B4, C4 = I.make_bc_per_channel(spec)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    alg = I.algorithmic_bytes_scan_bcd(spec)
    nsets = 2 if alg > 2 * L2_BYTES else max(2, min(8, math.ceil(2 * L2_BYTES / alg) + 1))
    base = {k: _upload(v, dev) for k, v in inp.items()}
    base["B"], base["C"] = _upload(B4, dev), _upload(C4, dev)
    sets = []
    for i in range(nsets):
        st = {k: (None if base[k] is None else (base[k] if (k in ("A", "D", "delta_bias") or i == 0)
                                                 else base[k].clone())) for k in base}
        st["out"] = torch.empty_like(base["x"])
        sets.append(st)
    B_, L_, D_, N_ = spec.batch, spec.L, spec.dim, spec.N
    F = libssm.SSM_FLAG_BC_PER_CHANNEL
    ws = libssm.alloc_workspace(B_, L_, D_, N_, io, dev, flags=F)
    dims = libssm.make_dims(B_, L_, D_, N_, io, None if ws is None else ws.data_ptr(),
                            0 if ws is None else ws.numel(), flags=F)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    sp = 1 if spec.delta_softplus else 0

    def call(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_selective_scan_fwd(
            _vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
            _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, _vp(st["out"]), None,
            ctypes.byref(dims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd (per-channel B, C)")

    for i in range(max(args.warmup, 3)):
        call(i)
    torch.cuda.synchronize()
    n = max(16, min(args.steps, 400))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / n
    peak, kind = measured_peaks()
    gbs = alg / sec / 1e9
    plan = libssm.ssm_scan_plan(B_, L_, D_, N_, io, flags=F)
    return {"us_per_call": sec * 1e6, "value": spec.elements / sec, "unit": "elems/s",
            "timed_calls": n, "input_sets": nsets, "kernels_per_call": plan["kernels"],
            "roofline": dict({"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                              "frac": gbs / peak, "traffic": None, "peak_kind": kind,
                              "algorithmic_bytes_per_call": alg}, **nominal(gbs))}


def bench_zoh(args, spec, dev, stream):
    """The scan with the exact zero-order-hold Bbar (SSM_FLAG_ZOH) on the scan
    workload: the same inputs, bytes and SFU operations per element as the
    first-order scan (the hold term (e^{dt A} - 1)/A reuses the exponential),
    plus its FP32 work; reported against the same SFU roofline."""
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    inp = I.make_scan_inputs(spec)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    alg = I.algorithmic_bytes_scan(spec)
    nsets = max(2, min(16, math.ceil(2 * L2_BYTES / alg) + 1))
    base = {k: _upload(v, dev) for k, v in inp.items()}
    sets = []
    for i in range(nsets):
        st = {k: (None if base[k] is None else (base[k] if (k in ("A", "D", "delta_bias") or i == 0)
                                                 else base[k].clone())) for k in base}
        st["out"] = torch.empty_like(base["x"])
        sets.append(st)
    B_, L_, D_, N_ = spec.batch, spec.L, spec.dim, spec.N
    F = libssm.SSM_FLAG_ZOH
    ws = libssm.alloc_workspace(B_, L_, D_, N_, io, dev, flags=F)
    dims = libssm.make_dims(B_, L_, D_, N_, io, None if ws is None else ws.data_ptr(),
                            0 if ws is None else ws.numel(), flags=F)
    sptr = ctypes.c_void_p(stream.cuda_stream)
    sp = 1 if spec.delta_softplus else 0

    def call(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_selective_scan_fwd(
            _vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
            _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, _vp(st["out"]), None,
            ctypes.byref(dims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd (exact zero-order hold)")

    for i in range(max(args.warmup, 3)):
        call(i)
    torch.cuda.synchronize()
    n = max(16, min(args.steps, 400))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / n
    plan = libssm.ssm_scan_plan(B_, L_, D_, N_, io, flags=F)
    roof = alu_roofline(spec, sec, plan)
    roof["kernel"] = roof["kernel"].replace("scan_kernel", "scan_kernel with the ZOH flag")
    return {"us_per_call": sec * 1e6, "value": spec.elements / sec, "unit": "elems/s",
            "timed_calls": n, "input_sets": nsets, "kernels_per_call": plan["kernels"],
            "roofline": roof, "algorithmic_bytes_per_call": alg}


# ---------------------------------------------------------------------------
# the CPU oracle arm
# ---------------------------------------------------------------------------
def cpu_oracle_rate(spec, inp, min_seconds: float, max_passes: int = 100):
    """Time the float64 oracle over whole passes of the workload on every host
    thread until min_seconds have passed (at least one pass). Returns the rate,
    the threads, the passes, the seconds and the output of the last pass."""
    import oracle
    from selective_state_space_119_b300 import inputs as I
    threads = oracle.default_threads()
    args = (I.widen(inp["x"]), I.widen(inp["delta"]), inp["A"], I.widen(inp["B"]),
            I.widen(inp["C"]))
    kw = dict(D=inp["D"], z=I.widen(inp["z"]), delta_bias=inp["delta_bias"],
              delta_softplus=spec.delta_softplus, nthreads=threads)
    passes, t0 = 0, time.perf_counter()
    while True:
        out, _ = oracle.selective_scan(*args, **kw)
        passes += 1
        el = time.perf_counter() - t0
        if el >= min_seconds or passes >= max_passes:
            break
    return spec.elements * passes / el, threads, passes, el, out


def run_reference(args, rank, world, budget_s: float = 120.0):
    """The float64 CPU oracle as the reference arm. One step = the oracle over
    every token and batch row of a rotating subset of channels, the subset
    sized so that warm-up + K steps stay within about budget_s seconds."""
    import numpy as np
    import oracle
    from selective_state_space_119_b300 import inputs as I
    if rank != 0:
        return
    spec = I.WORKLOADS[args.workload]
    inp = I.make_scan_inputs(spec)
    threads = oracle.default_threads()
    B, C = I.widen(inp["B"]), I.widen(inp["C"])

    def run(dsel):
        oracle.selective_scan(
            I.widen(inp["x"][:, :, dsel]), I.widen(inp["delta"][:, :, dsel]), inp["A"][dsel],
            B, C, D=None if inp["D"] is None else inp["D"][dsel],
            z=None if inp["z"] is None else I.widen(inp["z"][:, :, dsel]),
            delta_bias=None if inp["delta_bias"] is None else inp["delta_bias"][dsel],
            delta_softplus=spec.delta_softplus, nthreads=threads)
        return spec.batch * spec.L * len(dsel)

    probe = np.arange(0, spec.dim, max(1, spec.dim // 64))
    t0 = time.perf_counter()
    n = run(probe)
    per_elem = (time.perf_counter() - t0) / n
    nsteps = args.steps + args.warmup
    per_step = max(1, int(budget_s / nsteps / per_elem / (spec.batch * spec.L)))
    per_step = min(spec.dim, per_step)
    for w in range(args.warmup):
        run(np.arange(w * per_step, (w + 1) * per_step) % spec.dim)
    done, t0 = 0, time.perf_counter()
    for k in range(args.steps):
        done += run(np.arange(k * per_step, (k + 1) * per_step) % spec.dim)
    el = time.perf_counter() - t0
    rate = done / el
    sample = ("per step: %d of %d channels (rotating), every batch row and token; "
              "float64 oracle on %d host threads" % (per_step, spec.dim, threads))
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "elems/s",
            "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": el / args.steps * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(spec),
            "cpu_baseline": {"value": rate, "unit": "elems/s", "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": rate, "unit": "elems/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def workload_config(spec):
    return {"workload": _name_of(spec),
            "batch": spec.batch, "seqlen": spec.L, "dim": spec.dim, "dstate": spec.N,
            "io": spec.io, "delta": "softplus(u + bias)" if spec.delta_softplus else
            "log-uniform [%g, %g]" % (spec.delta_lo, spec.delta_hi),
            "A": spec.A_kind, "D": spec.D_kind, "gate": spec.gate,
            "final_state": spec.final_state,
            "l2": "rotating input sets, total > 2x the 126 MB L2 (no L2 reuse between steps)"}


def _name_of(spec):
    from selective_state_space_119_b300 import inputs as I
    for k, v in I.WORKLOADS.items():
        if v == spec:
            return k
    return "custom"


# ---------------------------------------------------------------------------
def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-decode", action="store_true")
    ap.add_argument("--no-input-stage", action="store_true",
                    help="skip the conv1d + SiLU input-stage timings")
    ap.add_argument("--no-train", action="store_true",
                    help="skip the training (checkpointing forward + backward) timings")
    ap.add_argument("--no-bcd", action="store_true",
                    help="skip the per-channel B, C scan timing")
    ap.add_argument("--no-zoh", action="store_true",
                    help="skip the exact zero-order-hold scan timing")
    ap.add_argument("--cpu-seconds", type=float, default=8.0,
                    help="minimum wall time of the CPU oracle baseline")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    rank, world, local = dist_env()
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import torch.distributed as dist
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    from selective_state_space_119_b300 import build
    if rank == 0 or world == 1:
        build.build(quiet=True)
    if world > 1:
        dist.barrier()

    res, spec = bench_scan(args, rank, world, local)
    if rank == 0:
        line = {"metric": METRIC, "value": res["value"], "unit": "elems/s", "n_gpus": world,
                "steps": args.steps, "warmup": args.warmup, "ms_per_step": res["ms_per_step"],
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
                "dtype": "f32", "io_dtype": spec.io, "data": "synthetic",
                "config": workload_config(spec), "gbps": res["gbps"],
                "roofline": res["roofline"], "hbm_roofline": res["hbm_roofline"],
                "floors_us": res["floors_us"], "e2e": res["e2e"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
                "plan": res["plan"], "check": None}
        for leg in ("decode", "input_stage", "train", "bc_per_channel", "zoh"):
            if leg in res:
                line[leg] = res[leg]
        if world == 1:
            from selective_state_space_119_b300 import inputs as I
            inp = I.make_scan_inputs(spec)
            rate, threads, passes, el, ref = cpu_oracle_rate(spec, inp, args.cpu_seconds)
            line["cpu_baseline"] = {
                "value": rate, "unit": "elems/s", "cores": threads, "kind": "oracle",
                "sample": "whole workload (%d x %d x %d), %d pass(es), %.1f s, all host threads"
                          % (spec.batch, spec.L, spec.dim, passes, el)}
            # the oracle's last pass against the last timed GPU output, every element
            line["check"] = dict(output_check(res["out_host"], ref),
                                 against="the cpu_baseline leg's oracle output")
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
