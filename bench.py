#!/usr/bin/env python
"""Benchmark of the selective scan (Mamba S6) on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]

One step is one ssm_selective_scan_fwd call over one batch of the workload
(default: the long-sequence workload, bf16, batch 1, L 131072, d_inner 5120,
d_state 16, delta log-uniform in [1e-4, 1e-2], A = -(n + 1), D = 1, gate,
final state), i.e. every step of the scan path. Rank 0 prints one JSON line.

* value: elements (batch * L * dim) per second over the K timed steps, inputs
  resident in HBM; the K steps rotate over input sets whose total is larger
  than twice the L2 cache, so every step reads its inputs from HBM.
* e2e: the same metric through the same C-ABI call with host buffers:
  pinned host -> device copies of the step's inputs and a device -> host copy
  of its output inside the timed region, every step; the copies of one step
  overlap the compute of its neighbours (three streams, two buffer sets).
* roofline: the unit with the highest floor for the workload (HBM bytes, SFU
  exponentials or FP32 operations the method needs), its achieved rate
  against its measured peak; hbm_roofline: algorithmic bytes per call / call
  time against the measured HBM copy bandwidth; floors_us: each unit's floor.
* check / cpu_baseline: the float64 CPU oracle over blocks of channels (every
  batch row and token) in a seeded order, within a time budget, compared
  element by element with the last timed output and final state; its rate on
  this host's cores (rank 0, N = 1).
* side: the other two bf16 scan workloads (batch 8, L 4096, d_inner 2048; and
  batch 4, L 2048, d_inner 1536 with softplus(delta + bias) and a general A),
  each with its own value, roofline and check.
* decode: the recurrent step ssm_state_update on the decode workload (batch
  256, dim 5120, N 16), rotating over several cached states.
* ssd: Mamba-2's SSD layer on the tensor cores (batch 16, L 8192, 8 heads of
  64 channels, d_state 128): its tensor-pipe and HBM rooflines and parity on
  sampled heads against the oracle.
* input_stage, train, bc_per_channel, zoh (on the batch 4, L 2048 workload):
  the causal conv1d + SiLU (width 4) alone, fused and as two calls; training
  through the scan (checkpointing forward and backward); the scan with
  per-channel B, C (HBM-bound); the scan with the exact zero-order hold.
  A side leg that fails reports {"error": ...} in its place; the headline
  line is still printed.

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
DEFAULT_WORKLOAD = "scan_bf16_b1_L131072_d5120"
# the other scan workloads, timed as side legs with their own roofline and check
SIDE_WORKLOADS = ("scan_bf16_b8_L4096_d2048", "scan_bf16_b4_L2048_d1536_softplus")
# the workload of the input-stage, training, per-channel B, C and exact-ZOH legs
LEG_WORKLOAD = "scan_bf16_b4_L2048_d1536_softplus"
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


def _scan_sets(spec, inp, dev, nsets):
    """nsets device copies of the per-element inputs (A, D and the bias are
    shared), each with its own output and final-state buffers."""
    import torch
    base = {k: _upload(v, dev) for k, v in inp.items()}
    sets = []
    for i in range(nsets):
        s = {k: (None if base[k] is None else (base[k] if (k in ("A", "D", "delta_bias") or i == 0)
                                                else base[k].clone()))
             for k in base}
        s["out"] = torch.empty_like(base["x"])
        s["fs"] = (torch.empty((spec.batch, spec.dim, spec.N), dtype=torch.float32, device=dev)
                   if spec.final_state else None)
        sets.append(s)
    return base, sets


def time_scan(name, args, rank, world, dev, steps, warmup, e2e=False):
    """Time ssm_selective_scan_fwd on one workload: `steps` calls over rotating
    input sets whose total exceeds twice the L2 (a single set already does for
    the long-sequence workload), CUDA events on the launching stream, barrier
    and maximum over ranks. Returns the result dict, the host inputs and the
    set whose output the oracle check reads."""
    import torch
    import torch.distributed as dist
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    spec = I.WORKLOADS[name]
    inp = I.make_scan_inputs(spec)
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    elems = spec.elements
    alg_bytes = I.algorithmic_bytes_scan(spec)
    nsets = max(2, min(16, math.ceil(2 * L2_BYTES / alg_bytes) + 1))
    base, sets = _scan_sets(spec, inp, dev, nsets)
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

    clocks = ClockSampler(dev.index if dev.index is not None else 0).start()
    for i in range(warmup):
        step(i)
    torch.cuda.synchronize()
    if dist.is_initialized():
        dist.barrier()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize()
    t_wall1 = time.time()
    if dist.is_initialized():
        dist.barrier()
    clocks.stop()
    sec = e0.elapsed_time(e1) / 1e3
    value, slowest = aggregate(elems * steps, sec)
    status = libssm.ssm_get_device_status(spec.batch, spec.L, spec.dim, spec.N, io, ws)
    if status != 0:
        raise libssm.SSMError(status, "device status")
    # the set the last timed step wrote (every set holds the same input values)
    last = sets[(steps - 1) % nsets]

    per_call = sec / steps
    peak, peak_kind = measured_peaks()
    achieved = alg_bytes / per_call / 1e9
    hbm = dict({"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak, "traffic": scan_traffic(name),
                "peak_kind": peak_kind, "algorithmic_bytes_per_call": alg_bytes},
               **nominal(achieved))
    res = {
        "workload": name, "value": value, "unit": "elems/s",
        "ms_per_step": slowest / steps * 1e3, "steps": steps, "warmup": warmup,
        "gbps": achieved,
        "roofline": binding_roofline(spec, per_call, plan, hbm, peak),
        "hbm_roofline": hbm,
        "floors_us": time_floors(spec, alg_bytes, peak),
        "gpu_launches": steps * plan["kernels"],
        "clocks": clocks.summary(t_wall0, t_wall1),
        "plan": plan, "input_sets": nsets, "config": workload_config(spec),
    }
    if e2e:
        res["e2e"] = time_scan_e2e(spec, sets, base, dims, fn, steps, dev)
    keep = {"out": last["out"], "fs": last["fs"]}
    del sets, base, call_args
    return res, spec, inp, keep


def time_scan_e2e(spec, sets, base, dims, fn, steps, dev):
    """The same metric through the same C-ABI call with host buffers: pinned
    host -> device copies of the step's inputs and a device -> host copy of its
    output inside the timed region, every step. The copies of one step overlap
    the compute of its neighbours: three streams (in, compute, out), two device
    buffer sets, ordered by events (a set's inputs are overwritten only after
    the compute two steps back has read them, its output only after the copy
    out two steps back has read it)."""
    import torch
    import torch.distributed as dist
    from selective_state_space_119_b300 import libssm
    host = {k: (None if base[k] is None else base[k].cpu().pin_memory())
            for k in ("x", "delta", "z", "B", "C")}
    e2e_sets = sets[:2]
    h_outs = [torch.empty(e2e_sets[0]["out"].shape, dtype=e2e_sets[0]["out"].dtype).pin_memory()
              for _ in range(2)]
    h2d = sum(t.numel() * t.element_size() for t in host.values() if t is not None)
    d2h = h_outs[0].numel() * h_outs[0].element_size()
    k_e2e = max(3, min(steps, 50))
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
    e2e_value, _ = aggregate(spec.elements * k_e2e, e2e_sec)
    out = {"value": e2e_value, "unit": "elems/s", "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "steps": k_e2e,
           "pipelined": "copies in, compute and copies out of neighbouring steps "
                        "overlap (3 streams, 2 device buffer sets)"}
    del host, h_outs
    return out


def oracle_check(spec, inp, keep, budget_s, block=256, seed=0):
    """The float64 oracle over blocks of channels (every batch row and token),
    taken in a seeded random order until budget_s seconds of oracle time have
    passed (at least one block), compared element by element with the GPU's
    timed output and final state. Returns (check, cpu_baseline): the errors,
    and the oracle's rate over the channels it ran (its own call time only)."""
    import numpy as np
    import oracle
    from selective_state_space_119_b300 import inputs as I
    threads = oracle.default_threads()
    nblk = (spec.dim + block - 1) // block
    order = np.random.Generator(np.random.PCG64(seed)).permutation(nblk)
    B, C = I.widen(inp["B"]), I.widen(inp["C"])
    se = sr = 0.0
    mx = fs_mx = 0.0
    done = 0
    osec = 0.0
    for bi in order:
        d0, d1 = int(bi) * block, min(spec.dim, (int(bi) + 1) * block)
        xs = I.widen(inp["x"][:, :, d0:d1])
        ds = I.widen(inp["delta"][:, :, d0:d1])
        zs = None if inp["z"] is None else I.widen(inp["z"][:, :, d0:d1])
        t0 = time.perf_counter()
        ref, rfs = oracle.selective_scan(
            xs, ds, inp["A"][d0:d1], B, C,
            D=None if inp["D"] is None else inp["D"][d0:d1], z=zs,
            delta_bias=None if inp["delta_bias"] is None else inp["delta_bias"][d0:d1],
            delta_softplus=spec.delta_softplus, nthreads=threads)
        osec += time.perf_counter() - t0
        got = keep["out"][:, :, d0:d1].float().cpu().numpy().astype(np.float64)
        err = got - ref
        se += float(np.sum(err * err))
        sr += float(np.sum(ref * ref))
        mx = max(mx, float(np.max(np.abs(err) / (1 + np.abs(ref)))))
        if keep["fs"] is not None:
            gfs = keep["fs"][:, d0:d1, :].cpu().numpy().astype(np.float64)
            fs_mx = max(fs_mx, float(np.max(np.abs(gfs - rfs) / (1 + np.abs(rfs)))))
        done += d1 - d0
        if osec >= budget_s:
            break
    elems = spec.batch * spec.L * done
    check = {"elements": elems, "channels": done, "of_channels": spec.dim,
             "rel_l2": math.sqrt(se / sr) if sr > 0 else 0.0, "max_scaled_err": mx,
             "against": "the float64 oracle (cpu_baseline leg) on the same inputs",
             "tolerance": ({"rel_l2": 3e-3, "max_scaled_err": 2e-2} if spec.io == "bf16"
                           else {"max_scaled_err": 1e-4})}
    if keep["fs"] is not None:
        check["final_state_max_scaled_err"] = fs_mx
        check["final_state_tolerance"] = 1e-4
    cpu = {"value": elems / osec, "unit": "elems/s", "cores": threads, "kind": "oracle",
           "sample": "%d of %d channels (blocks of %d in a seeded order, every batch row and "
                     "token), %.1f s of float64 oracle on %d host threads"
                     % (done, spec.dim, block, osec, threads)}
    return check, cpu


def bench_scan(args, rank, world, local):
    import torch
    from selective_state_space_119_b300 import inputs as I

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    check_here = rank == 0 and world == 1
    res, spec, inp, keep = time_scan(args.workload, args, rank, world, dev, args.steps,
                                     args.warmup, e2e=True)
    if check_here:
        res["check"], res["cpu_baseline"] = oracle_check(spec, inp, keep, args.cpu_seconds)
    del keep, inp
    torch.cuda.empty_cache()

    # the other scan workloads, each with its own roofline and oracle check
    side = {}
    if not args.no_side:
        for name in SIDE_WORKLOADS:
            if name == args.workload:
                continue
            try:
                r, sspec, sinp, skeep = time_scan(name, args, rank, world, dev,
                                                  max(args.steps, 10), args.warmup)
                if check_here:
                    r["check"], r["cpu_baseline"] = oracle_check(sspec, sinp, skeep,
                                                                 args.cpu_seconds / 4)
                for k in ("clocks", "steps", "warmup"):
                    r.pop(k, None)
                side[name] = r
                del skeep, sinp
            except Exception as e:   # a failed side leg is reported, not fatal
                side[name] = {"error": "%s: %s" % (type(e).__name__, e)}
            torch.cuda.empty_cache()
    res["side"] = side

    lspec = I.WORKLOADS[LEG_WORKLOAD]
    legs = (("decode", not args.no_decode, lambda: bench_decode(args, dev, stream)),
            ("input_stage", not args.no_input_stage,
             lambda: bench_input_stage(args, lspec, dev, stream)),
            ("train", not args.no_train, lambda: bench_train(args, lspec, dev, stream)),
            ("bc_per_channel", not args.no_bcd, lambda: bench_bcd(args, lspec, dev, stream)),
            ("zoh", not args.no_zoh, lambda: bench_zoh(args, lspec, dev, stream)),
            ("ssd", not args.no_ssd, lambda: bench_ssd(args, dev, stream)))
    for name, wanted, run in legs:
        if not wanted:
            continue
        try:
            res[name] = run()
        except Exception as e:   # a failed side leg is reported, not fatal to the headline
            res[name] = {"error": "%s: %s" % (type(e).__name__, e)}
        torch.cuda.empty_cache()
    return res, spec


# SFU (MUFU) exponential rate of one B300 SM per clock and FP32 lane
# operations per SM per clock, measured with a probe at full occupancy: 148 x 8
# CTAs of 256 threads, each thread running 16 independent chains of
# ex2.approx.ftz.f32, fma.rn.f32 or fma.rn.f32x2 for 2048 x 4 steps, cycles
# taken from each SM's own clock counter (first start to last end of its
# CTAs), the instruction counts confirmed with ncu (sm__inst_executed_pipe_fma,
# _fmaheavy, _fmalite, _xu). Results: ex2 32.0, FFMA 125.2 and FFMA2 127.6 FP32
# operations per SM per clock (an FFMA2 occupies both FMA half-pipes for one
# issue: packing halves the issue slots, not the pipe time), 8 FFMA2 + 2 ex2
# mixed 116. 148 SMs; the 2032 MHz maximum SM clock.
EX2_PER_SM_CLK = 32.0
FP32_PER_SM_CLK = 128.0
SMS = 148
SM_MAX_MHZ = 2032.0


def structured_A(spec):
    """A[d, n] = a_d (n + 1): exp(dt A[d, :]) is the powers 1..N of one
    exponential per channel and token."""
    return spec.A_kind == "s4d"


def exps_per_element(spec):
    """SFU operations the method needs per element: the exponentials of
    exp(dt A) (N of them, or one when A[d, n] = a_d (n + 1), whose powers give
    the rest), two for softplus (e^v and the log) and two for the silu gate
    (e^-z and the reciprocal)."""
    return ((1 if structured_A(spec) else spec.N) + (2 if spec.delta_softplus else 0)
            + (2 if spec.gate else 0))


def fp32_ops_per_element(spec):
    """FP32 operations the method needs per element: per state dt*A (or the
    power that replaces it), (dt x)*B, the h update and the C.h readout (4N),
    plus dt*x, the D skip and the gate."""
    return 4 * spec.N + 3


def time_floors(spec, alg_bytes, hbm_gbs):
    """Lower bounds on one call (us) from each unit: HBM bytes, SFU exps, FP32 ops."""
    sfu = spec.elements * exps_per_element(spec) / (EX2_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6)
    fp32 = spec.elements * fp32_ops_per_element(spec) / (FP32_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6)
    return {"hbm": alg_bytes / (hbm_gbs * 1e9) * 1e6, "sfu": sfu * 1e6, "fp32": fp32 * 1e6}


# DRAM traffic of one scan call (every launch of the call),
# dram__bytes_read.sum + dram__bytes_write.sum from one ncu capture per
# workload (a capture of a shorter sequence scaled by the tokens, where the
# full workload is too large to capture). A figure holds only for the kernel
# source it was taken on: the sha256 covers the scan kernel and the headers it
# includes; any change there reports null.
SCAN_TRAFFIC = {
    # both passes at L 16384 (the same 37-chunk plan, 1/8 of the tokens):
    # 339,388,672 + 686,803,200 bytes, scaled by 8 to L 131072
    "scan_bf16_b1_L131072_d5120": {"bytes_per_call": 8 * (339388672 + 686803200),
                                   "sha256": "314a8fdff130936bcf5a0e6edbe36697223d4209644377eb20e37eae59544864"},
}
SCAN_SOURCES = ("scan16.cu", "ssm_device.cuh", "ssm_tma.cuh", "ssm_tmap.h")


def scan_source_sha256():
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "selective_state_space_119_b300", "csrc")
    for name in SCAN_SOURCES:
        with open(os.path.join(csrc, name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()


def scan_traffic(spec_name):
    t = SCAN_TRAFFIC.get(spec_name)
    if t is None or scan_source_sha256() != t["sha256"]:
        return None
    return t["bytes_per_call"]


def binding_roofline(spec, per_call_s, plan, hbm, hbm_peak):
    """The roofline of the unit whose floor is highest for this workload: HBM
    (algorithmic bytes), the SFU (exponentials the method needs) or the FP32
    pipe (its FP32 operations), each achieved rate against that unit's peak."""
    floors = time_floors(spec, hbm["algorithmic_bytes_per_call"], hbm_peak)
    unit = max(floors, key=floors.get)
    kernel = ("scan_kernel, one ssm_selective_scan_fwd call (%d launch%s)"
              % (plan["kernels"], "es" if plan["kernels"] > 1 else ""))
    if unit == "hbm":
        return dict(hbm, kernel=kernel)
    if unit == "sfu":
        per_elem = exps_per_element(spec)
        peak = EX2_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6 / 1e12
        basis = "measured ex2 rate %.1f per SM per clock x %d SMs x %.0f MHz" % (
            EX2_PER_SM_CLK, SMS, SM_MAX_MHZ)
        name = "T SFU op/s"
    else:
        per_elem = fp32_ops_per_element(spec)
        peak = FP32_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6 / 1e12
        basis = "measured FP32 rate %.0f lane-ops per SM per clock x %d SMs x %.0f MHz" % (
            FP32_PER_SM_CLK, SMS, SM_MAX_MHZ)
        name = "T FP32 op/s"
    achieved = spec.elements * per_elem / per_call_s / 1e12
    return {"bound": "alu", "unit": name, "achieved": achieved, "peak": peak,
            "frac": achieved / peak, "traffic": hbm["traffic"], "ops_per_element": per_elem,
            "pipe": unit, "kernel": kernel, "peak_basis": basis}


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

    # the stage's backward: dx, dconv_w, dconv_b for dLoss/du = the u of a set
    cdims = libssm.make_dims(spec.batch, spec.L, spec.dim, 16, io)
    nbw = int(libssm.lib.ssm_causal_conv1d_silu_bwd_workspace_bytes(ctypes.byref(cdims), K))
    bws = torch.empty(nbw, dtype=torch.uint8, device=dev)
    bdims = libssm.make_dims(spec.batch, spec.L, spec.dim, 16, io, bws.data_ptr(), nbw)
    dxs = torch.empty_like(sets[0]["x"])
    dwt = torch.empty((spec.dim, K), dtype=torch.float32, device=dev)
    dbt = torch.empty((spec.dim,), dtype=torch.float32, device=dev)

    def conv_bwd(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_causal_conv1d_silu_bwd(
            _vp(st["x"]), _vp(wt), _vp(bt), K, _vp(st["u"]), _vp(dxs), _vp(dwt), _vp(dbt),
            ctypes.byref(bdims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_causal_conv1d_silu_bwd")

    n = max(64, min(args.steps, 2000))
    t_conv = timed(conv, n)
    t_fused = timed(fused, n)
    t_two = timed(two_calls, n)
    t_cbwd = timed(conv_bwd, n)
    status = libssm.ssm_get_device_status(spec.batch, spec.L, spec.dim, spec.N, io, ws)
    if status != 0:
        raise libssm.SSMError(status, "device status")
    peak, kind = measured_peaks()
    gbs = conv_bytes / t_conv / 1e9
    elems = spec.elements
    # the backward reads x and du and writes dx per element (the taps and the
    # per-block shares of dw, dbias are small)
    bwd_bytes = 3 * elems * (2 if spec.io == "bf16" else 4) + 2 * spec.dim * (K + 1) * 4
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
                               "unit": "elems/s", "kernels_per_call": plan["kernels"] + 1},
            "conv_bwd": {"us_per_call": t_cbwd * 1e6, "value": elems / t_cbwd, "unit": "elems/s",
                         "kernels_per_call": 2,
                         "roofline": dict({"bound": "hbm", "achieved": bwd_bytes / t_cbwd / 1e9,
                                           "peak": peak, "unit": "GB/s",
                                           "frac": bwd_bytes / t_cbwd / 1e9 / peak,
                                           "traffic": None, "peak_kind": kind,
                                           "algorithmic_bytes_per_call": bwd_bytes},
                                          **nominal(bwd_bytes / t_cbwd / 1e9))}}


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
    # The backward's binding unit: its FP32 operations per element are the
    # forward's 4N + 3 (the states recomputed from the checkpoints) plus 8 per
    # state for the adjoint sweep (dh carried back through a and fed by C dy;
    # the dC, dB, dt and dA terms) plus 7 per element (dx, dz, the softplus and
    # gate derivatives); its SFU operations the forward's N + 4 plus one (the
    # softplus derivative's sigmoid).
    fp32 = (4 * spec.N + 3) + 8 * spec.N + 7
    sfu = spec.N + (2 if spec.delta_softplus else 0) + (2 if spec.gate else 0) + 1
    f_peak = FP32_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6 / 1e12
    s_peak = EX2_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6 / 1e12
    fp32_t, sfu_t = elems * fp32 / f_peak / 1e12, elems * sfu / s_peak / 1e12
    pipe, per, peak = (("fp32", fp32, f_peak) if fp32_t >= sfu_t else ("sfu", sfu, s_peak))
    ach = elems * per / t_b / 1e12
    bwd_roof = {"bound": "alu", "unit": "T %s op/s" % pipe.upper(), "achieved": ach,
                "peak": peak, "frac": ach / peak, "traffic": None, "pipe": pipe,
                "ops_per_element": per,
                "floors_us": {"fp32": fp32_t * 1e6, "sfu": sfu_t * 1e6},
                "kernel": "scan_bwd_kernel (+ reverse-carry pass and reduction), one "
                          "ssm_selective_scan_bwd call"}
    return {"timed_calls": n, "input_sets": nsets, "dout": "N(0,1)",
            "fwd_ckpt": {"us_per_call": t_f * 1e6, "value": elems / t_f, "unit": "elems/s",
                         "kernels_per_call": plan["kernels"]},
            "bwd": {"us_per_call": t_b * 1e6, "value": elems / t_b, "unit": "elems/s",
                    "kernels_per_call": (2 if plan["nchunks"] > 1 else 1) + 1,
                    "workspace_bytes": nb, "roofline": bwd_roof},
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
    res = {"us_per_call": sec * 1e6, "value": spec.elements / sec, "unit": "elems/s",
           "timed_calls": n, "input_sets": nsets, "kernels_per_call": plan["kernels"],
           "roofline": dict({"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                             "frac": gbs / peak, "traffic": None, "peak_kind": kind,
                             "algorithmic_bytes_per_call": alg}, **nominal(gbs))}
    res["train"] = _bench_bcd_train(args, spec, sets, nsets, dev, stream, n)
    return res


def _bench_bcd_train(args, spec, sets, nsets, dev, stream, n):
    """Training with per-channel B, C: the checkpointing forward and the
    backward (dout ~ N(0, 1)), each timed alone over the rotating input sets;
    the backward against HBM (it moves the B, C rows in and the dB, dC rows out)."""
    import numpy as np
    import torch
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    B_, L_, D_, N_ = spec.batch, spec.L, spec.dim, spec.N
    io = libssm.SSM_BF16 if spec.io == "bf16" else libssm.SSM_F32
    F = libssm.SSM_FLAG_BC_PER_CHANNEL
    rng = np.random.default_rng(spec.seed + 900)
    for st in sets:
        st["dout"] = _upload(I.store(rng.standard_normal((B_, L_, D_)), spec.io), dev)
        st["ck"] = torch.empty((B_, (L_ + 7) // 8, D_, N_), dtype=torch.float32, device=dev)
    ws = libssm.alloc_workspace(B_, L_, D_, N_, io, dev, flags=F)
    dims = libssm.make_dims(B_, L_, D_, N_, io, None if ws is None else ws.data_ptr(),
                            0 if ws is None else ws.numel(), flags=F)
    nb = libssm.ssm_scan_bwd_workspace_bytes(B_, L_, D_, N_, io, flags=F)
    wsb = torch.empty(max(nb, 1), dtype=torch.uint8, device=dev)
    dims_b = libssm.make_dims(B_, L_, D_, N_, io, wsb.data_ptr(), nb, flags=F)
    x0 = sets[0]["x"]
    g = {"dx": torch.empty_like(x0), "ddelta": torch.empty_like(x0),
         "dz": torch.empty_like(x0) if spec.gate else None,
         "dB": torch.empty_like(sets[0]["B"]), "dC": torch.empty_like(sets[0]["C"]),
         "dA": torch.empty((D_, N_), dtype=torch.float32, device=dev),
         "dD": torch.empty(D_, dtype=torch.float32, device=dev),
         "dbias": torch.empty(D_, dtype=torch.float32, device=dev)}
    sptr = ctypes.c_void_p(stream.cuda_stream)
    sp = 1 if spec.delta_softplus else 0

    def fwd(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_selective_scan_fwd_ckpt(
            _vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
            _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, None, _vp(st["out"]), None,
            _vp(st["ck"]), ctypes.byref(dims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_fwd_ckpt (per-channel B, C)")

    def bwd(i):
        st = sets[i % nsets]
        rc = libssm.lib.ssm_selective_scan_bwd(
            _vp(st["x"]), _vp(st["delta"]), _vp(st["A"]), _vp(st["B"]), _vp(st["C"]),
            _vp(st["D"]), _vp(st["z"]), _vp(st["delta_bias"]), sp, _vp(st["ck"]),
            _vp(st["dout"]), None, _vp(g["dx"]), _vp(g["ddelta"]), _vp(g["dA"]), _vp(g["dB"]),
            _vp(g["dC"]), _vp(g["dD"]), _vp(g["dz"]), _vp(g["dbias"]), None,
            ctypes.byref(dims_b), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_selective_scan_bwd (per-channel B, C)")

    def timed(fn):
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

    for i in range(nsets):     # every set's checkpoints, before the backward reads them
        fwd(i)
    t_fwd = timed(fwd)
    t_bwd = timed(bwd)
    peak, kind = measured_peaks()
    alg = I.algorithmic_bytes_scan_bcd_bwd(spec)
    gbs = alg / t_bwd / 1e9
    plan = libssm.ssm_scan_plan(B_, L_, D_, N_, io, flags=F)
    return {"timed_calls": n, "dout": "N(0,1)",
            "fwd_ckpt": {"us_per_call": t_fwd * 1e6, "value": spec.elements / t_fwd,
                         "unit": "elems/s", "kernels_per_call": plan["kernels"]},
            "bwd": {"us_per_call": t_bwd * 1e6, "value": spec.elements / t_bwd, "unit": "elems/s",
                    "kernels_per_call": 3 if plan["nchunks"] > 1 else 2,
                    "workspace_bytes": nb,
                    "roofline": dict({"bound": "hbm", "achieved": gbs, "peak": peak,
                                      "unit": "GB/s", "frac": gbs / peak, "traffic": None,
                                      "peak_kind": kind, "algorithmic_bytes_per_call": alg,
                                      "kernel": "bcd_grad_kernel (+ reverse-carry pass and "
                                                "reduction), one ssm_selective_scan_bwd call"},
                                     **nominal(gbs))}}


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
    # the exact hold needs the N exponentials of exp(dt A) (its input term
    # reuses them), softplus's two and the gate's two: the SFU binds
    per_elem = spec.N + (2 if spec.delta_softplus else 0) + (2 if spec.gate else 0)
    peak = EX2_PER_SM_CLK * SMS * SM_MAX_MHZ * 1e6 / 1e12
    achieved = spec.elements * per_elem / sec / 1e12
    roof = {"bound": "alu", "unit": "T SFU op/s", "achieved": achieved, "peak": peak,
            "frac": achieved / peak, "traffic": None, "ops_per_element": per_elem, "pipe": "sfu",
            "kernel": "scan_kernel with the ZOH flag, one ssm_selective_scan_fwd call (%d "
                      "launches)" % plan["kernels"],
            "peak_basis": "measured ex2 rate %.1f per SM per clock x %d SMs x %.0f MHz"
                          % (EX2_PER_SM_CLK, SMS, SM_MAX_MHZ)}
    return {"us_per_call": sec * 1e6, "value": spec.elements / sec, "unit": "elems/s",
            "timed_calls": n, "input_sets": nsets, "kernels_per_call": plan["kernels"],
            "roofline": roof, "algorithmic_bytes_per_call": alg}


SSD_WORKLOAD = "ssd_bf16_b16_L8192_h8_p64_n128"


def ssd_flops_per_chunk_head(Q=128, P=64, N=128):
    """Tensor-core FLOPs the chunked SSD form needs per (chunk, head): C B^T
    (2 Q Q N), the masked product with X (2 Q Q P), the carried state read by
    C (2 Q N P) and the chunk state (2 Q N P), one bf16 product each."""
    return 2 * Q * Q * N + 2 * Q * Q * P + 2 * 2 * Q * N * P


def bench_ssd(args, dev, stream):
    """Mamba-2's SSD layer (tensor cores) on its workload: time per call, the
    tensor-pipe roofline (the FLOPs of the chunked form against the measured
    bf16 peak), the HBM roofline beside it, and parity on sampled (batch row,
    head) pairs against the oracle."""
    import numpy as np
    import torch
    import oracle
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm

    spec = I.SSD_WORKLOADS[SSD_WORKLOAD]
    inp = I.make_ssd_inputs(spec)
    t = {k: _upload(v, dev) for k, v in inp.items()}
    alg = I.algorithmic_bytes_ssd(spec)
    nsets = max(2, min(8, math.ceil(2 * L2_BYTES / alg) + 1))
    xs = [t["x"]] + [t["x"].clone() for _ in range(nsets - 1)]
    ys = [torch.empty_like(t["x"]) for _ in range(nsets)]
    fs = torch.empty((spec.batch, spec.H, spec.P, spec.N), dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    dims = libssm.make_ssd_dims(spec.batch, spec.L, spec.H, spec.P, spec.G, spec.N,
                                ws.data_ptr(), 256)
    sptr = ctypes.c_void_p(stream.cuda_stream)

    def call(i):
        rc = libssm.lib.ssm_ssd_fwd(
            _vp(xs[i % nsets]), _vp(t["dt"]), _vp(t["A"]), _vp(t["B"]), _vp(t["C"]), _vp(t["D"]),
            _vp(t["dt_bias"]), 1, None, _vp(ys[i % nsets]), _vp(fs), ctypes.byref(dims), sptr)
        if rc != 0:
            raise libssm.SSMError(rc, "ssm_ssd_fwd")

    for i in range(max(args.warmup, 3)):
        call(i)
    torch.cuda.synchronize()
    n = max(10, min(args.steps, 200))
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(n):
        call(i)
    e1.record(stream)
    torch.cuda.synchronize()
    sec = e0.elapsed_time(e1) / 1e3 / n
    st = libssm.ssm_ssd_get_device_status(spec.batch, spec.L, spec.H, spec.G, ws)
    if st != 0:
        raise libssm.SSMError(st, "ssd device status")
    chunks = (spec.L + 127) // 128
    flops = ssd_flops_per_chunk_head() * chunks * spec.H * spec.batch
    tf = flops / sec / 1e12
    peak_tf = measured_bf16_tflops()
    peak, kind = measured_peaks()
    gbs = alg / sec / 1e9
    # parity on a few (batch row, head) pairs of the last timed call
    y_last = ys[(n - 1) % nsets]
    bsel, hsel = np.array([0, spec.batch - 1]), np.array([0, spec.H - 1])
    sub = {k: (v if v is None or k in ("A", "D", "dt_bias") else v[bsel]) for k, v in inp.items()}
    ry, rfs = oracle.ssd(I.widen(sub["x"][:, :, hsel]), I.widen(sub["dt"][:, :, hsel]),
                         sub["A"][hsel], I.widen(sub["B"]), I.widen(sub["C"]), D=sub["D"][hsel],
                         dt_bias=sub["dt_bias"][hsel], dt_softplus=True)
    bt, ht = torch.as_tensor(bsel, device=dev), torch.as_tensor(hsel, device=dev)
    got = y_last[bt][:, :, ht].float().cpu().numpy().astype(np.float64)
    gfs = fs[bt][:, ht].cpu().numpy().astype(np.float64)
    return {"workload": SSD_WORKLOAD, "us_per_call": sec * 1e6,
            "value": spec.elements / sec, "unit": "elems/s (batch * L * heads * head_dim)",
            "timed_calls": n, "input_sets": nsets, "kernels_per_call": 1,
            "roofline": {"bound": "tensor", "achieved": tf, "peak": peak_tf, "unit": "TFLOP/s",
                         "frac": tf / peak_tf, "traffic": None,
                         "flops_per_call": flops,
                         "peak_kind": "measured bf16 dense (burst)",
                         "kernel": "ssd_kernel (tcgen05.mma, one launch)"},
            "hbm_roofline": dict({"bound": "hbm", "achieved": gbs, "peak": peak, "unit": "GB/s",
                                  "frac": gbs / peak, "traffic": None, "peak_kind": kind,
                                  "algorithmic_bytes_per_call": alg}, **nominal(gbs)),
            "check": dict(output_check(got, ry),
                          final_state_max_scaled_err=float(
                              np.max(np.abs(gfs - rfs) / (1 + np.abs(rfs)))),
                          against="the float64 oracle on batch rows %s, heads %s"
                                  % (bsel.tolist(), hsel.tolist()))}


def measured_bf16_tflops():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["bf16_tflops"])
    except Exception:
        return 1800.0


# ---------------------------------------------------------------------------
# the CPU oracle arm
# ---------------------------------------------------------------------------
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
    ap.add_argument("--no-ssd", action="store_true",
                    help="skip the Mamba-2 SSD layer timing")
    ap.add_argument("--no-side", action="store_true",
                    help="skip the other scan workloads (side legs)")
    ap.add_argument("--cpu-seconds", type=float, default=30.0,
                    help="oracle time budget of the headline's check and cpu_baseline "
                         "(the side legs get a quarter each)")
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
                "config": res["config"], "gbps": res["gbps"],
                "roofline": res["roofline"], "hbm_roofline": res["hbm_roofline"],
                "floors_us": res["floors_us"], "e2e": res["e2e"],
                "gpu_launches": res["gpu_launches"], "clocks": res["clocks"],
                "plan": res["plan"], "check": res.get("check"),
                "cpu_baseline": res.get("cpu_baseline")}
        for leg in ("side", "decode", "input_stage", "train", "bc_per_channel", "zoh", "ssd"):
            if leg in res:
                line[leg] = res[leg]
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
