"""Run one kernel case a few times, for profilers (ncu) and quick timings.

    python -m selective_state_space_119_b300.profile_case scan --batch 1 --seqlen 16384 \\
        --dim 5120 [--A s4d|lognormal] [--softplus] [--chunk-len 0] [--calls 3]
    python -m selective_state_space_119_b300.profile_case ssd --batch 16 --seqlen 1024 \\
        [--heads 8] [--groups 1] [--calls 3]
    python -m selective_state_space_119_b300.profile_case bcd_train --batch 4 --seqlen 2048 \\
        --dim 1536 [--chunk-len 0] [--calls 3]
    python -m selective_state_space_119_b300.profile_case conv --batch 4 --seqlen 2048 \\
        --dim 1536 [--calls 3]
    python -m selective_state_space_119_b300.profile_case train --batch 4 --seqlen 2048 \\
        --dim 1536 [--A s4d|lognormal] [--calls 3]
    python -m selective_state_space_119_b300.profile_case decode --batch 256 --seqlen 1 \\
        --dim 5120 [--calls 3]

The inputs are the seeded workload distributions of ``inputs`` (the scan's
long-sequence recipe by default: delta log-uniform in [1e-4, 1e-2], gate, D = 1,
final state). Every call goes through the C ABI; the script prints the plan and
the CUDA-event time of the last call and exits non-zero on any library error.
"""
from __future__ import annotations

import argparse
import ctypes
import sys

import numpy as np


def _dev(torch, a):
    if a is None:
        return None
    if a.dtype == np.uint16:
        return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda().view(torch.bfloat16)
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def run_scan(args, torch):
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    if args.softplus:
        spec = I.ScanSpec(args.batch, args.seqlen, args.dim, io="bf16",
                          delta_kind="softplus_bias", A_kind=args.A, D_kind="uniform", seed=3)
    else:
        spec = I.ScanSpec(args.batch, args.seqlen, args.dim, io="bf16", delta_lo=1e-4,
                          delta_hi=1e-2, A_kind=args.A, seed=3)
    t = {k: _dev(torch, v) for k, v in I.make_scan_inputs(spec).items()}
    plan = libssm.ssm_scan_plan(spec.batch, spec.L, spec.dim, 16, "bf16",
                                chunk_len_hint=args.chunk_len)
    print("plan", plan, flush=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.calls):
        e0.record()
        libssm.ssm_selective_scan_fwd(t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"],
                                      z=t["z"], delta_bias=t["delta_bias"],
                                      delta_softplus=spec.delta_softplus,
                                      chunk_len_hint=args.chunk_len)
        e1.record()
    torch.cuda.synchronize()
    print("last call %.3f ms" % e0.elapsed_time(e1), flush=True)


def run_ssd(args, torch):
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    spec = I.SsdSpec(args.batch, args.seqlen, H=args.heads, G=args.groups, seed=5)
    t = {k: _dev(torch, v) for k, v in I.make_ssd_inputs(spec).items()}
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.calls):
        e0.record()
        libssm.ssm_ssd_fwd(t["x"], t["dt"], t["A"], t["B"], t["C"], D=t["D"],
                           dt_bias=t["dt_bias"], dt_softplus=True)
        e1.record()
    torch.cuda.synchronize()
    print("last call %.3f ms" % e0.elapsed_time(e1), flush=True)


def run_bcd_train(args, torch):
    """Training with per-channel B, C on the softplus recipe: each call is one
    plain forward, one checkpointing forward and one backward (dout ~ N(0, 1))."""
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(args.batch, args.seqlen, args.dim, io="bf16", delta_kind="softplus_bias",
                      A_kind=args.A, D_kind="uniform", seed=3)
    t = {k: _dev(torch, v) for k, v in I.make_scan_inputs(spec).items()}
    B4, C4 = (_dev(torch, v) for v in I.make_bc_per_channel(spec))
    rng = np.random.default_rng(4)
    dout = _dev(torch, I.store(rng.standard_normal((spec.batch, spec.L, spec.dim)), "bf16"))
    plan = libssm.ssm_scan_plan(spec.batch, spec.L, spec.dim, 16, "bf16",
                                chunk_len_hint=args.chunk_len,
                                flags=libssm.SSM_FLAG_BC_PER_CHANNEL)
    print("plan", plan, flush=True)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    kw = dict(D=t["D"], z=t["z"], delta_bias=t["delta_bias"], delta_softplus=True,
              chunk_len_hint=args.chunk_len)
    for i in range(args.calls):
        ev[0].record()
        libssm.ssm_selective_scan_fwd(t["x"], t["delta"], t["A"], B4, C4, **kw)
        ev[1].record()
        _, _, ck = libssm.ssm_selective_scan_fwd_ckpt(t["x"], t["delta"], t["A"], B4, C4, **kw)
        ev[2].record()
        libssm.ssm_selective_scan_bwd(t["x"], t["delta"], t["A"], B4, C4, ck, dout, **kw)
        ev[3].record()
    torch.cuda.synchronize()
    print("last call: fwd %.3f ms, fwd_ckpt %.3f ms, bwd %.3f ms (allocations included)"
          % (ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2]), ev[2].elapsed_time(ev[3])),
          flush=True)


def run_train(args, torch):
    """Training through the scan with shared B, C on the softplus recipe: each
    call is one checkpointing forward and one backward (dout ~ N(0, 1))."""
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(args.batch, args.seqlen, args.dim, io="bf16", delta_kind="softplus_bias",
                      A_kind=args.A, D_kind="uniform", seed=3)
    t = {k: _dev(torch, v) for k, v in I.make_scan_inputs(spec).items()}
    rng = np.random.default_rng(4)
    dout = _dev(torch, I.store(rng.standard_normal((spec.batch, spec.L, spec.dim)), "bf16"))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    kw = dict(D=t["D"], z=t["z"], delta_bias=t["delta_bias"], delta_softplus=True,
              chunk_len_hint=args.chunk_len)
    for i in range(args.calls):
        ev[0].record()
        _, _, ck = libssm.ssm_selective_scan_fwd_ckpt(t["x"], t["delta"], t["A"], t["B"], t["C"],
                                                      **kw)
        ev[1].record()
        libssm.ssm_selective_scan_bwd(t["x"], t["delta"], t["A"], t["B"], t["C"], ck, dout, **kw)
        ev[2].record()
    torch.cuda.synchronize()
    print("last call: fwd_ckpt %.3f ms, bwd %.3f ms (allocations included)"
          % (ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])), flush=True)


def run_decode(args, torch):
    """Decode steps on the recipe of the decode workload (state N(0, 1), one
    token set per call, --seqlen ignored); every call updates the state."""
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    spec = I.DecodeSpec(args.batch, args.dim, steps=1, seed=7)
    inp = I.make_decode_inputs(spec)
    t = {k: _dev(torch, v) for k, v in inp.items()}
    state = t["state0"].clone()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for i in range(args.calls):
        e0.record()
        libssm.ssm_state_update(state, t["x"][0], t["delta"][0], t["A"], t["B"][0], t["C"][0],
                                D=t.get("D"), z=None if t.get("z") is None else t["z"][0],
                                delta_bias=t.get("delta_bias"),
                                delta_softplus=False)
        e1.record()
    torch.cuda.synchronize()
    print("last call %.3f ms (output allocation included)" % e0.elapsed_time(e1), flush=True)


def run_conv(args, torch):
    """The input stage (causal conv1d of width 4 + SiLU) and its backward, each
    call one forward and one backward (du ~ N(0, 1)), bf16."""
    from selective_state_space_119_b300 import inputs as I
    from selective_state_space_119_b300 import libssm
    rng = np.random.default_rng(6)
    x = _dev(torch, I.store(rng.standard_normal((args.batch, args.seqlen, args.dim)), "bf16"))
    du = _dev(torch, I.store(rng.standard_normal((args.batch, args.seqlen, args.dim)), "bf16"))
    w = _dev(torch, (rng.standard_normal((args.dim, 4)) * 0.5).astype(np.float32))
    bias = _dev(torch, (rng.standard_normal(args.dim) * 0.1).astype(np.float32))
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for i in range(args.calls):
        ev[0].record()
        libssm.ssm_causal_conv1d_silu(x, w, bias)
        ev[1].record()
        libssm.ssm_causal_conv1d_silu_bwd(x, w, du, conv_b=bias)
        ev[2].record()
    torch.cuda.synchronize()
    print("last call: fwd %.3f ms, bwd %.3f ms (allocations included)"
          % (ev[0].elapsed_time(ev[1]), ev[1].elapsed_time(ev[2])), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("kernel", choices=["scan", "ssd", "bcd_train", "conv", "train", "decode"])
    ap.add_argument("--batch", type=int, required=True)
    ap.add_argument("--seqlen", type=int, required=True)
    ap.add_argument("--dim", type=int, default=5120)
    ap.add_argument("--A", default="s4d", choices=["s4d", "lognormal"])
    ap.add_argument("--softplus", action="store_true")
    ap.add_argument("--chunk-len", type=int, default=0)
    ap.add_argument("--heads", type=int, default=8)
    ap.add_argument("--groups", type=int, default=1)
    ap.add_argument("--calls", type=int, default=3)
    args = ap.parse_args(argv)
    import torch
    if not torch.cuda.is_available():
        sys.exit("no CUDA device")
    {"scan": run_scan, "ssd": run_ssd, "bcd_train": run_bcd_train,
     "conv": run_conv, "train": run_train, "decode": run_decode}[args.kernel](args, torch)


if __name__ == "__main__":
    main()
