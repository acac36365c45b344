"""GPU parity of training through the scan: the checkpointing forward
(ssm_selective_scan_fwd_ckpt) and the gradients (ssm_selective_scan_bwd)
against the float64 oracle ("State-space models (Mamba, S4)", "Training vs
Inference Modes"; "State Space Models -- Mamba, S4, and Beyond", "Verification
Checklist": gradients flow through the discretization).

Covered: the saved states equal the oracle's state after each 8-token prefix
(with and without L-chunks, from h0); every gradient (dx, ddelta, dz, dB, dC,
dA, dD, ddelta_bias, dh0) against the oracle's backward over fp32 and bf16
I/O, softplus on/off, gate on/off, D and bias on/off, dLoss/dfinal_state
on/off, several L-chunk plans, ragged sequence ends and channel tiles; an empty
sequence; the benchmark-size workload; the exact zero-order hold; per-channel B
and C (checkpoints, every gradient, equal rows against the shared-row backward,
guard bands, the benchmark-size workload on sampled channels).

Tolerances.
  Per-element gradients (dx, ddelta, dz: one value per element, each a sum
  along the reverse recurrence of one channel), element by element:
    fp32 I/O: |err| <= 2e-4 * (1 + |ref|), rel L2 <= 5e-5
    bf16 I/O: |err| <= 2e-2 * (1 + |ref|), rel L2 <= 5e-3 (outputs rounded to bf16)
  (with per-channel B and C, dB and dC are per-element gradients too)
  Summed gradients (dB, dC over every channel; dA, dD, dbias, dh0 over rows
  and tokens: signed terms that cancel), against the largest entry of each
  array, at least 1, and the L2 norm, at least sqrt(size):
    fp32 I/O: max |err| <= 2e-4 * max(1, max|ref|), rel L2 <= 5e-5
    bf16 I/O: max |err| <= 2e-2 * max(1, max|ref|), rel L2 <= 1e-2
"""
import numpy as np
import pytest

import gpu_util as G
import oracle
from selective_state_space_119_b300 import inputs as I

pytestmark = pytest.mark.gpu

TOL = {"f32": (2e-4, 5e-5), "bf16": (2e-2, 1e-2), "state": (2e-4, 5e-5)}


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_119_b300 import build
    build.build(quiet=True)
    return t


def grad_parity(got, ref, kind, what):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite" % what
    mx, l2 = TOL[kind]
    # scales floored at 1 (and sqrt(size)): a gradient that is exactly zero
    # (dA with h0 = 0 and one token) is compared in absolute terms
    scale = max(float(np.abs(ref).max()), 1.0) if ref.size else 1.0
    err = np.abs(got - ref)
    worst = float(err.max()) / scale if err.size else 0.0
    nref = max(float(np.linalg.norm(ref)), float(np.sqrt(ref.size)))
    rel = float(np.linalg.norm(got - ref)) / nref if ref.size else 0.0
    assert worst <= mx, "%s: max|err|/max|ref| = %.3e > %.0e" % (what, worst, mx)
    assert rel <= l2, "%s: rel L2 %.3e > %.0e" % (what, rel, l2)


ELEM_TOL = {"f32": (2e-4, 5e-5), "bf16": (2e-2, 5e-3)}


def elem_parity(got, ref, kind, what):
    """Per-element bound |err| <= tol * (1 + |ref|) and relative L2."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite" % what
    mx, l2 = ELEM_TOL[kind]
    worst = float((np.abs(got - ref) / (1.0 + np.abs(ref))).max()) if ref.size else 0.0
    nref = max(float(np.linalg.norm(ref)), float(np.sqrt(ref.size)))
    rel = float(np.linalg.norm(got - ref)) / nref if ref.size else 0.0
    assert worst <= mx, "%s: max|err|/(1+|ref|) = %.3e > %.0e" % (what, worst, mx)
    assert rel <= l2, "%s: rel L2 %.3e > %.0e" % (what, rel, l2)


def _store(arr, io):
    return I.store(np.asarray(arr, np.float64), io)


def _case(spec, seed, with_h0=False, with_dfinal=False):
    inp = I.make_scan_inputs(spec)
    r = np.random.default_rng(seed)
    dout = _store(r.standard_normal((spec.batch, spec.L, spec.dim)), spec.io)
    h0 = (r.standard_normal((spec.batch, spec.dim, spec.N)).astype(np.float32)
          if with_h0 else None)
    dfin = (r.standard_normal((spec.batch, spec.dim, spec.N)).astype(np.float32)
            if with_dfinal else None)
    return inp, dout, h0, dfin


def _gpu_train(inp, softplus, dout, h0=None, dfinal=None, hint=0, want_dh0=False, zoh=False):
    from selective_state_space_119_b300 import libssm
    t = {k: G.dev(v) for k, v in inp.items()}
    out, fs, ck = libssm.ssm_selective_scan_fwd_ckpt(
        t["x"], t["delta"], t["A"], t["B"], t["C"], D=t.get("D"), z=t.get("z"),
        delta_bias=t.get("delta_bias"), delta_softplus=softplus, h0=G.dev(h0),
        chunk_len_hint=hint, zoh=zoh)
    g = libssm.ssm_selective_scan_bwd(
        t["x"], t["delta"], t["A"], t["B"], t["C"], ck, G.dev(dout), D=t.get("D"), z=t.get("z"),
        delta_bias=t.get("delta_bias"), delta_softplus=softplus, dfinal_state=G.dev(dfinal),
        want_dh0=want_dh0, chunk_len_hint=hint, zoh=zoh)
    return out, fs, ck, g


def _oracle_bwd(inp, softplus, dout, h0=None, dfinal=None, zoh=False):
    return oracle.selective_scan_bwd(
        I.widen(inp["x"]), I.widen(inp["delta"]), np.asarray(inp["A"], np.float64),
        I.widen(inp["B"]), I.widen(inp["C"]), I.widen(dout),
        D=None if inp.get("D") is None else np.asarray(inp["D"], np.float64),
        z=I.widen(inp.get("z")),
        delta_bias=None if inp.get("delta_bias") is None else np.asarray(inp["delta_bias"], np.float64),
        delta_softplus=softplus, h0=None if h0 is None else h0.astype(np.float64),
        dh_final=None if dfinal is None else dfinal.astype(np.float64), zoh=zoh)


def _check_grads(g, ref, io, what, z_given=True, dh0=False):
    for k in ("dx", "ddelta"):
        elem_parity(G.host64(g[k]), ref[k], io, "%s %s" % (k, what))
    for k in ("dB", "dC"):
        grad_parity(G.host64(g[k]), ref[k], io, "%s %s" % (k, what))
    if z_given:
        elem_parity(G.host64(g["dz"]), ref["dz"], io, "dz " + what)
    grad_parity(G.host64(g["dA"]), ref["dA"], "state", "dA " + what)
    if ref["dD"] is not None:
        grad_parity(G.host64(g["dD"]), ref["dD"], "state", "dD " + what)
    if ref["ddelta_bias"] is not None:
        grad_parity(G.host64(g["ddelta_bias"]), ref["ddelta_bias"], "state", "dbias " + what)
    if dh0:
        grad_parity(G.host64(g["dh0"]), ref["dh0"], "state", "dh0 " + what)


@pytest.mark.parametrize("hint", [0, 64, 96])
def test_checkpoints_are_prefix_states(torch, hint):
    spec = I.ScanSpec(2, 301, 264, io="f32", delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=61)
    inp, dout, h0, _ = _case(spec, 62, with_h0=True)
    out, fs, ck, _ = _gpu_train(inp, True, dout, h0=h0, hint=hint)
    ck = G.host64(ck)
    assert ck.shape == (2, 38, 264, 16)
    for m in (0, 1, 8, 12, 37):
        L = 8 * m
        sub = {k: (np.ascontiguousarray(v[:, :L]) if k in ("x", "delta", "z", "B", "C")
                   and v is not None else v) for k, v in inp.items()}
        _, ref = G.oracle_scan(sub, True, h0=h0.astype(np.float64)) if L > 0 else (None, h0)
        G.parity(ck[:, m], ref, "state", "checkpoint %d (hint %d)" % (m, hint))
    ry, rh = G.oracle_scan(inp, True, h0=h0.astype(np.float64))
    G.parity(G.host64(out), ry, "f32", "checkpointing forward y")
    G.parity(G.host64(fs), rh, "state", "checkpointing forward final state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 40, 64, 96])
def test_gradients_softplus_gate(torch, io, hint):
    """hint 40: the forward's chunks are 64 tokens, the backward's 40 (its chunks
    need only start on a checkpoint)."""
    spec = I.ScanSpec(2, 300, 264, io=io, delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=63)
    inp, dout, h0, dfin = _case(spec, 64, with_h0=True, with_dfinal=True)
    _, _, _, g = _gpu_train(inp, True, dout, h0=h0, dfinal=dfin, hint=hint, want_dh0=True)
    ref = _oracle_bwd(inp, True, dout, h0=h0, dfinal=dfin)
    _check_grads(g, ref, io, "(%s, hint %d)" % (io, hint), dh0=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("gate,D_kind", [(False, "none"), (True, "one"), (False, "uniform")])
def test_gradients_plain_delta(torch, io, gate, D_kind):
    spec = I.ScanSpec(1, 203, 136, io=io, gate=gate, D_kind=D_kind, seed=65)
    inp, dout, _, _ = _case(spec, 66)
    _, _, _, g = _gpu_train(inp, False, dout, hint=64)
    ref = _oracle_bwd(inp, False, dout)
    _check_grads(g, ref, io, "(%s, gate %s, D %s)" % (io, gate, D_kind), z_given=gate)
    # dD and ddelta_bias are the gradients at zero when D / bias are absent
    if D_kind == "none":
        x, gy = I.widen(inp["x"]), I.widen(dout)
        if gate:
            zz = I.widen(inp["z"])
            gy = gy * zz / (1 + np.exp(-zz))
        grad_parity(G.host64(g["dD"]), (gy * x).sum(axis=(0, 1)), "state", "dD at D = 0")
    grad_parity(G.host64(g["ddelta_bias"]), ref["ddelta"].sum(axis=(0, 1)), "state",
                "ddelta_bias = sum of ddelta")


@pytest.mark.parametrize("L", [1, 7, 8, 9, 33])
def test_gradients_short_sequences(torch, L):
    spec = I.ScanSpec(2, L, 128, io="f32", delta_kind="softplus_bias", seed=67)
    inp, dout, _, dfin = _case(spec, 68, with_dfinal=True)
    _, _, _, g = _gpu_train(inp, True, dout, dfinal=dfin, want_dh0=True)
    ref = _oracle_bwd(inp, True, dout, dfinal=dfin)
    _check_grads(g, ref, "f32", "(L %d)" % L, dh0=True)


def test_empty_sequence(torch):
    from selective_state_space_119_b300 import libssm
    t = torch
    x = t.zeros((2, 0, 16), dtype=t.float32, device="cuda")
    BC = t.zeros((2, 0, 16), dtype=t.float32, device="cuda")
    A = -t.ones((16, 16), device="cuda")
    ck = t.zeros((2, 0, 16, 16), device="cuda")
    dfin = t.randn(2, 16, 16, device="cuda")
    g = libssm.ssm_selective_scan_bwd(x, x, A, BC, BC, ck, x, dfinal_state=dfin, want_dh0=True)
    assert float(g["dA"].abs().max()) == 0.0 and float(g["dD"].abs().max()) == 0.0
    assert t.equal(g["dh0"], dfin)


def test_benchmark_workload_gradients(torch):
    """Batch 4, L 2048, dim 1536, bf16, softplus(delta + bias), gate: every
    gradient against the oracle's full backward."""
    spec = I.WORKLOADS["scan_bf16_b4_L2048_d1536_softplus"]
    inp, dout, _, _ = _case(spec, 69)
    _, _, _, g = _gpu_train(inp, True, dout)
    ref = _oracle_bwd(inp, True, dout)
    _check_grads(g, ref, "bf16", "(benchmark workload)")


def _guarded(torch, shape, dtype, fill, pad=4096):
    n = 1
    for s in shape:
        n *= s
    big = torch.full((pad + n + pad,), fill, dtype=dtype, device="cuda")
    return big, big[pad:pad + n].view(*shape), pad, n


def test_gradients_guard_bands_and_bitwise_repeat(torch):
    """Every gradient written into the middle of a pattern-filled buffer: the
    bands before and after stay untouched (no write out of bounds, ragged
    sequence end and channel tile), and a second call gives bit-identical
    gradients (the sums are added in a fixed order)."""
    import ctypes
    from selective_state_space_119_b300 import libssm
    t = torch
    spec = I.ScanSpec(2, 203, 136, io="bf16", delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=75)
    inp, dout, h0, dfin = _case(spec, 76, with_h0=True, with_dfinal=True)
    d = {k: G.dev(v) for k, v in inp.items()}
    _, _, ck = libssm.ssm_selective_scan_fwd_ckpt(
        d["x"], d["delta"], d["A"], d["B"], d["C"], D=d["D"], z=d["z"],
        delta_bias=d["delta_bias"], delta_softplus=True, h0=G.dev(h0), chunk_len_hint=64)
    b, L, D, N = 2, 203, 136, 16
    io = t.bfloat16
    # keep every uploaded input referenced until the kernels have run (a freed
    # temporary would be handed to the next upload by the caching allocator)
    dout_t, dfin_t = G.dev(dout), G.dev(dfin)

    def run():
        outs = {"dx": _guarded(t, (b, L, D), io, 3.0), "ddelta": _guarded(t, (b, L, D), io, 3.0),
                "dz": _guarded(t, (b, L, D), io, 3.0), "dB": _guarded(t, (b, L, N), io, 3.0),
                "dC": _guarded(t, (b, L, N), io, 3.0),
                "dA": _guarded(t, (D, N), t.float32, -5.0), "dD": _guarded(t, (D,), t.float32, -5.0),
                "dbias": _guarded(t, (D,), t.float32, -5.0),
                "dh0": _guarded(t, (b, D, N), t.float32, -5.0)}
        nb = libssm.ssm_scan_bwd_workspace_bytes(b, L, D, N, "bf16", chunk_len_hint=64)
        ws = t.full((nb,), 0x5A, dtype=t.uint8, device="cuda")     # no initial contents needed
        dims = libssm.make_dims(b, L, D, N, "bf16", ws.data_ptr(), nb, chunk_len_hint=64)
        p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
        rc = libssm.lib.ssm_selective_scan_bwd(
            p(d["x"]), p(d["delta"]), p(d["A"]), p(d["B"]), p(d["C"]), p(d["D"]), p(d["z"]),
            p(d["delta_bias"]), 1, p(ck), p(dout_t), p(dfin_t),
            p(outs["dx"][1]), p(outs["ddelta"][1]), p(outs["dA"][1]), p(outs["dB"][1]),
            p(outs["dC"][1]), p(outs["dD"][1]), p(outs["dz"][1]), p(outs["dbias"][1]),
            p(outs["dh0"][1]), ctypes.byref(dims),
            ctypes.c_void_p(t.cuda.current_stream().cuda_stream))
        assert rc == 0
        t.cuda.synchronize()
        for k, (big, view, pad, n) in outs.items():
            fill = 3.0 if big.dtype == io else -5.0
            assert t.all(big[:pad] == fill) and t.all(big[pad + n:] == fill), "guard band of " + k
        return {k: v[1].clone() for k, v in outs.items()}

    g1 = run()
    g2 = run()
    for k in g1:
        assert t.equal(g1[k], g2[k]), "not bit-identical: " + k
    ref = _oracle_bwd(inp, True, dout, h0=h0, dfinal=dfin)
    g = {"dx": g1["dx"], "ddelta": g1["ddelta"], "dz": g1["dz"], "dB": g1["dB"], "dC": g1["dC"],
         "dA": g1["dA"], "dD": g1["dD"], "ddelta_bias": g1["dbias"], "dh0": g1["dh0"]}
    _check_grads(g, ref, "bf16", "(guarded buffers)", dh0=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 64])
@pytest.mark.parametrize("softplus", [True, False])
def test_zero_order_hold_gradients(torch, io, hint, softplus):
    """Training through the scan with the exact zero-order hold: the
    checkpointing forward equals the oracle's ZOH scan, and every gradient the
    oracle's ZOH backward (the hold term's e^{dt A} in dt and dt^2 phi'(dt A) in
    A), from h0 and with dLoss/dfinal_state, on both sides of the series /
    closed-form switches of m and phi' (delta up to 0.3 with |A| up to ~5)."""
    spec = I.ScanSpec(2, 300, 136, io=io, delta_kind="softplus_bias" if softplus else "loguniform",
                      delta_lo=1e-3, delta_hi=0.3, A_kind="lognormal", D_kind="uniform", seed=67)
    inp, dout, h0, dfin = _case(spec, 68, with_h0=True, with_dfinal=True)
    out, fs, _, g = _gpu_train(inp, softplus, dout, h0=h0, dfinal=dfin, hint=hint,
                               want_dh0=True, zoh=True)
    ry, rh = oracle.selective_scan(
        I.widen(inp["x"]), I.widen(inp["delta"]), np.asarray(inp["A"], np.float64),
        I.widen(inp["B"]), I.widen(inp["C"]), D=np.asarray(inp["D"], np.float64),
        z=I.widen(inp["z"]),
        delta_bias=None if inp["delta_bias"] is None else np.asarray(inp["delta_bias"], np.float64),
        delta_softplus=softplus, h0=h0.astype(np.float64), zoh=True)
    G.parity(G.host64(out), ry, io, "ZOH checkpointing forward y")
    G.parity(G.host64(fs), rh, "state", "ZOH checkpointing forward final state")
    ref = _oracle_bwd(inp, softplus, dout, h0=h0, dfinal=dfin, zoh=True)
    _check_grads(g, ref, io, "(ZOH, %s, hint %d, softplus %s)" % (io, hint, softplus), dh0=True)


# ---------------------------------------------------------------------------
# per-channel B and C (SSM_FLAG_BC_PER_CHANNEL): B, C, dB, dC [batch, L, dim, 16]
# ---------------------------------------------------------------------------
def _bcd_case(spec, seed, with_h0=False, with_dfinal=False):
    inp, dout, h0, dfin = _case(spec, seed, with_h0, with_dfinal)
    B4, C4 = I.make_bc_per_channel(spec)
    return inp, B4, C4, dout, h0, dfin


def _gpu_train_bcd(inp, B4, C4, softplus, dout, h0=None, dfinal=None, hint=0, want_dh0=False):
    from selective_state_space_119_b300 import libssm
    t = {k: G.dev(v) for k, v in inp.items()}
    B, C = G.dev(B4), G.dev(C4)
    out, fs, ck = libssm.ssm_selective_scan_fwd_ckpt(
        t["x"], t["delta"], t["A"], B, C, D=t.get("D"), z=t.get("z"),
        delta_bias=t.get("delta_bias"), delta_softplus=softplus, h0=G.dev(h0),
        chunk_len_hint=hint)
    g = libssm.ssm_selective_scan_bwd(
        t["x"], t["delta"], t["A"], B, C, ck, G.dev(dout), D=t.get("D"), z=t.get("z"),
        delta_bias=t.get("delta_bias"), delta_softplus=softplus, dfinal_state=G.dev(dfinal),
        want_dh0=want_dh0, chunk_len_hint=hint)
    return out, fs, ck, g


def _oracle_bcd(inp, B4, C4, softplus, dout=None, h0=None, dfinal=None, dsel=None):
    """The oracle's per-channel scan (dout None) or backward, on the channels
    dsel (all when None): channels are independent with per-channel rows."""
    sel = (lambda a: a) if dsel is None else (lambda a: np.ascontiguousarray(a[:, :, dsel]))
    vec = (lambda a: a) if dsel is None else (lambda a: np.ascontiguousarray(a[dsel]))
    st = (lambda a: a) if dsel is None else (lambda a: np.ascontiguousarray(a[:, dsel]))
    kw = dict(D=None if inp.get("D") is None else vec(np.asarray(inp["D"], np.float64)),
              z=None if inp.get("z") is None else sel(I.widen(inp["z"])),
              delta_bias=(None if inp.get("delta_bias") is None
                          else vec(np.asarray(inp["delta_bias"], np.float64))),
              delta_softplus=softplus, h0=None if h0 is None else st(h0.astype(np.float64)))
    args = (sel(I.widen(inp["x"])), sel(I.widen(inp["delta"])),
            vec(np.asarray(inp["A"], np.float64)), sel(I.widen(B4)), sel(I.widen(C4)))
    if dout is None:
        return oracle.selective_scan_bcd(*args, **kw)
    return oracle.selective_scan_bcd_bwd(
        *args, sel(I.widen(dout)), dh_final=None if dfinal is None else st(dfinal.astype(np.float64)),
        **kw)


def _check_bcd_grads(g, ref, io, what, z_given=True, dh0=False, dsel=None):
    """dx, ddelta, dz, dB, dC are per element here (nothing sums over
    channels): the per-element bound. dA, dD, dbias, dh0 sum over rows and
    tokens: the array-scaled bound."""
    sel = (lambda a: a) if dsel is None else (lambda a: a[:, :, dsel])
    vec = (lambda a: a) if dsel is None else (lambda a: a[dsel])
    st = (lambda a: a) if dsel is None else (lambda a: a[:, dsel])
    for k in ("dx", "ddelta", "dB", "dC") + (("dz",) if z_given else ()):
        elem_parity(sel(G.host64(g[k])), ref[k], io, "%s %s" % (k, what))
    grad_parity(vec(G.host64(g["dA"])), ref["dA"], "state", "dA " + what)
    if ref["dD"] is not None:
        grad_parity(vec(G.host64(g["dD"])), ref["dD"], "state", "dD " + what)
    if ref["ddelta_bias"] is not None:
        grad_parity(vec(G.host64(g["ddelta_bias"])), ref["ddelta_bias"], "state", "dbias " + what)
    if dh0:
        grad_parity(st(G.host64(g["dh0"])), ref["dh0"], "state", "dh0 " + what)


@pytest.mark.parametrize("hint", [0, 64])
def test_bcd_checkpoints_are_prefix_states(torch, hint):
    spec = I.ScanSpec(2, 203, 136, io="f32", delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=91)
    inp, B4, C4, dout, h0, _ = _bcd_case(spec, 92, with_h0=True)
    out, fs, ck, _ = _gpu_train_bcd(inp, B4, C4, True, dout, h0=h0, hint=hint)
    ck = G.host64(ck)
    assert ck.shape == (2, 26, 136, 16)
    for m in (0, 1, 8, 17, 25):
        L = 8 * m
        if L == 0:
            G.parity(ck[:, 0], h0.astype(np.float64), "state", "checkpoint 0 = h0")
            continue
        sub = {k: (np.ascontiguousarray(v[:, :L]) if k in ("x", "delta", "z") and v is not None
                   else v) for k, v in inp.items()}
        _, ref = _oracle_bcd(sub, B4[:, :L], C4[:, :L], True, h0=h0)
        G.parity(ck[:, m], ref, "state", "per-channel checkpoint %d (hint %d)" % (m, hint))
    ry, rh = _oracle_bcd(inp, B4, C4, True, h0=h0)
    G.parity(G.host64(out), ry, "f32", "per-channel checkpointing forward y")
    G.parity(G.host64(fs), rh, "state", "per-channel checkpointing forward final state")


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 64, 96])
def test_bcd_gradients_softplus_gate(torch, io, hint):
    spec = I.ScanSpec(2, 300, 264, io=io, delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=93)
    inp, B4, C4, dout, h0, dfin = _bcd_case(spec, 94, with_h0=True, with_dfinal=True)
    _, _, _, g = _gpu_train_bcd(inp, B4, C4, True, dout, h0=h0, dfinal=dfin, hint=hint,
                                want_dh0=True)
    ref = _oracle_bcd(inp, B4, C4, True, dout, h0=h0, dfinal=dfin)
    _check_bcd_grads(g, ref, io, "(per-channel, %s, hint %d)" % (io, hint), dh0=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("gate,D_kind", [(False, "none"), (True, "one")])
def test_bcd_gradients_plain_delta(torch, io, gate, D_kind):
    spec = I.ScanSpec(1, 203, 136, io=io, gate=gate, D_kind=D_kind, seed=95)
    inp, B4, C4, dout, _, _ = _bcd_case(spec, 96)
    _, _, _, g = _gpu_train_bcd(inp, B4, C4, False, dout, hint=64)
    ref = _oracle_bcd(inp, B4, C4, False, dout)
    _check_bcd_grads(g, ref, io, "(per-channel, %s, gate %s, D %s)" % (io, gate, D_kind),
                     z_given=gate)
    grad_parity(G.host64(g["ddelta_bias"]), ref["ddelta"].sum(axis=(0, 1)), "state",
                "per-channel ddelta_bias = sum of ddelta")


@pytest.mark.parametrize("io,L,dim", [("f32", 1, 128), ("f32", 7, 128), ("f32", 8, 128),
                                       ("f32", 9, 132), ("f32", 33, 132), ("bf16", 1, 136),
                                       ("bf16", 7, 136), ("bf16", 9, 136), ("bf16", 33, 256)])
def test_bcd_gradients_short_sequences(torch, io, L, dim):
    """dim 132 (fp32) ends half-way through a warp's 8 channels; bf16 runs the
    staged gradient pass, whose blocks here hold fewer than 8 tokens and whose
    last channel tile (dim 136) holds 8 channels."""
    spec = I.ScanSpec(2, L, dim, io=io, delta_kind="softplus_bias", seed=97)
    inp, B4, C4, dout, _, dfin = _bcd_case(spec, 98, with_dfinal=True)
    _, _, _, g = _gpu_train_bcd(inp, B4, C4, True, dout, dfinal=dfin, want_dh0=True)
    ref = _oracle_bcd(inp, B4, C4, True, dout, dfinal=dfin)
    _check_bcd_grads(g, ref, io, "(per-channel, %s, L %d, dim %d)" % (io, L, dim), dh0=True)


def test_bcd_equal_rows_give_the_shared_gradients(torch):
    """Rows equal across channels: the per-channel gradients dB, dC summed over
    channels are the shared-row backward's dB, dC, and every other gradient is
    the same (two GPU paths and the oracle)."""
    spec = I.ScanSpec(2, 200, 128, io="f32", delta_kind="softplus_bias", D_kind="uniform",
                      seed=99)
    inp, dout, _, dfin = _case(spec, 100, with_dfinal=True)
    B4 = np.ascontiguousarray(np.repeat(inp["B"][:, :, None, :], 128, 2))
    C4 = np.ascontiguousarray(np.repeat(inp["C"][:, :, None, :], 128, 2))
    _, _, _, g4 = _gpu_train_bcd(inp, B4, C4, True, dout, dfinal=dfin, hint=64, want_dh0=True)
    _, _, _, g = _gpu_train(inp, True, dout, dfinal=dfin, hint=64, want_dh0=True)
    for k in ("dB", "dC"):
        G.parity(G.host64(g4[k]).sum(axis=2), G.host64(g[k]), "f32", "summed per-channel " + k)
    for k in ("dx", "ddelta", "dz", "dA", "dD", "ddelta_bias", "dh0"):
        G.parity(G.host64(g4[k]), G.host64(g[k]), "f32", "per-channel vs shared " + k)
    ref = _oracle_bwd(inp, True, dout, dfinal=dfin)
    grad_parity(G.host64(g4["dB"]).sum(axis=2), ref["dB"], "f32", "summed per-channel dB")


def test_bcd_benchmark_workload_gradients(torch):
    """Batch 4, L 2048, dim 1536, bf16, softplus(delta + bias), gate, per-channel
    rows, in the planner's chunks: every gradient of 48 sampled channels
    against the oracle's backward of those channels (channels are independent
    with per-channel rows, so the sample is exact)."""
    spec = I.WORKLOADS["scan_bf16_b4_L2048_d1536_softplus"]
    inp, B4, C4, dout, _, _ = _bcd_case(spec, 101)
    _, _, _, g = _gpu_train_bcd(inp, B4, C4, True, dout)
    dsel = np.sort(np.random.default_rng(102).choice(spec.dim, 48, replace=False))
    ref = _oracle_bcd(inp, B4, C4, True, dout, dsel=dsel)
    _check_bcd_grads(g, ref, "bf16", "(per-channel benchmark workload)", dsel=dsel)


def test_bcd_gradients_guard_bands_and_bitwise_repeat(torch):
    """Per-channel gradients written into the middle of pattern-filled buffers:
    the bands stay untouched (ragged sequence end and channel tile) and a second
    call gives bit-identical gradients."""
    from selective_state_space_119_b300 import libssm
    t = torch
    spec = I.ScanSpec(2, 203, 136, io="bf16", delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=103)
    inp, B4, C4, dout, h0, dfin = _bcd_case(spec, 104, with_h0=True, with_dfinal=True)
    d = {k: G.dev(v) for k, v in inp.items()}
    B, C = G.dev(B4), G.dev(C4)
    _, _, ck = libssm.ssm_selective_scan_fwd_ckpt(
        d["x"], d["delta"], d["A"], B, C, D=d["D"], z=d["z"], delta_bias=d["delta_bias"],
        delta_softplus=True, h0=G.dev(h0), chunk_len_hint=64)
    b, L, D, N = 2, 203, 136, 16
    io = t.bfloat16
    dout_t, dfin_t = G.dev(dout), G.dev(dfin)

    def run():
        bufs = {"dx": _guarded(t, (b, L, D), io, 3.0), "ddelta": _guarded(t, (b, L, D), io, 3.0),
                "dz": _guarded(t, (b, L, D), io, 3.0), "dB": _guarded(t, (b, L, D, N), io, 3.0),
                "dC": _guarded(t, (b, L, D, N), io, 3.0),
                "dA": _guarded(t, (D, N), t.float32, -5.0),
                "dD": _guarded(t, (D,), t.float32, -5.0),
                "dbias": _guarded(t, (D,), t.float32, -5.0),
                "dh0": _guarded(t, (b, D, N), t.float32, -5.0)}
        g = {k: v[1] for k, v in bufs.items()}
        nb = libssm.ssm_scan_bwd_workspace_bytes(b, L, D, N, "bf16", chunk_len_hint=64,
                                                 flags=libssm.SSM_FLAG_BC_PER_CHANNEL)
        ws = t.full((nb,), 0x5A, dtype=t.uint8, device="cuda")
        dims = libssm.make_dims(b, L, D, N, "bf16", ws.data_ptr(), nb, chunk_len_hint=64,
                                flags=libssm.SSM_FLAG_BC_PER_CHANNEL)
        import ctypes
        p = lambda x: None if x is None else ctypes.c_void_p(x.data_ptr())
        rc = libssm.lib.ssm_selective_scan_bwd(
            p(d["x"]), p(d["delta"]), p(d["A"]), p(B), p(C), p(d["D"]), p(d["z"]),
            p(d["delta_bias"]), 1, p(ck), p(dout_t), p(dfin_t), p(g["dx"]), p(g["ddelta"]),
            p(g["dA"]), p(g["dB"]), p(g["dC"]), p(g["dD"]), p(g["dz"]), p(g["dbias"]),
            p(g["dh0"]), ctypes.byref(dims), ctypes.c_void_p(t.cuda.current_stream().cuda_stream))
        assert rc == 0
        t.cuda.synchronize()
        for k, (big, view, pad, n) in bufs.items():
            fill = 3.0 if big.dtype == io else -5.0
            assert t.all(big[:pad] == fill) and t.all(big[pad + n:] == fill), "guard band of " + k
        return {k: v.clone() for k, v in g.items()}

    g1 = run()
    g2 = run()
    for k in g1:
        assert t.equal(g1[k], g2[k]), "not bit-identical: " + k
    ref = _oracle_bcd(inp, B4, C4, True, dout, h0=h0, dfinal=dfin)
    g1["ddelta_bias"] = g1.pop("dbias")
    _check_bcd_grads(g1, ref, "bf16", "(per-channel, guarded buffers)", dh0=True)
