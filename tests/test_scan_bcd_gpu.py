"""GPU parity of the scan with per-channel B and C (SSM_FLAG_BC_PER_CHANNEL):
B, C of shape [batch, L, dim, N] ("Mamba: State Space Models Challenge
Transformers", "Selective Scan Algorithm", the docstring's shapes), against
the oracle (each channel the one-channel scan with its own rows).

Covered: fp32 and bf16; softplus(delta + bias) and plain delta; gate on/off;
L-chunk plans; an initial state; ragged channel tiles and sequence ends; rows
equal across channels reproduce the shared-B, C scan; the benchmark-size
workload on sampled channels."""
import numpy as np
import pytest

import gpu_util as G
import oracle
from selective_state_space_119_b300 import inputs as I

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def torch():
    t = pytest.importorskip("torch")
    if not t.cuda.is_available():
        pytest.skip("no CUDA device")
    from selective_state_space_119_b300 import build
    build.build(quiet=True)
    return t


def _gpu(inp, B4, C4, softplus, hint=0, h0=None):
    from selective_state_space_119_b300 import libssm
    return libssm.ssm_selective_scan_fwd(
        G.dev(inp["x"]), G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(B4), G.dev(C4),
        D=G.dev(inp.get("D")), z=G.dev(inp.get("z")), delta_bias=G.dev(inp.get("delta_bias")),
        delta_softplus=softplus, chunk_len_hint=hint, h0=G.dev(h0))


def _ref(inp, B4, C4, softplus, dsel=None, h0=None):
    sel = (lambda a: a) if dsel is None else (lambda a: np.ascontiguousarray(a[:, :, dsel]))
    vec = (lambda a: a) if dsel is None else (lambda a: a[dsel])
    return oracle.selective_scan_bcd(
        sel(I.widen(inp["x"])), sel(I.widen(inp["delta"])), vec(np.asarray(inp["A"], np.float64)),
        sel(I.widen(B4)), sel(I.widen(C4)),
        D=None if inp.get("D") is None else vec(np.asarray(inp["D"], np.float64)),
        z=None if inp.get("z") is None else sel(I.widen(inp["z"])),
        delta_bias=None if inp.get("delta_bias") is None else vec(np.asarray(inp["delta_bias"], np.float64)),
        delta_softplus=softplus, h0=None if h0 is None else h0.astype(np.float64))


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 64])
def test_bcd_matches_oracle(torch, io, hint):
    spec = I.ScanSpec(2, 301, 264, io=io, delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=81)
    inp = I.make_scan_inputs(spec)
    B4, C4 = I.make_bc_per_channel(spec)
    out, fs = _gpu(inp, B4, C4, True, hint)
    ry, rh = _ref(inp, B4, C4, True)
    G.parity(G.host64(out), ry, io, "per-channel y (%s, hint %d)" % (io, hint))
    G.parity(G.host64(fs), rh, "state", "per-channel final state (%s, hint %d)" % (io, hint))


@pytest.mark.parametrize("gate,dim", [(True, 136), (False, 136), (True, 132)])
def test_bcd_plain_delta_and_h0(torch, gate, dim):
    """dim 132 (fp32) ends half-way through a warp's 8 channels."""
    spec = I.ScanSpec(1, 130, dim, io="f32", gate=gate, D_kind="none", seed=82)
    inp = I.make_scan_inputs(spec)
    B4, C4 = I.make_bc_per_channel(spec)
    h0 = np.random.default_rng(83).standard_normal((1, dim, 16)).astype(np.float32)
    out, fs = _gpu(inp, B4, C4, False, 32, h0=h0)
    ry, rh = _ref(inp, B4, C4, False, h0=h0)
    G.parity(G.host64(out), ry, "f32", "per-channel y from h0 (gate %s)" % gate)
    G.parity(G.host64(fs), rh, "state", "per-channel final state from h0 (gate %s)" % gate)


def test_bcd_equal_rows_give_the_shared_scan(torch):
    spec = I.ScanSpec(2, 200, 128, io="f32", seed=84)
    inp = I.make_scan_inputs(spec)
    B4 = np.ascontiguousarray(np.repeat(inp["B"][:, :, None, :], 128, 2))
    C4 = np.ascontiguousarray(np.repeat(inp["C"][:, :, None, :], 128, 2))
    out4, fs4 = _gpu(inp, B4, C4, False, 64)
    out, fs = G.gpu_scan(inp, False, chunk_len_hint=64)
    G.parity(G.host64(out4), G.host64(out), "f32", "equal rows vs shared B, C")
    G.parity(G.host64(fs4), G.host64(fs), "state", "equal rows vs shared B, C: state")


def test_bcd_benchmark_size_sampled(torch):
    """Batch 4, L 2048, dim 1536, bf16, softplus(delta + bias), gate, with
    per-channel B, C: sampled channels against the oracle."""
    spec = I.WORKLOADS["scan_bf16_b4_L2048_d1536_softplus"]
    inp = I.make_scan_inputs(spec)
    B4, C4 = I.make_bc_per_channel(spec)
    out, fs = _gpu(inp, B4, C4, True)
    dsel = np.array([0, 1, 127, 128, 999, 1535])
    ry, rh = _ref(inp, B4, C4, True, dsel=dsel)
    G.parity(G.host64(out)[:, :, dsel], ry, "bf16", "per-channel y, benchmark size")
    G.parity(G.host64(fs)[:, dsel], rh, "state", "per-channel final state, benchmark size")


def test_bcd_guard_bands_and_bitwise_repeat(torch):
    from selective_state_space_119_b300 import libssm
    t = torch
    spec = I.ScanSpec(2, 203, 136, io="bf16", seed=85)
    inp = I.make_scan_inputs(spec)
    B4, C4 = I.make_bc_per_channel(spec)
    n, nf, pad = 2 * 203 * 136, 2 * 136 * 16, 4096
    big = t.full((pad + n + pad,), 9.0, dtype=t.bfloat16, device="cuda")
    fbig = t.full((pad + nf + pad,), -9.0, dtype=t.float32, device="cuda")
    out = big[pad:pad + n].view(2, 203, 136)
    fs = fbig[pad:pad + nf].view(2, 136, 16)
    args = (G.dev(inp["x"]), G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(B4), G.dev(C4))
    libssm.ssm_selective_scan_fwd(*args, D=G.dev(inp["D"]), z=G.dev(inp["z"]), out=out,
                                  final_state=fs, chunk_len_hint=64)
    t.cuda.synchronize()
    assert t.all(big[:pad] == 9.0) and t.all(big[pad + n:] == 9.0)
    assert t.all(fbig[:pad] == -9.0) and t.all(fbig[pad + nf:] == -9.0)
    o2, f2 = libssm.ssm_selective_scan_fwd(*args, D=G.dev(inp["D"]), z=G.dev(inp["z"]),
                                           chunk_len_hint=64)
    assert t.equal(out, o2) and t.equal(fs, f2)
    ry, rh = _ref(inp, B4, C4, False)
    G.parity(G.host64(out), ry, "bf16", "per-channel y in guarded buffer")
