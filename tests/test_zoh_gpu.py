"""GPU parity of the exact zero-order-hold discretization (SSM_FLAG_ZOH):
Bbar = A^-1 (e^{A dt} - 1) B instead of dt B ("State-space models (Mamba, S4)",
"From Continuous to Discrete: The Key Step"), for the scan and the decode step,
against the oracle's ZOH scan (pinned to the continuous solution and to ODE
integration on the CPU).

Covered: fp32 and bf16 I/O; softplus(delta + bias) and plain delta; L-chunk
plans (the chunk-state pass uses the same Bbar); steps whose dt*A falls on
both sides of the kernel's series / (e^z - 1)/A switch at |dt A| = 0.1; the
flag really changes the result; the decode step for several dstate."""
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


def _gpu(inp, softplus, hint=0, zoh=True):
    from selective_state_space_119_b300 import libssm
    return libssm.ssm_selective_scan_fwd(
        G.dev(inp["x"]), G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(inp["B"]), G.dev(inp["C"]),
        D=G.dev(inp.get("D")), z=G.dev(inp.get("z")), delta_bias=G.dev(inp.get("delta_bias")),
        delta_softplus=softplus, chunk_len_hint=hint, zoh=zoh)


def _ref(inp, softplus):
    return oracle.selective_scan(
        I.widen(inp["x"]), I.widen(inp["delta"]), np.asarray(inp["A"], np.float64),
        I.widen(inp["B"]), I.widen(inp["C"]),
        D=None if inp.get("D") is None else np.asarray(inp["D"], np.float64),
        z=I.widen(inp.get("z")),
        delta_bias=None if inp.get("delta_bias") is None else np.asarray(inp["delta_bias"], np.float64),
        delta_softplus=softplus, zoh=True)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("hint", [0, 64])
def test_zoh_scan_matches_oracle(torch, io, hint):
    # log-uniform dt in [1e-3, 1e-1] with A = -(n+1): dt*A from -1e-3 to -1.6
    spec = I.ScanSpec(2, 300, 264, io=io, seed=71)
    inp = I.make_scan_inputs(spec)
    out, fs = _gpu(inp, False, hint)
    ry, rh = _ref(inp, False)
    G.parity(G.host64(out), ry, io, "ZOH y (%s, hint %d)" % (io, hint))
    G.parity(G.host64(fs), rh, "state", "ZOH final state (%s, hint %d)" % (io, hint))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_zoh_scan_softplus(torch, io):
    spec = I.ScanSpec(3, 200, 136, io=io, delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=72)
    inp = I.make_scan_inputs(spec)
    out, fs = _gpu(inp, True, 96)
    ry, rh = _ref(inp, True)
    G.parity(G.host64(out), ry, io, "ZOH y softplus")
    G.parity(G.host64(fs), rh, "state", "ZOH final state softplus")


def test_zoh_benchmark_size_sampled(torch):
    """Batch 4, L 2048, dim 1536, bf16, softplus(delta + bias), gate, with the
    exact zero-order hold and the library's plan (6 chunks): sampled channels,
    every token, against the oracle."""
    spec = I.WORKLOADS["scan_bf16_b4_L2048_d1536_softplus"]
    inp = I.make_scan_inputs(spec)
    out, fs = _gpu(inp, True)
    dsel = np.array([0, 1, 127, 128, 999, 1535])
    sub = dict(inp)
    for k in ("x", "delta", "z"):
        if inp.get(k) is not None:
            sub[k] = inp[k][:, :, dsel]
    for k in ("A", "D", "delta_bias"):
        if inp.get(k) is not None:
            sub[k] = np.asarray(inp[k])[dsel]
    ry, rh = _ref(sub, True)
    G.parity(G.host64(out)[:, :, dsel], ry, "bf16", "ZOH y, benchmark size")
    G.parity(G.host64(fs)[:, dsel], rh, "state", "ZOH final state, benchmark size")


def test_zoh_changes_the_result(torch):
    spec = I.ScanSpec(1, 128, 128, io="f32", delta_lo=0.05, delta_hi=0.5, seed=73)
    inp = I.make_scan_inputs(spec)
    out_z, _ = _gpu(inp, False)
    out_1, _ = _gpu(inp, False, zoh=False)
    diff = np.abs(G.host64(out_z) - G.host64(out_1)).max()
    assert diff > 1e-2, diff


@pytest.mark.parametrize("N", [4, 16])
def test_zoh_decode_matches_oracle(torch, N):
    from selective_state_space_119_b300 import libssm
    dspec = I.DecodeSpec(8, 256, N=N, steps=3, io="f32", delta_lo=1e-3, delta_hi=0.5, seed=74)
    d = I.make_decode_inputs(dspec)
    state = G.dev(d["state0"]).clone()
    ref_state = d["state0"].astype(np.float64)
    for t in range(3):
        y = libssm.ssm_state_update(state, G.dev(d["x"][t]), G.dev(d["delta"][t]), G.dev(d["A"]),
                                    G.dev(d["B"][t]), G.dev(d["C"][t]), D=G.dev(d["D"]),
                                    z=G.dev(d["z"][t]), zoh=True)
        ry, ref_state = oracle.state_update(ref_state, d["x"][t], d["delta"][t], d["A"],
                                            d["B"][t], d["C"][t], D=d["D"], z=d["z"][t], zoh=True)
        G.parity(G.host64(y), ry, "f32", "ZOH decode y step %d" % t)
        G.parity(G.host64(state), ref_state, "state", "ZOH decode state step %d" % t)
