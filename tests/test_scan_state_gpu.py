"""GPU parity of ssm_selective_scan_fwd_from_state: the scan started from a
given state h0 instead of zero ("State-space models (Mamba, S4)", "Worked
Example: 2D SSM Step" runs the recurrence from h_0 != 0; "Training vs
Inference Modes" keeps h between tokens).

Covered: the oracle started from the same h0 (y and final state), with and
without L-chunks, over every tile configuration; a sequence split in two and
continued from the first part's final state equals the oracle's unsplit scan;
seqlen 0 copies h0; a decode step continues a from-state scan; argument errors.
"""
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


def _state(batch, dim, N, seed):
    return np.random.default_rng(seed).standard_normal((batch, dim, N)).astype(np.float32)


def _scan(inp, softplus, h0, hint=0, tile=0):
    from selective_state_space_119_b300 import libssm
    return libssm.ssm_selective_scan_fwd(
        G.dev(inp["x"]), G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(inp["B"]), G.dev(inp["C"]),
        D=G.dev(inp.get("D")), z=G.dev(inp.get("z")), delta_bias=G.dev(inp.get("delta_bias")),
        delta_softplus=softplus, chunk_len_hint=hint, tile_config_hint=tile, h0=G.dev(h0))


@pytest.mark.parametrize("tile", [0, 1, 2, 3, 4])
@pytest.mark.parametrize("hint", [0, 32, 96])
def test_from_state_matches_oracle(torch, hint, tile):
    spec = I.ScanSpec(2, 300, 264, io="bf16", delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=31)
    inp = I.make_scan_inputs(spec)
    h0 = _state(2, 264, 16, 32)
    out, fs = _scan(inp, True, h0, hint, tile)
    ry, rh = G.oracle_scan(inp, True, h0=h0.astype(np.float64))
    G.parity(G.host64(out), ry, "bf16", "y from h0 (hint %d, tile %d)" % (hint, tile))
    G.parity(G.host64(fs), rh, "state", "final state from h0 (hint %d, tile %d)" % (hint, tile))


@pytest.mark.parametrize("io", ["f32", "bf16"])
def test_split_sequence_continues(torch, io):
    spec = I.ScanSpec(2, 400, 64, io=io, delta_lo=1e-4, delta_hi=1e-2, D_kind="none",
                      gate=False, seed=33)
    inp = I.make_scan_inputs(spec)
    L1 = 160
    first = {k: (v[:, :L1] if k in ("x", "delta", "z", "B", "C") and v is not None else v)
             for k, v in inp.items()}
    second = {k: (np.ascontiguousarray(v[:, L1:]) if k in ("x", "delta", "z", "B", "C")
                  and v is not None else v) for k, v in inp.items()}
    first = {k: (np.ascontiguousarray(v) if isinstance(v, np.ndarray) else v) for k, v in first.items()}
    _, fs1 = G.gpu_scan(first, False, chunk_len_hint=64)
    out2, fs2 = _scan(second, False, G.host64(fs1).astype(np.float32), hint=64)
    ry, rh = G.oracle_scan(inp, False)
    G.parity(G.host64(out2), ry[:, L1:], io, "continued y")
    G.parity(G.host64(fs2), rh, "state", "continued final state")


def test_zero_length_copies_state(torch):
    from selective_state_space_119_b300 import libssm
    t = torch
    x = t.zeros((2, 0, 8), dtype=t.bfloat16, device="cuda")
    BC = t.zeros((2, 0, 16), dtype=t.bfloat16, device="cuda")
    A = t.full((8, 16), -1.0, device="cuda")
    h0 = t.randn(2, 8, 16, device="cuda")
    out, fs = libssm.ssm_selective_scan_fwd(x, x, A, BC, BC, h0=h0)
    t.cuda.synchronize()
    assert t.equal(fs, h0)


def test_decode_continues_from_state_scan(torch):
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(1, 64, 32, io="bf16", seed=35)
    inp = I.make_scan_inputs(spec)
    h0 = _state(1, 32, 16, 36)
    _, fs = _scan(inp, False, h0)
    dspec = I.DecodeSpec(1, 32, steps=1, seed=37)
    dinp = I.make_decode_inputs(dspec)
    state = fs.clone()
    yd = libssm.ssm_state_update(state, G.dev(dinp["x"][0]), G.dev(dinp["delta"][0]),
                                 G.dev(dinp["A"]), G.dev(dinp["B"][0]), G.dev(dinp["C"][0]),
                                 D=G.dev(dinp["D"]), z=G.dev(dinp["z"][0]))
    torch.cuda.synchronize()
    _, rh = G.oracle_scan(inp, False, h0=h0.astype(np.float64))
    ro, rs = oracle.state_update(rh, I.widen(dinp["x"][0]), I.widen(dinp["delta"][0]), dinp["A"],
                                 I.widen(dinp["B"][0]), I.widen(dinp["C"][0]), D=dinp["D"],
                                 z=I.widen(dinp["z"][0]))
    G.parity(G.host64(yd), ro, "bf16", "decode after a from-state scan")
    G.parity(G.host64(state), rs, "state", "decode state after a from-state scan")


def test_from_state_argument_errors(torch):
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(1, 40, 16, io="bf16", seed=38)
    inp = I.make_scan_inputs(spec)
    h0 = torch.zeros(1, 16, 16, device="cuda")
    x = G.dev(inp["x"])
    with pytest.raises(libssm.SSMError) as e:       # h0 is the final-state buffer
        libssm.ssm_selective_scan_fwd(x, G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(inp["B"]),
                                      G.dev(inp["C"]), h0=h0, final_state=h0)
    assert e.value.code == libssm.SSM_ERR_ALIAS
