"""GPU parity of ssm_state_update (one token of recurrent generation) through
the C ABI.

* The full decode workload (batch 256, dim 5120, N 16, bf16 tokens, fp32
  state ~ N(0,1)) stepped 64 times equals the oracle's scan over the same 64
  tokens started from that state (sampled batch rows, every channel).
* 64 steps from a zero state equal the GPU scan over the same tokens, token by
  token and in the final state ("State Space Models -- Mamba, S4, and Beyond",
  "Common Pitfalls" / "Verification Checklist": recurrent inference must
  reproduce the parallel scan).
* Small cases over dstate, I/O type and every optional argument against the
  oracle's step; guard bands around the state; argument errors.
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


def _steps(inp, t):
    return {k: (None if inp.get(k) is None else inp[k][t]) for k in ("x", "delta", "z", "B", "C")}


def _run_decode(inp, state, softplus=False, bias=None):
    from selective_state_space_119_b300 import libssm
    ys = []
    A, D = G.dev(inp["A"]), G.dev(inp.get("D"))
    for t in range(inp["x"].shape[0]):
        s = _steps(inp, t)
        ys.append(libssm.ssm_state_update(state, G.dev(s["x"]), G.dev(s["delta"]), A,
                                          G.dev(s["B"]), G.dev(s["C"]), D=D, z=G.dev(s["z"]),
                                          delta_bias=bias, delta_softplus=softplus))
    return ys


def test_decode_workload_equals_scan_from_state(torch):
    spec = I.WORKLOADS["decode_bf16_b256_d5120_x64"]
    inp = I.make_decode_inputs(spec)
    state = G.dev(inp["state0"])
    ys = _run_decode(inp, state)
    y = torch.stack(ys, dim=1)                           # [b, steps, d]
    bsel = np.array([0, 1, 128, 255])
    tr = lambda a: None if a is None else np.ascontiguousarray(np.swapaxes(a, 0, 1))
    seq = {"x": tr(inp["x"]), "delta": tr(inp["delta"]), "z": tr(inp["z"]), "B": tr(inp["B"]),
           "C": tr(inp["C"]), "A": inp["A"], "D": inp["D"], "delta_bias": None}
    ry, rh = G.oracle_scan(seq, False, bsel=bsel, h0=inp["state0"][bsel].astype(np.float64))
    G.parity(G.host64(y[torch.as_tensor(bsel, device="cuda")]), ry, "bf16", "decode y")
    G.parity(G.host64(state[torch.as_tensor(bsel, device="cuda")]), rh, "state", "decode state")


def test_decode_from_zero_equals_gpu_scan(torch):
    spec = I.DecodeSpec(8, 512, steps=64, state_init="zero", seed=77)
    inp = I.make_decode_inputs(spec)
    state = G.dev(inp["state0"])
    ys = _run_decode(inp, state)
    y_dec = torch.stack(ys, dim=1)
    tr = lambda a: None if a is None else np.ascontiguousarray(np.swapaxes(a, 0, 1))
    seq = {"x": tr(inp["x"]), "delta": tr(inp["delta"]), "z": tr(inp["z"]), "B": tr(inp["B"]),
           "C": tr(inp["C"]), "A": inp["A"], "D": inp["D"], "delta_bias": None}
    for hint in (16, 64):
        y_scan, fs = G.gpu_scan(seq, False, chunk_len_hint=hint)
        G.parity(G.host64(y_dec), G.host64(y_scan), "bf16", "decode vs scan y")
        G.parity(G.host64(state), G.host64(fs), "state", "decode vs scan state")


@pytest.mark.parametrize("N", [1, 2, 4, 8, 16])
@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("opts", ["all", "bare", "softplus_bias"])
def test_step_matches_oracle(torch, N, io, opts):
    spec = I.DecodeSpec(3, 40, N=N, steps=3, io=io, seed=31, A_kind="lognormal",
                        D_kind="none" if opts == "bare" else "uniform", gate=opts != "bare")
    inp = I.make_decode_inputs(spec)
    bias = None
    softplus = opts == "softplus_bias"
    if softplus:
        bias = np.linspace(-3.0, 0.5, 40).astype(np.float32)
    state = G.dev(inp["state0"])
    st = inp["state0"].astype(np.float64)
    ys = _run_decode(inp, state, softplus, None if bias is None else G.dev(bias))
    for t in range(spec.steps):
        s = _steps(inp, t)
        ry, st = oracle.state_update(st, I.widen(s["x"]), I.widen(s["delta"]), inp["A"],
                                     I.widen(s["B"]), I.widen(s["C"]), D=inp["D"],
                                     z=I.widen(s["z"]), delta_bias=bias, delta_softplus=softplus)
        G.parity(G.host64(ys[t]), ry, io, "step %d y" % t)
    G.parity(G.host64(state), st, "state", "state after steps")


def test_state_guard_bands_and_errors(torch):
    from selective_state_space_119_b300 import libssm
    spec = I.DecodeSpec(4, 64, steps=1, seed=5)
    inp = I.make_decode_inputs(spec)
    n = 4 * 64 * 16
    pad = 1024
    big = torch.full((pad + n + pad,), 3.5, device="cuda")
    state = big[pad:pad + n].view(4, 64, 16)
    state.copy_(G.dev(inp["state0"]))
    _run_decode(inp, state)
    torch.cuda.synchronize()
    assert torch.all(big[:pad] == 3.5) and torch.all(big[pad + n:] == 3.5)
    s = _steps(inp, 0)
    x = G.dev(s["x"])
    with pytest.raises(libssm.SSMError) as e:     # out aliases the state
        libssm.ssm_state_update(state, x, G.dev(s["delta"]), G.dev(inp["A"]), G.dev(s["B"]),
                                G.dev(s["C"]),
                                out=state.view(torch.bfloat16).view(-1)[:256].view(4, 64))
    assert e.value.code == libssm.SSM_ERR_ALIAS


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("N", [4, 16])
@pytest.mark.parametrize("zoh", [False, True])
def test_per_channel_rows_decode_step(torch, io, N, zoh):
    """B, C with one row per channel ([batch, dim, N]): each step against the
    oracle's per-channel step (Oracle.state_update_bcd) over three tokens, with
    softplus(delta + bias), D and the gate; rows past the last full warp and
    batch rows past a CTA row are covered by dim 264 and batch 5."""
    from selective_state_space_119_b300 import libssm
    spec = I.DecodeSpec(5, 264, N=N, steps=3, io=io, seed=31 + N)
    inp = I.make_decode_inputs(spec)
    r = np.random.default_rng(77 + N)
    B4 = I.store(r.standard_normal((3, 5, 264, N)), io)
    C4 = I.store(r.standard_normal((3, 5, 264, N)), io)
    bias = r.uniform(-3.0, -1.0, 264).astype(np.float32)
    state = G.dev(inp["state0"])
    ref_state = inp["state0"].astype(np.float64)
    for t in range(3):
        y = libssm.ssm_state_update(state, G.dev(inp["x"][t]), G.dev(inp["delta"][t]),
                                    G.dev(inp["A"]), G.dev(B4[t]), G.dev(C4[t]),
                                    D=G.dev(inp["D"]), z=G.dev(inp["z"][t]),
                                    delta_bias=G.dev(bias), delta_softplus=True, zoh=zoh)
        ry, ref_state = oracle.default().state_update_bcd(
            ref_state, I.widen(inp["x"][t]), I.widen(inp["delta"][t]),
            np.asarray(inp["A"], np.float64), I.widen(B4[t]), I.widen(C4[t]),
            D=np.asarray(inp["D"], np.float64), z=I.widen(inp["z"][t]), delta_bias=bias,
            delta_softplus=True, zoh=zoh)
        G.parity(G.host64(y), ry, io, "per-channel step %d y" % t)
        G.parity(G.host64(state), ref_state, "state", "per-channel step %d state" % t)


def test_per_channel_rows_decode_equals_per_channel_scan(torch):
    """k per-channel steps from zero equal the GPU's per-channel scan over the
    same k tokens (y per token and the final state)."""
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(2, 40, 128, io="bf16", seed=45)
    inp = I.make_scan_inputs(spec)
    B4, C4 = I.make_bc_per_channel(spec)
    t = {k: G.dev(v) for k, v in inp.items()}
    out, fs = libssm.ssm_selective_scan_fwd(t["x"], t["delta"], t["A"], G.dev(B4), G.dev(C4),
                                            D=t["D"], z=t["z"], delta_softplus=False)
    state = torch.zeros((2, 128, 16), dtype=torch.float32, device="cuda")
    ys = []
    for k in range(40):
        ys.append(libssm.ssm_state_update(
            state, t["x"][:, k].contiguous(), t["delta"][:, k].contiguous(), t["A"],
            G.dev(B4[:, k]), G.dev(C4[:, k]), D=t["D"], z=t["z"][:, k].contiguous()))
    G.parity(G.host64(torch.stack(ys, dim=1)), G.host64(out), "bf16", "steps vs per-channel scan")
    G.parity(G.host64(state), G.host64(fs), "state", "steps vs per-channel scan state")
