"""GPU parity of the Mamba block's input stage: the causal depthwise conv1d +
SiLU on its own (ssm_causal_conv1d_silu) and fused in front of the scan
(ssm_selective_scan_fwd_conv). "State Space Models -- Mamba, S4, and Beyond",
"Mamba (S6 -- Selective State Space)", MambaBlock: Conv1d(kernel_size=d_conv,
groups=d_inner, padding=d_conv-1) cut to seq_len, then SiLU, then the scan
on its output.

Covered: every conv width 1..4, with and without bias, fp32 and bf16, ragged
sequence ends and sequences shorter than the conv window; the fused scan
against the oracle's conv followed by the oracle's scan, over L-chunk hints
(a chunk's first tokens take their conv window from the previous chunk) and
both tile configurations it runs; the fused call equals the two-call path;
the full-size workload (batch 4, L 2048, dim 1536) on sampled channels.
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


def _conv_gpu(x, w, b):
    from selective_state_space_119_b300 import libssm
    return libssm.ssm_causal_conv1d_silu(G.dev(x), G.dev(w), G.dev(b))


def _conv_ref(x, w, b, dsel=None):
    xw = I.widen(x)
    w64 = np.asarray(w, np.float64)
    b64 = None if b is None else np.asarray(b, np.float64)
    if dsel is not None:
        xw, w64 = np.ascontiguousarray(xw[:, :, dsel]), w64[dsel]
        b64 = None if b64 is None else b64[dsel]
    return oracle.causal_conv1d_silu(xw, w64, b64)


def _fused_gpu(inp, softplus, w, b, hint=0, tile=0):
    from selective_state_space_119_b300 import libssm
    return libssm.ssm_selective_scan_fwd(
        G.dev(inp["x"]), G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(inp["B"]), G.dev(inp["C"]),
        D=G.dev(inp.get("D")), z=G.dev(inp.get("z")), delta_bias=G.dev(inp.get("delta_bias")),
        delta_softplus=softplus, chunk_len_hint=hint, tile_config_hint=tile,
        conv_w=G.dev(w), conv_b=G.dev(b))


def _fused_ref(inp, softplus, w, b, dsel=None):
    """The oracle's conv, then the oracle's scan on its output."""
    u = _conv_ref(inp["x"], w, b, dsel)
    a = {k: v for k, v in inp.items()}
    sel = (lambda v: v) if dsel is None else (lambda v: np.ascontiguousarray(v[:, :, dsel]))
    A = np.asarray(a["A"], np.float64)
    D = None if a.get("D") is None else np.asarray(a["D"], np.float64)
    bias = None if a.get("delta_bias") is None else np.asarray(a["delta_bias"], np.float64)
    if dsel is not None:
        A = A[dsel]
        D = None if D is None else D[dsel]
        bias = None if bias is None else bias[dsel]
    z = None if a.get("z") is None else sel(I.widen(a["z"]))
    return oracle.selective_scan(u, sel(I.widen(a["delta"])), A, I.widen(a["B"]),
                                 I.widen(a["C"]), D=D, z=z, delta_bias=bias,
                                 delta_softplus=softplus)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("bias", [True, False])
def test_conv_matches_oracle(torch, io, K, bias):
    spec = I.ScanSpec(2, 45, 264, io=io, gate=False, seed=41)
    x = I.make_scan_inputs(spec)["x"]
    w, b = I.make_conv_weights(264, K, bias, seed=42 + K)
    u = _conv_gpu(x, w, b)
    G.parity(G.host64(u), _conv_ref(x, w, b), io, "conv K=%d bias=%s" % (K, bias))


@pytest.mark.parametrize("L", [1, 2, 3, 8, 9, 17])
def test_conv_short_and_ragged_sequences(torch, L):
    # shorter than the window, one run, a run plus one token
    spec = I.ScanSpec(3, L, 64, io="bf16", gate=False, seed=43)
    x = I.make_scan_inputs(spec)["x"]
    w, b = I.make_conv_weights(64, 4, True, seed=44)
    G.parity(G.host64(_conv_gpu(x, w, b)), _conv_ref(x, w, b), "bf16", "conv L=%d" % L)


def test_conv_empty(torch):
    t = torch
    from selective_state_space_119_b300 import libssm
    x = t.zeros((2, 0, 16), dtype=t.bfloat16, device="cuda")
    w = t.ones((16, 4), device="cuda")
    u = libssm.ssm_causal_conv1d_silu(x, w)
    assert u.shape == (2, 0, 16)


@pytest.mark.parametrize("io", ["f32", "bf16"])
@pytest.mark.parametrize("K,bias", [(4, True), (4, False), (3, True), (1, True)])
@pytest.mark.parametrize("hint", [0, 32, 96])
def test_fused_scan_matches_oracle(torch, io, K, bias, hint):
    spec = I.ScanSpec(2, 300, 264, io=io, delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=45)
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(264, K, bias, seed=46)
    out, fs = _fused_gpu(inp, True, w, b, hint=hint)
    ry, rh = _fused_ref(inp, True, w, b)
    what = "fused K=%d bias=%s hint=%d" % (K, bias, hint)
    G.parity(G.host64(out), ry, io, "y " + what)
    G.parity(G.host64(fs), rh, "state", "final state " + what)


@pytest.mark.parametrize("tile", [0, 1])
@pytest.mark.parametrize("gate", [True, False])
def test_fused_scan_tiles_and_gate(torch, tile, gate):
    spec = I.ScanSpec(1, 200, 136, io="bf16", gate=gate, D_kind="none", seed=47)
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(136, 4, True, seed=48)
    out, fs = _fused_gpu(inp, False, w, b, hint=64, tile=tile)
    ry, rh = _fused_ref(inp, False, w, b)
    G.parity(G.host64(out), ry, "bf16", "fused tile %d gate %s" % (tile, gate))
    G.parity(G.host64(fs), rh, "state", "fused final state tile %d" % tile)


def test_fused_rejects_other_tiles(torch):
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(1, 64, 128, io="bf16", seed=49)
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(128, 4, True, seed=50)
    with pytest.raises(libssm.SSMError) as e:
        _fused_gpu(inp, False, w, b, tile=2)
    assert e.value.code == libssm.SSM_ERR_DIMS


def test_fused_equals_two_calls_f32(torch):
    # fp32 I/O: u is not rounded between the two calls, so the fused scan and
    # conv-then-scan differ only by fp32 evaluation order
    spec = I.ScanSpec(2, 260, 128, io="f32", delta_kind="softplus_bias", seed=51)
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(128, 4, True, seed=52)
    out_f, fs_f = _fused_gpu(inp, True, w, b, hint=64)
    u = _conv_gpu(inp["x"], w, b)
    out_2, fs_2 = G.gpu_scan(dict(inp, x=u.cpu().numpy()), True, chunk_len_hint=64)
    np.testing.assert_allclose(G.host64(out_f), G.host64(out_2), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(G.host64(fs_f), G.host64(fs_2), rtol=1e-5, atol=1e-5)


def test_full_size_workload_sampled(torch):
    """Batch 4, L 2048, dim 1536, bf16, softplus(delta + bias): the standalone
    conv and the fused scan against the oracle on sampled channels."""
    spec = I.WORKLOADS["scan_bf16_b4_L2048_d1536_softplus"]
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(spec.dim, 4, True, seed=53)
    dsel = np.array([0, 1, 127, 128, 777, 1535])
    u = G.host64(_conv_gpu(inp["x"], w, b))
    G.parity(u[:, :, dsel], _conv_ref(inp["x"], w, b, dsel), "bf16", "conv full size")
    out, fs = _fused_gpu(inp, True, w, b)
    ry, rh = _fused_ref(inp, True, w, b, dsel)
    G.parity(G.host64(out)[:, :, dsel], ry, "bf16", "fused y full size")
    G.parity(G.host64(fs)[:, dsel], rh, "state", "fused final state full size")


def test_guard_bands_untouched(torch):
    """u of the standalone conv and y of the fused scan, written into the middle
    of pattern-filled buffers (ragged sequence end, channel count not a multiple
    of a tile): the bands stay untouched; a second call is bit-identical."""
    from selective_state_space_119_b300 import libssm
    t = torch
    spec = I.ScanSpec(2, 203, 136, io="bf16", gate=True, seed=57)
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(136, 4, True, seed=58)
    n, pad = 2 * 203 * 136, 4096
    big = t.full((pad + n + pad,), 7.0, dtype=t.bfloat16, device="cuda")
    u = big[pad:pad + n].view(2, 203, 136)
    libssm.ssm_causal_conv1d_silu(G.dev(inp["x"]), G.dev(w), G.dev(b), out=u)
    t.cuda.synchronize()
    assert t.all(big[:pad] == 7.0) and t.all(big[pad + n:] == 7.0)
    G.parity(G.host64(u), _conv_ref(inp["x"], w, b), "bf16", "conv in guarded buffer")
    u2 = libssm.ssm_causal_conv1d_silu(G.dev(inp["x"]), G.dev(w), G.dev(b))
    assert t.equal(u, u2)
    big2 = t.full((pad + n + pad,), 7.0, dtype=t.bfloat16, device="cuda")
    out = big2[pad:pad + n].view(2, 203, 136)
    libssm.ssm_selective_scan_fwd(
        G.dev(inp["x"]), G.dev(inp["delta"]), G.dev(inp["A"]), G.dev(inp["B"]), G.dev(inp["C"]),
        D=G.dev(inp["D"]), z=G.dev(inp["z"]), out=out, chunk_len_hint=64, conv_w=G.dev(w),
        conv_b=G.dev(b))
    t.cuda.synchronize()
    assert t.all(big2[:pad] == 7.0) and t.all(big2[pad + n:] == 7.0)
