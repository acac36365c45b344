"""GPU parity of the input stage's gradients (ssm_causal_conv1d_silu_bwd,
through the C ABI) against the float64 oracle (oracle_causal_conv1d_silu_bwd,
itself pinned to finite differences and to autograd through torch's conv1d):
every conv width 1..4, with and without bias, fp32 and bf16, ragged sequence
ends and sequences shorter than the window; the full-size shapes of the
input-stage benchmark; and the chain of the scan's backward into the input
stage's against the oracle's gradients of the whole stage-plus-scan
(selective_scan_conv_bwd).

Tolerances: dx per element as the scan's per-element gradients (bf16:
2e-2 (1 + |ref|), relative L2 5e-3; fp32: 2e-4 (1 + |ref|), relative L2
5e-5); dconv_w and dconv_b, sums over every row and token, against the
largest entry of the array, at least 1 (2e-4, relative L2 5e-5)."""
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


def elem(got, ref, io, what):
    mx, l2 = {"f32": (2e-4, 5e-5), "bf16": (2e-2, 5e-3)}[io]
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), what
    worst = float((np.abs(got - ref) / (1 + np.abs(ref))).max()) if ref.size else 0.0
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), np.sqrt(ref.size))) if ref.size else 0.0
    assert worst <= mx, "%s: max %.3e" % (what, worst)
    assert rel <= l2, "%s: rel L2 %.3e" % (what, rel)


def summed(got, ref, what):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape and np.all(np.isfinite(got)), what
    scale = max(float(np.abs(ref).max()), 1.0)
    assert float(np.abs(got - ref).max()) / scale <= 2e-4, what
    rel = float(np.linalg.norm(got - ref) / max(np.linalg.norm(ref), np.sqrt(ref.size)))
    assert rel <= 5e-5, "%s: rel L2 %.3e" % (what, rel)


def _case(batch, L, dim, K, io, bias, seed):
    spec = I.ScanSpec(batch, L, dim, io=io, seed=seed)
    x = I.make_scan_inputs(spec)["x"]
    w, b = I.make_conv_weights(dim, K, bias, seed=seed + 1)
    du = I.store(np.random.default_rng(seed + 2).standard_normal((batch, L, dim)), io)
    return x, w, b, du


@pytest.mark.parametrize("io", ["bf16", "f32"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("bias", [True, False])
@pytest.mark.parametrize("L", [2, 77, 300])
def test_input_stage_gradients(torch, io, K, bias, L):
    from selective_state_space_119_b300 import libssm
    x, w, b, du = _case(2, L, 264, K, io, bias, 100 + K + L)
    dx, dw, db = libssm.ssm_causal_conv1d_silu_bwd(G.dev(x), G.dev(w), G.dev(du),
                                                   conv_b=G.dev(b))
    ref = oracle.causal_conv1d_silu_bwd(I.widen(x), np.asarray(w, np.float64), I.widen(du),
                                        bias=None if b is None else np.asarray(b, np.float64))
    elem(G.host64(dx), ref["dx"], io, "dx K %d L %d" % (K, L))
    summed(G.host64(dw), ref["dw"], "dconv_w K %d L %d" % (K, L))
    summed(G.host64(db), ref["dbias"], "dconv_b K %d L %d" % (K, L))


@pytest.mark.parametrize("io,K", [("bf16", 4), ("f32", 3)])
def test_input_stage_gradients_guard_bands(torch, io, K):
    """dx, dconv_w and dconv_b written into the middle of pattern-filled
    buffers through the C ABI (a ragged last token tile and channel tile): the
    bands before and after stay untouched, and the values match the oracle."""
    import ctypes
    from selective_state_space_119_b300 import libssm
    t = torch
    batch, L, dim = 2, 77, 264
    x, w, b, du = _case(batch, L, dim, K, io, True, 211 + K)
    xd, wd, bd, dud = G.dev(x), G.dev(w), G.dev(b), G.dev(du)
    pad = 4096

    def guarded(n, dtype, fill):
        big = t.full((pad + n + pad,), fill, dtype=dtype, device="cuda")
        return big, big[pad:pad + n]

    big_dx, dx = guarded(batch * L * dim, xd.dtype, 3.0)
    big_dw, dw = guarded(dim * K, t.float32, -5.0)
    big_db, db = guarded(dim, t.float32, -5.0)
    code = libssm.SSM_BF16 if io == "bf16" else libssm.SSM_F32
    dims = libssm.make_dims(batch, L, dim, 16, code)
    nb = int(libssm.lib.ssm_causal_conv1d_silu_bwd_workspace_bytes(ctypes.byref(dims), K))
    ws = t.full((nb,), 0x5A, dtype=t.uint8, device="cuda")
    dims = libssm.make_dims(batch, L, dim, 16, code, ws.data_ptr(), nb)
    p = lambda v: ctypes.c_void_p(v.data_ptr())
    rc = libssm.lib.ssm_causal_conv1d_silu_bwd(p(xd), p(wd), p(bd), K, p(dud), p(dx), p(dw), p(db),
                                               ctypes.byref(dims), None)
    assert rc == libssm.SSM_OK
    t.cuda.synchronize()
    for big, fill, name in ((big_dx, 3.0, "dx"), (big_dw, -5.0, "dconv_w"), (big_db, -5.0, "dconv_b")):
        assert t.all(big[:pad] == fill) and t.all(big[-pad:] == fill), name + " band written"
    ref = oracle.causal_conv1d_silu_bwd(I.widen(x), np.asarray(w, np.float64), I.widen(du),
                                        bias=np.asarray(b, np.float64))
    elem(G.host64(dx.view(batch, L, dim)), ref["dx"], io, "guarded dx")
    summed(G.host64(dw.view(dim, K)), ref["dw"], "guarded dconv_w")
    summed(G.host64(db), ref["dbias"], "guarded dconv_b")


def test_input_stage_gradients_full_size(torch):
    """The input-stage benchmark's shapes (batch 4, L 2048, dim 1536, width 4),
    every element of dx and every weight; and bit-identical on a repeat."""
    from selective_state_space_119_b300 import libssm
    x, w, b, du = _case(4, 2048, 1536, 4, "bf16", True, 7)
    args = (G.dev(x), G.dev(w), G.dev(du))
    dx, dw, db = libssm.ssm_causal_conv1d_silu_bwd(*args, conv_b=G.dev(b))
    dx2, dw2, db2 = libssm.ssm_causal_conv1d_silu_bwd(*args, conv_b=G.dev(b))
    assert torch.equal(dx, dx2) and torch.equal(dw, dw2) and torch.equal(db, db2)
    ref = oracle.causal_conv1d_silu_bwd(I.widen(x), np.asarray(w, np.float64), I.widen(du),
                                        bias=np.asarray(b, np.float64))
    elem(G.host64(dx), ref["dx"], "bf16", "dx full size")
    summed(G.host64(dw), ref["dw"], "dconv_w full size")
    summed(G.host64(db), ref["dbias"], "dconv_b full size")


@pytest.mark.parametrize("hint", [0, 64])
def test_stage_then_scan_gradients_chain(torch, hint):
    """The training path of the block's stage plus scan: u = the stage's
    output, the checkpointing scan on u, the scan's backward (its dx is dLoss/du),
    then the stage's backward; against the oracle's gradients of the whole
    (selective_scan_conv_bwd), fp32 I/O so that u is not rounded between the two."""
    from selective_state_space_119_b300 import libssm
    spec = I.ScanSpec(2, 200, 128, io="f32", delta_kind="softplus_bias", A_kind="lognormal",
                      D_kind="uniform", seed=211)
    inp = I.make_scan_inputs(spec)
    w, b = I.make_conv_weights(128, 4, True, seed=212)
    dout = I.store(np.random.default_rng(213).standard_normal((2, 200, 128)), "f32")
    t = {k: G.dev(v) for k, v in inp.items()}
    u = libssm.ssm_causal_conv1d_silu(t["x"], G.dev(w), G.dev(b))
    _, _, ck = libssm.ssm_selective_scan_fwd_ckpt(
        u, t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"], delta_bias=t["delta_bias"],
        delta_softplus=True, chunk_len_hint=hint)
    g = libssm.ssm_selective_scan_bwd(
        u, t["delta"], t["A"], t["B"], t["C"], ck, G.dev(dout), D=t["D"], z=t["z"],
        delta_bias=t["delta_bias"], delta_softplus=True, chunk_len_hint=hint)
    dx, dw, db = libssm.ssm_causal_conv1d_silu_bwd(t["x"], G.dev(w), g["dx"], conv_b=G.dev(b))
    ref = oracle.selective_scan_conv_bwd(
        I.widen(inp["x"]), I.widen(inp["delta"]), np.asarray(inp["A"], np.float64),
        I.widen(inp["B"]), I.widen(inp["C"]), np.asarray(w, np.float64), I.widen(dout),
        conv_bias=np.asarray(b, np.float64), D=np.asarray(inp["D"], np.float64),
        z=I.widen(inp["z"]), delta_bias=np.asarray(inp["delta_bias"], np.float64),
        delta_softplus=True)
    elem(G.host64(dx), ref["dx"], "f32", "dx through stage and scan")
    elem(G.host64(g["ddelta"]), ref["ddelta"], "f32", "ddelta through stage and scan")
    summed(G.host64(dw), ref["dconv_w"], "dconv_w through stage and scan")
    summed(G.host64(db), ref["dconv_bias"], "dconv_b through stage and scan")
    summed(G.host64(g["dA"]), ref["dA"], "dA through stage and scan")
