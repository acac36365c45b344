"""Helpers for the GPU parity tests: upload seeded inputs, run the CUDA path
through the C ABI, run the oracle on the same (widened) inputs, and compare
with the tolerances the workloads fix:

  fp32 I/O : max |err| <= 1e-4 * (1 + |y|)
  bf16 I/O : relative L2 <= 3e-3 and max |err| <= 2e-2 * (1 + |y|)
  fp32 states (final_state, decode state): max |err| <= 1e-4 * (1 + |h|)
"""
from __future__ import annotations

import numpy as np

import oracle
from selective_state_space_119_b300 import inputs as I

TOL_F32 = 1e-4
TOL_BF16_L2 = 3e-3
TOL_BF16_MAX = 2e-2
TOL_STATE = 1e-4


def torch():
    import torch as t
    return t


def dev(arr, device="cuda"):
    """numpy stored array (fp32, or uint16 bf16 bits) -> CUDA tensor."""
    t = torch()
    if arr is None:
        return None
    if arr.dtype == np.uint16:
        return t.from_numpy(np.ascontiguousarray(arr).view(np.int16)).to(device).view(t.bfloat16)
    return t.from_numpy(np.ascontiguousarray(arr)).to(device)


def host64(tensor):
    """CUDA tensor -> float64 numpy (exact)."""
    t = torch()
    return tensor.detach().to(t.float32).cpu().numpy().astype(np.float64)


def parity(got, ref, io, what=""):
    """Assert the tolerance of the I/O type; return the error statistics."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (what, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), "%s: non-finite output" % what
    err = np.abs(got - ref)
    scale = 1.0 + np.abs(ref)
    max_rel = float((err / scale).max()) if err.size else 0.0
    nref = float(np.linalg.norm(ref))
    rel_l2 = float(np.linalg.norm(got - ref) / nref) if nref > 0 else float(np.linalg.norm(got))
    stats = {"max_scaled_err": max_rel, "rel_l2": rel_l2}
    if io == "f32":
        assert max_rel <= TOL_F32, "%s: max|err|/(1+|y|) = %.3e > %.0e" % (what, max_rel, TOL_F32)
    elif io == "state":
        assert max_rel <= TOL_STATE, "%s: max|err|/(1+|h|) = %.3e > %.0e" % (what, max_rel, TOL_STATE)
    else:
        assert rel_l2 <= TOL_BF16_L2, "%s: rel L2 %.3e > %.0e" % (what, rel_l2, TOL_BF16_L2)
        assert max_rel <= TOL_BF16_MAX, "%s: max|err|/(1+|y|) = %.3e > %.0e" % (
            what, max_rel, TOL_BF16_MAX)
    return stats


def gpu_scan(inp, softplus, final_state=True, chunk_len_hint=0, workspace=None, tile_config_hint=0,
             **override):
    """Run ssm_selective_scan_fwd on stored inputs; returns (out tensor, fs tensor)."""
    from selective_state_space_119_b300 import libssm
    a = dict(inp)
    a.update(override)
    out, fs = libssm.ssm_selective_scan_fwd(
        dev(a["x"]), dev(a["delta"]), dev(a["A"]), dev(a["B"]), dev(a["C"]),
        D=dev(a.get("D")), z=dev(a.get("z")), delta_bias=dev(a.get("delta_bias")),
        delta_softplus=softplus, return_final_state=final_state,
        chunk_len_hint=chunk_len_hint, workspace=workspace, tile_config_hint=tile_config_hint)
    return out, fs


def oracle_scan(inp, softplus, dsel=None, bsel=None, h0=None, **override):
    """Oracle on the widened stored inputs, optionally on a subset of channels
    (dsel) and batch rows (bsel); selection is plain indexing."""
    a = dict(inp)
    a.update(override)
    x, delta, z, B, C = a["x"], a["delta"], a.get("z"), a["B"], a["C"]
    A = np.asarray(a["A"], np.float64)
    D = None if a.get("D") is None else np.asarray(a["D"], np.float64)
    bias = None if a.get("delta_bias") is None else np.asarray(a["delta_bias"], np.float64)
    if bsel is not None:
        x, delta, B, C = x[bsel], delta[bsel], B[bsel], C[bsel]
        z = None if z is None else z[bsel]
    if dsel is not None:
        x, delta = x[:, :, dsel], delta[:, :, dsel]
        z = None if z is None else z[:, :, dsel]
        A = A[dsel]
        D = None if D is None else D[dsel]
        bias = None if bias is None else bias[dsel]
    return oracle.selective_scan(I.widen(x), I.widen(delta), A, I.widen(B), I.widen(C), D=D,
                                 z=I.widen(z), delta_bias=bias, delta_softplus=softplus, h0=h0)
