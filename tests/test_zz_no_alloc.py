"""ssm_selective_scan_fwd_static: the scan for callers that cannot allocate.

Plain C hosts, plugins handed only their inputs and outputs, and callers that
must not call cudaMalloc on the hot path use this entry point; its scratch is
a fixed array inside the library instead of a caller workspace. This file runs
it through the C ABI and checks it against the workspace entry point, with the
tolerances of the other parity tests, on two calls in a row (different inputs,
so a stale carry left in the shared array by the first call would show in the
second). It also checks that a size needing more than the array is refused
before anything is enqueued. The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import gpu_util as G
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


def _vp(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def test_static_scratch_matches_workspace_entry_point(torch):
    from selective_state_space_119_b300 import libssm
    hint = 64
    for call, seed in enumerate((901, 902)):
        spec = I.ScanSpec(2, 600, 264, io="bf16", delta_kind="softplus_bias",
                          A_kind="lognormal", D_kind="uniform", seed=seed)
        need = libssm.ssm_scan_workspace_bytes(2, 600, 264, 16, "bf16", chunk_len_hint=hint)
        assert 0 < need <= libssm.SSM_STATIC_SCRATCH_BYTES     # the scratch is really used
        inp = I.make_scan_inputs(spec)
        t = {k: G.dev(v) for k, v in inp.items()}
        ref_out, ref_fs = libssm.ssm_selective_scan_fwd(
            t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
            delta_bias=t["delta_bias"], delta_softplus=True, chunk_len_hint=hint)

        out = torch.full_like(t["x"], float("nan"))
        fs = torch.full((2, 264, 16), float("nan"), device="cuda")
        dims = libssm.make_dims(2, 600, 264, 16, libssm.SSM_BF16, chunk_len_hint=hint)
        stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
        rc = libssm.lib.ssm_selective_scan_fwd_static(
            _vp(t["x"]), _vp(t["delta"]), _vp(t["A"]), _vp(t["B"]), _vp(t["C"]), _vp(t["D"]),
            _vp(t["z"]), _vp(t["delta_bias"]), 1, _vp(out), _vp(fs), ctypes.byref(dims), stream)
        assert rc == 0, libssm.ssm_strerror(rc)
        torch.cuda.synchronize()
        G.parity(G.host64(out), G.host64(ref_out), "bf16", "static scratch y (call %d)" % call)
        G.parity(G.host64(fs), G.host64(ref_fs), "state", "static scratch state (call %d)" % call)
        # and against the oracle on a few channels
        dsel = np.array([0, 7, 131, 263])
        ry, _ = G.oracle_scan(inp, True, dsel=dsel)
        G.parity(G.host64(out[:, :, torch.as_tensor(dsel, device="cuda")]), ry, "bf16",
                 "static scratch vs oracle (call %d)" % call)


def test_static_scratch_refuses_oversized_problems(torch):
    from selective_state_space_119_b300 import libssm
    # 64 x 255 chunk carries of 4096 channels need far more than 16 MiB; the
    # buffers are NULL, so no ordering of the checks can reach a launch
    dims = libssm.make_dims(64, 4096, 4096, 16, libssm.SSM_BF16, chunk_len_hint=16)
    assert libssm.lib.ssm_scan_workspace_bytes(ctypes.byref(dims)) > libssm.SSM_STATIC_SCRATCH_BYTES
    rc = libssm.lib.ssm_selective_scan_fwd_static(
        None, None, None, None, None, None, None, None, 0, None, None, ctypes.byref(dims), None)
    assert rc == libssm.SSM_ERR_WORKSPACE


def test_static_scratch_reports_a_wait_that_gave_up(torch):
    """A bounded wait that runs out on the static scratch's status word is
    reported by ssm_get_static_status (once: reading clears it), and the next
    static call still matches the workspace entry point."""
    from selective_state_space_119_b300 import libssm
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert libssm.lib.ssm_get_static_status(stream) == libssm.SSM_OK
    assert libssm.lib.ssm_debug_timeout_probe_static(1 << 12, stream) == libssm.SSM_OK
    assert libssm.lib.ssm_get_static_status(stream) == libssm.SSM_ERR_TIMEOUT
    assert libssm.lib.ssm_get_static_status(stream) == libssm.SSM_OK
    spec = I.ScanSpec(1, 300, 128, io="bf16", delta_kind="softplus_bias",
                      A_kind="lognormal", D_kind="uniform", seed=903)
    inp = I.make_scan_inputs(spec)
    t = {k: G.dev(v) for k, v in inp.items()}
    ref_out, _ = libssm.ssm_selective_scan_fwd(
        t["x"], t["delta"], t["A"], t["B"], t["C"], D=t["D"], z=t["z"],
        delta_bias=t["delta_bias"], delta_softplus=True, chunk_len_hint=64)
    out = torch.full_like(t["x"], float("nan"))
    dims = libssm.make_dims(1, 300, 128, 16, libssm.SSM_BF16, chunk_len_hint=64)
    rc = libssm.lib.ssm_selective_scan_fwd_static(
        _vp(t["x"]), _vp(t["delta"]), _vp(t["A"]), _vp(t["B"]), _vp(t["C"]), _vp(t["D"]),
        _vp(t["z"]), _vp(t["delta_bias"]), 1, _vp(out), None, ctypes.byref(dims), stream)
    assert rc == 0, libssm.ssm_strerror(rc)
    assert libssm.lib.ssm_get_static_status(stream) == libssm.SSM_OK
    G.parity(G.host64(out), G.host64(ref_out), "bf16", "static scratch after a timeout")
