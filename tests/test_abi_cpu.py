"""The C-ABI library on a host without a GPU: it loads, exports every symbol
include/ssm.h declares, sizes workspaces and plans, and rejects bad arguments
with the documented codes before touching CUDA (no compute calls here)."""
import ctypes
import os
import re

import pytest

from selective_state_space_119_b300 import build

build.build(quiet=True)
from selective_state_space_119_b300 import libssm as L  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "ssm.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ssm_[a-z_0-9]+)\s*\(", text)))


def test_exports_every_declared_symbol():
    names = declared_functions()
    assert set(names) == set(L.EXPORTED), names
    for n in names:
        assert hasattr(L.lib, n), n


def test_version_and_strerror():
    assert L.lib.ssm_version() >> 16 == 1
    for code in (0, -1, -2, -3, -4, -5, -6, -7, -8):
        assert L.ssm_strerror(code) and "unknown" not in L.ssm_strerror(code)
    assert "unknown" in L.ssm_strerror(-99)


def test_struct_layout_matches_header():
    # int64 x4, int32 x2, pointer, size_t, int32 x2
    assert ctypes.sizeof(L.ssm_dims) == 4 * 8 + 2 * 4 + 8 + 8 + 2 * 4
    assert ctypes.sizeof(L.ssm_plan) == 4 * 8 + 2 * 4


def test_workspace_and_plan():
    # one chunk -> only the 256-byte header (status word)
    assert L.ssm_scan_workspace_bytes(1, 64, 256, 16, "bf16", chunk_len_hint=64) == 256
    assert L.ssm_scan_workspace_bytes(0, 64, 256, 16, "bf16") == 0      # empty problem
    p = L.ssm_scan_plan(1, 64, 256, 16, "bf16", chunk_len_hint=64)
    assert p["nchunks"] == 1 and p["kernels"] == 1
    # several chunks -> header + carries; chunks are whole 32-token stages
    p = L.ssm_scan_plan(2, 1000, 512, 16, "bf16", chunk_len_hint=100)
    assert p["chunk_len"] == 128 and p["nchunks"] == 8 and p["kernels"] == 2
    # channels per CTA = 32 lanes (one channel each) * warps
    for cfg, ch in ((1, 128), (2, 64), (3, 32), (4, 96)):
        p = L.ssm_scan_plan(2, 1000, 512, 16, "bf16", tile_config_hint=cfg)
        assert p["tile_config"] == cfg - 1 and p["channels_per_cta"] == ch
    with pytest.raises(L.SSMError):
        L.ssm_scan_plan(2, 1000, 512, 16, "bf16", tile_config_hint=5)
    ws = L.ssm_scan_workspace_bytes(2, 1000, 512, 16, "bf16", chunk_len_hint=100)
    carries = 2 * 7 * 512
    assert ws >= 256 + carries * 16 * 4 + carries * 4
    # automatic plan fills the GPU for the long-sequence workload
    p = L.ssm_scan_plan(1, 131072, 5120, 16, "bf16")
    assert p["ctas"] >= 148 and p["chunk_len"] % 32 == 0
    # a channel-rich workload needs no L-split
    p = L.ssm_scan_plan(64, 2048, 4096, 16, "bf16")
    assert p["nchunks"] == 1
    # invalid sizes
    assert L.ssm_scan_workspace_bytes(1, 64, 256, 3, "bf16") == 0
    with pytest.raises(L.SSMError) as e:
        L.ssm_scan_plan(1, 64, 256, 32, "bf16")
    assert e.value.code == L.SSM_ERR_DIMS
    with pytest.raises(L.SSMError) as e:
        L.ssm_scan_plan(1, 64, 12, 16, "bf16")       # dim not a multiple of 8
    assert e.value.code == L.SSM_ERR_ALIGN
    with pytest.raises(L.SSMError) as e:
        L.ssm_scan_plan(-1, 64, 256, 16, "f32")
    assert e.value.code == L.SSM_ERR_DIMS


FAKE = 0x7f0000000000   # never dereferenced: every call below fails validation


def _scan(dims, x=FAKE, delta=FAKE + 4096, A=FAKE + 8192, B=FAKE + 12288, C=FAKE + 16384,
          D=None, z=None, bias=None, out=FAKE + (1 << 30), fs=None):
    return L.lib.ssm_selective_scan_fwd(x, delta, A, B, C, D, z, bias, 0, out, fs,
                                        ctypes.byref(dims), None)


def test_scan_rejects_bad_arguments_before_launch():
    d = L.make_dims(1, 4, 8, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 20)
    assert _scan(d, x=None) == L.SSM_ERR_NULL
    assert _scan(d, out=None) == L.SSM_ERR_NULL
    assert L.lib.ssm_selective_scan_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, 0,
                                        FAKE, None, None, None) == L.SSM_ERR_NULL
    assert _scan(L.make_dims(1, 4, 8, 5, "bf16")) == L.SSM_ERR_DIMS
    assert _scan(L.make_dims(1, -4, 8, 16, "bf16")) == L.SSM_ERR_DIMS
    bad = L.make_dims(1, 4, 8, 16, "bf16")
    bad.io_dtype = 7
    assert _scan(bad) == L.SSM_ERR_DTYPE
    assert _scan(L.make_dims(1, 4, 12, 16, "bf16")) == L.SSM_ERR_ALIGN
    assert _scan(L.make_dims(1, 4, 6, 16, "f32")) == L.SSM_ERR_ALIGN
    assert _scan(d, x=FAKE + 2) == L.SSM_ERR_ALIGN
    assert _scan(d, z=FAKE + 8) == L.SSM_ERR_ALIGN
    # out overlapping x
    assert _scan(d, out=FAKE + 16) == L.SSM_ERR_ALIAS
    # final_state overlapping out
    assert _scan(d, fs=FAKE + (1 << 30) + 16) == L.SSM_ERR_ALIAS
    # workspace missing / too small
    assert _scan(L.make_dims(1, 4, 8, 16, "bf16")) == L.SSM_ERR_WORKSPACE
    dw = L.make_dims(1, 4096, 8, 16, "bf16", chunk_len_hint=64)
    assert L.ssm_scan_workspace_bytes(1, 4096, 8, 16, "bf16", chunk_len_hint=64) > 0
    assert _scan(dw) == L.SSM_ERR_WORKSPACE
    dw.workspace = FAKE + (1 << 32)
    dw.workspace_bytes = 256
    assert _scan(dw) == L.SSM_ERR_WORKSPACE


def test_state_update_rejects_bad_arguments_before_launch():
    d = L.make_dims(2, 1, 8, 16, "bf16")
    f = L.lib.ssm_state_update

    def call(state=FAKE, x=FAKE + (1 << 20), out=FAKE + (2 << 20), dims=d):
        return f(state, x, FAKE + (3 << 20), FAKE + (4 << 20), FAKE + (5 << 20), FAKE + (6 << 20), None,
                 None, None, 0, out, ctypes.byref(dims) if dims is not None else None, None)

    assert call(state=None) == L.SSM_ERR_NULL
    assert call(dims=None) == L.SSM_ERR_NULL
    assert call(x=FAKE + (1 << 20) + 4) == L.SSM_ERR_ALIGN
    assert call(out=FAKE + 16) == L.SSM_ERR_ALIAS          # out inside the state
    assert call(dims=L.make_dims(2, 1, 8, 7, "bf16")) == L.SSM_ERR_DIMS


def test_binding_refuses_cpu_tensors():
    torch = pytest.importorskip("torch")
    x = torch.zeros(1, 4, 8, dtype=torch.bfloat16)
    A = torch.zeros(8, 16)
    with pytest.raises(ValueError):
        L.ssm_selective_scan_fwd(x, x, A, torch.zeros(1, 4, 16, dtype=torch.bfloat16),
                                 torch.zeros(1, 4, 16, dtype=torch.bfloat16),
                                 out=torch.empty_like(x), return_final_state=False)


def test_from_state_rejects_bad_arguments_before_launch():
    f = L.lib.ssm_selective_scan_fwd_from_state
    d = L.make_dims(1, 4, 8, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 20)

    def call(h0=FAKE + (1 << 31), fs=None, dims=d):
        return f(FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, None, None, None, 0,
                 h0, FAKE + (1 << 30), fs, ctypes.byref(dims), None)

    assert call(h0=None) == L.SSM_ERR_NULL                     # the state is required
    assert call(h0=FAKE + (1 << 31) + 4) == L.SSM_ERR_ALIGN
    assert call(fs=FAKE + (1 << 31)) == L.SSM_ERR_ALIAS         # final state over h0


def test_conv_entry_points_reject_bad_arguments_before_launch():
    d = L.make_dims(1, 4, 8, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 20)
    W = FAKE + (1 << 32)

    def scan(w=W, k=4, b=None, out=FAKE + (1 << 30), dims=d):
        return L.lib.ssm_selective_scan_fwd_conv(
            FAKE, w, b, k, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, None, None,
            None, 0, out, None, ctypes.byref(dims), None)

    def conv(w=W, k=4, b=None, u=FAKE + (1 << 30), x=FAKE, dims=d):
        return L.lib.ssm_causal_conv1d_silu(x, w, b, k, u, ctypes.byref(dims), None)

    for f in (scan, conv):
        assert f(w=None) == L.SSM_ERR_NULL                      # the taps are required
        assert f(k=0) == L.SSM_ERR_DIMS and f(k=5) == L.SSM_ERR_DIMS
        assert f(w=W + 4) == L.SSM_ERR_ALIGN
        assert f(b=W + 8) == L.SSM_ERR_ALIGN
    assert scan(out=W) == L.SSM_ERR_ALIAS                       # out over the taps
    assert conv(u=W + 16) == L.SSM_ERR_ALIAS
    assert conv(u=FAKE) == L.SSM_ERR_ALIAS                      # not in-place
    assert conv(u=FAKE + 16) == L.SSM_ERR_ALIAS                 # nor shifted over x
    # the fused stage runs tile configuration 0 only
    for hint, ok in ((0, True), (1, True), (2, False), (4, False)):
        dh = L.make_dims(1, 4, 8, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 20,
                         tile_config_hint=hint)
        rc = scan(dims=dh, out=W)      # an alias is reported after the hint check
        assert rc == (L.SSM_ERR_ALIAS if ok else L.SSM_ERR_DIMS), (hint, rc)
    # the standalone conv ignores dstate and the hints
    dz = L.make_dims(1, 4, 8, 3, "bf16", tile_config_hint=4, chunk_len_hint=7)
    assert conv(w=None, dims=dz) == L.SSM_ERR_NULL
    # empty problems enqueue nothing and need no pointers
    de = L.make_dims(0, 4, 8, 16, "bf16")
    assert conv(w=None, u=None, x=None, dims=de) == L.SSM_OK
    # bf16 dim must be a multiple of 8
    assert conv(dims=L.make_dims(1, 4, 12, 16, "bf16")) == L.SSM_ERR_ALIGN


def test_training_entry_points_reject_bad_arguments_before_launch():
    d = L.make_dims(1, 20, 16, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 24)
    CK = FAKE + (1 << 32)

    def fwd(ck=CK, dims=d, out=FAKE + (1 << 30)):
        return L.lib.ssm_selective_scan_fwd_ckpt(FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288,
                                                 FAKE + 16384, None, None, None, 0, None, out,
                                                 None, ck, ctypes.byref(dims), None)

    assert fwd(ck=None) == L.SSM_ERR_NULL
    assert fwd(ck=CK + 4) == L.SSM_ERR_ALIGN
    assert fwd(out=CK) == L.SSM_ERR_ALIAS                              # out over the checkpoints
    assert fwd(dims=L.make_dims(1, 20, 16, 8, "bf16")) == L.SSM_ERR_DIMS   # dstate 16 only
    assert fwd(dims=L.make_dims(1, 20, 16, 16, "bf16", tile_config_hint=3)) == L.SSM_ERR_DIMS
    # sizes: a state before every 8th token
    assert L.ssm_scan_checkpoint_bytes(2, 20, 16, 16, "bf16") == 2 * 3 * 16 * 16 * 4
    assert L.ssm_scan_checkpoint_bytes(2, 0, 16, 16, "bf16") == 0

    G = FAKE + (1 << 36)   # gradients live here, far from the inputs

    def bwd(dims=d, z=None, dz=None, dx=G, dA=G + 65536, ckpt=CK, dh0=None):
        return L.lib.ssm_selective_scan_bwd(
            FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, None, z, None, 0, ckpt,
            FAKE + 20480, None, dx, G + 4096, dA, G + 8192, G + 12288, None, dz, None, dh0,
            ctypes.byref(dims), None)

    assert bwd(ckpt=None) == L.SSM_ERR_NULL
    assert bwd(dA=None) == L.SSM_ERR_NULL
    assert bwd(z=FAKE + 24576) == L.SSM_ERR_NULL                       # z without dz
    assert bwd(dz=G + 16384) == L.SSM_ERR_NULL                         # dz without z
    assert bwd(dx=G + 2) == L.SSM_ERR_ALIGN
    assert bwd(dx=FAKE) == L.SSM_ERR_ALIAS                              # dx over x
    assert bwd(dx=G + 4096) == L.SSM_ERR_ALIAS                          # dx over ddelta
    assert bwd(dh0=CK) == L.SSM_ERR_ALIAS                               # dh0 over the checkpoints
    assert bwd(dims=L.make_dims(1, 20, 16, 4, "bf16")) == L.SSM_ERR_DIMS
    small = L.make_dims(1, 20, 16, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=256)
    assert bwd(dims=small) == L.SSM_ERR_WORKSPACE
    # workspace: the per-tile shares of dB | dC, dA, dD, dbias (+ carries when chunked)
    ws1 = L.ssm_scan_bwd_workspace_bytes(2, 1000, 512, 16, "bf16", chunk_len_hint=1024)
    ws8 = L.ssm_scan_bwd_workspace_bytes(2, 1000, 512, 16, "bf16", chunk_len_hint=128)
    assert ws1 >= 256 + 2 * 4 * 1000 * 32 * 4 + 2 * 512 * 16 * 4
    assert ws8 > ws1
    assert L.ssm_scan_bwd_workspace_bytes(2, 1000, 512, 8, "bf16") == 0


def test_flags_are_validated():
    assert ctypes.sizeof(L.ssm_dims) == 4 * 8 + 2 * 4 + 8 + 8 + 2 * 4   # flags took the spare slot
    d = L.make_dims(1, 20, 16, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 24,
                    flags=4)                                            # unknown bit
    scan = L.lib.ssm_selective_scan_fwd
    args = (FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, None, None, None, 0,
            FAKE + (1 << 30), None)
    assert scan(*args, ctypes.byref(d), None) == L.SSM_ERR_DIMS
    # the exact zero-order hold: dstate 16, tile configuration 0, no fused conv
    z8 = L.make_dims(1, 20, 16, 8, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 24,
                     flags=L.SSM_FLAG_ZOH)
    assert scan(*args, ctypes.byref(z8), None) == L.SSM_ERR_DIMS
    zt = L.make_dims(1, 20, 16, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 24,
                     flags=L.SSM_FLAG_ZOH, tile_config_hint=3)
    assert scan(*args, ctypes.byref(zt), None) == L.SSM_ERR_DIMS
    z16 = L.make_dims(1, 20, 16, 16, "bf16", workspace=FAKE + (1 << 34), workspace_bytes=1 << 24,
                      flags=L.SSM_FLAG_ZOH)
    # accepted up to the alias check (out over x), so no launch happens here
    bad = args[:9] + (FAKE, None)
    assert scan(*bad, ctypes.byref(z16), None) == L.SSM_ERR_ALIAS
    # the checkpointing forward takes the hold too: accepted up to the alias
    # check (its checkpoints over x), so no launch happens here
    assert L.lib.ssm_selective_scan_fwd_ckpt(*args[:9], None, FAKE + (1 << 30), None,
                                             FAKE, ctypes.byref(z16),
                                             None) == L.SSM_ERR_ALIAS
    assert L.lib.ssm_selective_scan_fwd_conv(FAKE, FAKE + (1 << 32), None, 4, *args[1:],
                                             ctypes.byref(z16), None) == L.SSM_ERR_DIMS
    # the backward takes the hold too: accepted up to the alias check (dx over
    # x), so no launch happens here
    G = FAKE + (1 << 36)
    assert L.lib.ssm_selective_scan_bwd(
        FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288, FAKE + 16384, None, None, None, 0,
        FAKE + (1 << 32), FAKE + 20480, None, FAKE, G + 4096, G + 65536, G + 8192, G + 12288,
        None, None, None, None, ctypes.byref(z16), None) == L.SSM_ERR_ALIAS


def test_bc_per_channel_flag_is_validated():
    F = L.SSM_FLAG_BC_PER_CHANNEL
    scan = L.lib.ssm_selective_scan_fwd

    def dims(**kw):
        base = dict(workspace=FAKE + (1 << 34), workspace_bytes=1 << 24, flags=F)
        base.update(kw)
        return L.make_dims(1, 20, 16, 16, "bf16", **base)

    # out over B, where B now spans batch * L * dim * N elements (20 * 16 * 16 * 2 bytes)
    args = (FAKE, FAKE + (1 << 20), FAKE + (2 << 20), FAKE + (3 << 20), FAKE + (4 << 20), None,
            None, None, 0)
    assert scan(*args, FAKE + (3 << 20) + 8192, None, ctypes.byref(dims()), None) == L.SSM_ERR_ALIAS
    assert scan(*args, FAKE + (3 << 20) + 10240 - 64, None, ctypes.byref(dims()),
                None) == L.SSM_ERR_ALIAS
    # with shared B (no flag) the same out lies past B's 640 bytes: accepted up to the next check
    d0 = dims(flags=0)
    assert scan(*args, FAKE + (3 << 20) + 8192, FAKE, ctypes.byref(d0), None) == L.SSM_ERR_ALIAS
    # dstate 16 only, tile configuration 0, not with the exact zero-order hold
    assert scan(*args, FAKE + (5 << 20), None,
                ctypes.byref(L.make_dims(1, 20, 16, 8, "bf16", flags=F)), None) == L.SSM_ERR_DIMS
    assert scan(*args, FAKE + (5 << 20), None, ctypes.byref(dims(tile_config_hint=2)),
                None) == L.SSM_ERR_DIMS
    assert scan(*args, FAKE + (5 << 20), None, ctypes.byref(dims(flags=F | L.SSM_FLAG_ZOH)),
                None) == L.SSM_ERR_DIMS
    # the training pair takes per-channel rows: the checkpointing forward is
    # accepted up to the alias check (its checkpoints over x), the backward too,
    # with dB 1024 bytes into B (inside B's per-channel 10240 bytes, past the
    # 640 of a shared row set); both variants at once are refused
    assert L.lib.ssm_selective_scan_fwd_ckpt(*args, None, FAKE + (5 << 20), None, FAKE,
                                             ctypes.byref(dims()), None) == L.SSM_ERR_ALIAS
    G = FAKE + (1 << 36)
    bwd = L.lib.ssm_selective_scan_bwd
    grads = lambda dB: (G, G + (1 << 20), G + (2 << 20), dB, G + (3 << 20), None, None, None,
                        None)
    assert bwd(*args, FAKE + (6 << 20), FAKE + (7 << 20), None, *grads(FAKE + (3 << 20) + 1024),
               ctypes.byref(dims()), None) == L.SSM_ERR_ALIAS
    assert bwd(*args, FAKE + (6 << 20), FAKE + (7 << 20), None, *grads(G + (4 << 20)),
               ctypes.byref(dims(flags=F | L.SSM_FLAG_ZOH)), None) == L.SSM_ERR_DIMS
    # the decode step takes per-channel rows too; B then spans [batch, dim, N]
    # (2 x 16 x 16 bf16 = 1024 bytes), so an output 640 bytes into it overlaps
    st = L.make_dims(2, 1, 16, 16, "bf16", flags=F)
    assert L.lib.ssm_state_update(FAKE + (6 << 20), FAKE, FAKE + 4096, FAKE + 8192, FAKE + 12288,
                                  FAKE + 16384, None, None, None, 0, FAKE + 12288 + 640,
                                  ctypes.byref(st), None) == L.SSM_ERR_ALIAS


def test_timeout_probe_rejects_bad_arguments_before_launch():
    f = L.lib.ssm_debug_timeout_probe
    assert f(None, 256, 1000, None) == L.SSM_ERR_NULL
    assert f(FAKE, 255, 1000, None) == L.SSM_ERR_WORKSPACE
    assert f(FAKE + 4, 256, 1000, None) == L.SSM_ERR_ALIGN
    assert f(FAKE, 256, 0, None) == L.SSM_ERR_DIMS
    assert f(FAKE, 256, (1 << 24) + 1, None) == L.SSM_ERR_DIMS


def test_plans_of_the_measured_workloads():
    """The planner's choices for the benchmark workloads are the ones measured
    fastest on the B300 (chunk counts swept; 16 chunks for b8 L4096 d2048 is
    within 1 % of the fastest measured, 8), planned here for 148 SMs (no
    device): a change to the plan model that moves them must be re-measured,
    not slip in."""
    p = L.ssm_scan_plan(4, 2048, 1536, 16, "bf16")
    assert (p["chunk_len"], p["nchunks"], p["ctas"], p["kernels"]) == (352, 6, 288, 2)
    p = L.ssm_scan_plan(8, 4096, 2048, 16, "bf16")
    assert p["nchunks"] == 16 and p["ctas"] == 2048 and p["kernels"] == 2
    p = L.ssm_scan_plan(1, 131072, 5120, 16, "bf16")
    assert p["nchunks"] == 37
    p = L.ssm_scan_plan(4, 2048, 1536, 16, "bf16", flags=L.SSM_FLAG_BC_PER_CHANNEL)
    assert (p["chunk_len"], p["nchunks"]) == (256, 8)
