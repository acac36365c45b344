"""Python binding of libssm (ctypes). Argument marshalling only.

Every step of the scan and of the decode step runs in the CUDA kernels of
``libssm.so``; PyTorch only supplies device memory, the current stream and
the output allocations. Importing this module fails loudly when the library
has not been built (``python -m selective_state_space_119_b300.build``); there
is no CPU fallback.

The functions carry the C names (``ssm_selective_scan_fwd``,
``ssm_state_update``, ``ssm_causal_conv1d_silu``, ``ssm_scan_workspace_bytes``,
``ssm_scan_plan``, ``ssm_get_device_status``, ``ssm_strerror``) and take torch
tensors. The raw
ctypes handle is ``lib`` for callers that hold plain device pointers.
"""
from __future__ import annotations

import contextlib
import ctypes
import os
from typing import Optional, Tuple

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "lib", "libssm.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libssm.so is not built (%s); run `python -m selective_state_space_119_b300.build`"
        % LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

SSM_F32, SSM_BF16 = 0, 1
SSM_OK = 0
SSM_ERR_NULL = -1
SSM_ERR_DIMS = -2
SSM_ERR_DTYPE = -3
SSM_ERR_ALIGN = -4
SSM_ERR_WORKSPACE = -5
SSM_ERR_CUDA = -6
SSM_ERR_TIMEOUT = -7
SSM_ERR_ALIAS = -8
SSM_FLAG_ZOH = 1      # exact zero-order-hold Bbar (include/ssm.h)
SSM_FLAG_BC_PER_CHANNEL = 2   # B, C of shape [batch, L, dim, N] (include/ssm.h)

# Every symbol include/ssm.h declares.
EXPORTED = ("ssm_selective_scan_fwd", "ssm_state_update", "ssm_scan_workspace_bytes",
            "ssm_scan_plan", "ssm_get_device_status", "ssm_strerror", "ssm_last_cuda_error",
            "ssm_version", "ssm_selective_scan_fwd_static", "ssm_selective_scan_fwd_from_state",
            "ssm_selective_scan_fwd_conv", "ssm_causal_conv1d_silu", "ssm_scan_checkpoint_bytes",
            "ssm_selective_scan_fwd_ckpt", "ssm_scan_bwd_workspace_bytes",
            "ssm_selective_scan_bwd", "ssm_debug_timeout_probe", "ssm_get_static_status",
            "ssm_debug_timeout_probe_static", "ssm_ssd_fwd", "ssm_ssd_workspace_bytes",
            "ssm_ssd_get_device_status", "ssm_causal_conv1d_silu_bwd",
            "ssm_causal_conv1d_silu_bwd_workspace_bytes")

# Size of the library-owned scratch of ssm_selective_scan_fwd_static (include/ssm.h).
SSM_STATIC_SCRATCH_BYTES = 16 << 20


class ssm_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("dim", ctypes.c_int64),
                ("dstate", ctypes.c_int64), ("io_dtype", ctypes.c_int32),
                ("chunk_len_hint", ctypes.c_int32), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t), ("tile_config_hint", ctypes.c_int32),
                ("flags", ctypes.c_int32)]


class ssm_plan(ctypes.Structure):
    _fields_ = [("chunk_len", ctypes.c_int64), ("nchunks", ctypes.c_int64),
                ("channels_per_cta", ctypes.c_int64), ("ctas", ctypes.c_int64),
                ("kernels", ctypes.c_int32), ("tile_config", ctypes.c_int32)]


class ssm_ssd_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int64), ("seqlen", ctypes.c_int64), ("nheads", ctypes.c_int64),
                ("headdim", ctypes.c_int64), ("ngroups", ctypes.c_int64), ("dstate", ctypes.c_int64),
                ("io_dtype", ctypes.c_int32), ("flags", ctypes.c_int32),
                ("workspace", ctypes.c_void_p), ("workspace_bytes", ctypes.c_size_t)]


_vp = ctypes.c_void_p
_dims_p = ctypes.POINTER(ssm_dims)
_ssd_p = ctypes.POINTER(ssm_ssd_dims)
lib.ssm_ssd_fwd.restype = ctypes.c_int
lib.ssm_ssd_fwd.argtypes = [_vp] * 7 + [ctypes.c_int] + [_vp] * 3 + [_ssd_p, _vp]
lib.ssm_ssd_workspace_bytes.restype = ctypes.c_size_t
lib.ssm_ssd_workspace_bytes.argtypes = [_ssd_p]
lib.ssm_ssd_get_device_status.restype = ctypes.c_int
lib.ssm_ssd_get_device_status.argtypes = [_ssd_p, _vp]
lib.ssm_selective_scan_fwd.restype = ctypes.c_int
lib.ssm_selective_scan_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                       _vp, _vp, _dims_p, _vp]
lib.ssm_selective_scan_fwd_from_state.restype = ctypes.c_int
lib.ssm_selective_scan_fwd_from_state.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                                  ctypes.c_int, _vp, _vp, _vp, _dims_p, _vp]
lib.ssm_selective_scan_fwd_conv.restype = ctypes.c_int
lib.ssm_selective_scan_fwd_conv.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp, _vp,
                                            _vp, _vp, ctypes.c_int, _vp, _vp, _dims_p, _vp]
lib.ssm_causal_conv1d_silu.restype = ctypes.c_int
lib.ssm_causal_conv1d_silu.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _dims_p, _vp]
lib.ssm_causal_conv1d_silu_bwd.restype = ctypes.c_int
lib.ssm_causal_conv1d_silu_bwd.argtypes = [_vp, _vp, _vp, ctypes.c_int, _vp, _vp, _vp, _vp,
                                           _dims_p, _vp]
lib.ssm_causal_conv1d_silu_bwd_workspace_bytes.restype = ctypes.c_size_t
lib.ssm_causal_conv1d_silu_bwd_workspace_bytes.argtypes = [_dims_p, ctypes.c_int]
lib.ssm_scan_checkpoint_bytes.restype = ctypes.c_size_t
lib.ssm_scan_checkpoint_bytes.argtypes = [_dims_p]
lib.ssm_selective_scan_fwd_ckpt.restype = ctypes.c_int
lib.ssm_selective_scan_fwd_ckpt.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                            _vp, _vp, _vp, _vp, _dims_p, _vp]
lib.ssm_scan_bwd_workspace_bytes.restype = ctypes.c_size_t
lib.ssm_scan_bwd_workspace_bytes.argtypes = [_dims_p]
lib.ssm_selective_scan_bwd.restype = ctypes.c_int
lib.ssm_selective_scan_bwd.argtypes = ([_vp] * 8 + [ctypes.c_int] + [_vp] * 12 +
                                       [_dims_p, _vp])
lib.ssm_selective_scan_fwd_static.restype = ctypes.c_int
lib.ssm_selective_scan_fwd_static.argtypes = list(lib.ssm_selective_scan_fwd.argtypes)
lib.ssm_state_update.restype = ctypes.c_int
lib.ssm_state_update.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, ctypes.c_int,
                                 _vp, _dims_p, _vp]
lib.ssm_scan_workspace_bytes.restype = ctypes.c_size_t
lib.ssm_scan_workspace_bytes.argtypes = [_dims_p]
lib.ssm_scan_plan.restype = ctypes.c_int
lib.ssm_scan_plan.argtypes = [_dims_p, ctypes.POINTER(ssm_plan)]
lib.ssm_debug_timeout_probe.restype = ctypes.c_int
lib.ssm_debug_timeout_probe.argtypes = [_vp, ctypes.c_size_t, ctypes.c_uint32, _vp]
lib.ssm_debug_timeout_probe_static.restype = ctypes.c_int
lib.ssm_debug_timeout_probe_static.argtypes = [ctypes.c_uint32, _vp]
lib.ssm_get_static_status.restype = ctypes.c_int
lib.ssm_get_static_status.argtypes = [_vp]
lib.ssm_get_device_status.restype = ctypes.c_int
lib.ssm_get_device_status.argtypes = [_dims_p, _vp]
lib.ssm_strerror.restype = ctypes.c_char_p
lib.ssm_strerror.argtypes = [ctypes.c_int]
lib.ssm_last_cuda_error.restype = ctypes.c_int
lib.ssm_last_cuda_error.argtypes = []
lib.ssm_version.restype = ctypes.c_int
lib.ssm_version.argtypes = []


class SSMError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        msg = "%s: %s (%d)" % (where, ssm_strerror(code), code)
        if code == SSM_ERR_CUDA:
            msg += ", cudaError %d" % lib.ssm_last_cuda_error()
        super().__init__(msg)


def ssm_strerror(code: int) -> str:
    return lib.ssm_strerror(int(code)).decode()


def _check(rc: int, where: str) -> None:
    if rc != SSM_OK:
        raise SSMError(rc, where)


def make_dims(batch, seqlen, dim, dstate, io, workspace=None, workspace_bytes=0,
              chunk_len_hint=0, tile_config_hint=0, flags=0) -> ssm_dims:
    io_code = io if isinstance(io, int) else (SSM_BF16 if str(io) in ("bf16", "torch.bfloat16") else SSM_F32)
    return ssm_dims(int(batch), int(seqlen), int(dim), int(dstate), io_code, int(chunk_len_hint),
                    workspace, int(workspace_bytes), int(tile_config_hint), int(flags))


def ssm_scan_workspace_bytes(batch, seqlen, dim, dstate, io, chunk_len_hint=0,
                             tile_config_hint=0, flags=0) -> int:
    d = make_dims(batch, seqlen, dim, dstate, io, chunk_len_hint=chunk_len_hint,
                  tile_config_hint=tile_config_hint, flags=flags)
    return int(lib.ssm_scan_workspace_bytes(ctypes.byref(d)))


def ssm_scan_plan(batch, seqlen, dim, dstate, io, chunk_len_hint=0, tile_config_hint=0,
                  flags=0) -> dict:
    d = make_dims(batch, seqlen, dim, dstate, io, chunk_len_hint=chunk_len_hint,
                  tile_config_hint=tile_config_hint, flags=flags)
    p = ssm_plan()
    _check(lib.ssm_scan_plan(ctypes.byref(d), ctypes.byref(p)), "ssm_scan_plan")
    return {k: getattr(p, k) for k, _ in ssm_plan._fields_}


# ---------------------------------------------------------------------------
# torch front end
# ---------------------------------------------------------------------------
def _torch():
    import torch
    return torch


def _io_code(t) -> int:
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return SSM_BF16
    if t.dtype == torch.float32:
        return SSM_F32
    raise TypeError("I/O tensors must be float32 or bfloat16, got %s" % t.dtype)


def _ptr(t, name, dtype=None, shape=None, device=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, expected %s" % (name, t.device, device))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)
    if dtype is not None and t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))
    return t.data_ptr()


def _device_of(t, name):
    """The CUDA device of t; host tensors are refused (there is no CPU path)."""
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    return t.device


@contextlib.contextmanager
def _launch_on(device, stream):
    """Device and stream of one call, yielding the stream handle for the C call.
    The wrapper allocates its outputs and per-call workspace (and zero-fills the
    workspace) inside this context, on the stream the kernels are enqueued on,
    so the kernels run after the fill and the caching allocator does not hand
    that memory to other work before they finish."""
    torch = _torch()
    with torch.cuda.device(device):
        s = stream if stream is not None else torch.cuda.current_stream(device)
        with torch.cuda.stream(s):
            yield ctypes.c_void_p(s.cuda_stream)


def alloc_workspace(batch, seqlen, dim, dstate, io, device, chunk_len_hint=0, tile_config_hint=0,
                    flags=0):
    """Zero-filled workspace tensor (uint8) of the size the scan needs, or None."""
    torch = _torch()
    n = ssm_scan_workspace_bytes(batch, seqlen, dim, dstate, io, chunk_len_hint, tile_config_hint,
                                 flags)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device)


def ssm_selective_scan_fwd(x, delta, A, B, C, D=None, z=None, delta_bias=None,
                           delta_softplus=False, out=None, final_state=None,
                           return_final_state=True, workspace=None, chunk_len_hint=0,
                           tile_config_hint=0, stream=None, h0=None, conv_w=None,
                           conv_b=None, zoh=False) -> Tuple[object, Optional[object]]:
    """Selective scan over x [batch, L, dim] (see include/ssm.h).

    Returns (out, final_state); final_state is None when not requested.
    ``out`` / ``final_state`` may be passed preallocated; ``workspace`` is a
    zero-initialised uint8 CUDA tensor of at least ssm_scan_workspace_bytes
    (allocated per call when omitted). ``h0`` ([batch, dim, N] fp32), when
    given, is the state before the first token
    (ssm_selective_scan_fwd_from_state); otherwise the scan starts from zero.
    ``conv_w`` ([dim, K] fp32, K <= 4) and ``conv_b`` ([dim] fp32 or None)
    put the causal conv1d + SiLU input stage in front of the scan
    (ssm_selective_scan_fwd_conv): x is then the conv's input. ``zoh=True``
    takes the exact zero-order-hold Bbar (SSM_FLAG_ZOH). B and C of shape
    [batch, L, dim, N] select per-channel rows (SSM_FLAG_BC_PER_CHANNEL).
    """
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    if conv_w is not None and h0 is not None:
        raise ValueError("the fused conv input stage starts from h = 0; h0 is not supported")
    if conv_w is None and conv_b is not None:
        raise ValueError("conv_b needs conv_w")
    bcd = B.dim() == 4          # per-channel B, C: [batch, L, dim, N]
    bc_shape = (batch, L, dim, N) if bcd else (batch, L, N)
    flags = (SSM_FLAG_ZOH if zoh else 0) | (SSM_FLAG_BC_PER_CHANNEL if bcd else 0)
    with _launch_on(dev, stream) as sp:
        if out is None:
            out = torch.empty_like(x)
        if final_state is None and return_final_state:
            final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = alloc_workspace(batch, L, dim, N, _io_code(x), dev, chunk_len_hint,
                                        tile_config_hint, flags)
        rc, where = _scan_fwd_call(x, delta, A, B, C, D, z, delta_bias, delta_softplus, out,
                                   final_state, workspace, chunk_len_hint, tile_config_hint,
                                   h0, conv_w, conv_b, flags, bc_shape, sp)
    _check(rc, where)
    return out, final_state


def _scan_fwd_call(x, delta, A, B, C, D, z, delta_bias, delta_softplus, out, final_state,
                   workspace, chunk_len_hint, tile_config_hint, h0, conv_w, conv_b, flags,
                   bc_shape, sp):
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    ws_ptr = _ptr(workspace, "workspace", torch.uint8, device=dev)
    ws_bytes = workspace.numel() if workspace is not None else 0
    dims = make_dims(batch, L, dim, N, _io_code(x), ws_ptr, ws_bytes, chunk_len_hint,
                     tile_config_hint, flags)
    args = (
        _ptr(x, "x", io, (batch, L, dim), dev),
        _ptr(delta, "delta", io, (batch, L, dim), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", io, bc_shape, dev),
        _ptr(C, "C", io, bc_shape, dev),
        _ptr(D, "D", torch.float32, (dim,), dev),
        _ptr(z, "z", io, (batch, L, dim), dev),
        _ptr(delta_bias, "delta_bias", torch.float32, (dim,), dev),
        1 if delta_softplus else 0,
        _ptr(out, "out", io, (batch, L, dim), dev),
        _ptr(final_state, "final_state", torch.float32, (batch, dim, N), dev),
    )
    if conv_w is not None:
        if conv_w.dim() != 2 or conv_w.shape[0] != dim:
            raise ValueError("conv_w must have shape (dim, K), got %s" % (tuple(conv_w.shape),))
        K = int(conv_w.shape[1])
        wp = _ptr(conv_w, "conv_w", torch.float32, (dim, K), dev)
        bp = _ptr(conv_b, "conv_b", torch.float32, (dim,), dev)
        return (lib.ssm_selective_scan_fwd_conv(args[0], wp, bp, K, *args[1:],
                                                ctypes.byref(dims), sp),
                "ssm_selective_scan_fwd_conv")
    if h0 is None:
        return lib.ssm_selective_scan_fwd(*args, ctypes.byref(dims), sp), "ssm_selective_scan_fwd"
    h0p = _ptr(h0, "h0", torch.float32, (batch, dim, N), dev)
    return (lib.ssm_selective_scan_fwd_from_state(*args[:9], h0p, *args[9:], ctypes.byref(dims),
                                                  sp),
            "ssm_selective_scan_fwd_from_state")


def ssm_causal_conv1d_silu(x, conv_w, conv_b=None, out=None, stream=None):
    """u = silu(causal depthwise conv1d(x)) over x [batch, L, dim] with taps
    conv_w [dim, K] fp32 (K <= 4) and bias conv_b [dim] fp32 or None. Returns u
    (same shape and dtype as x; ``out`` may be passed preallocated)."""
    torch = _torch()
    batch, L, dim = x.shape
    dev = _device_of(x, "x")
    if conv_w.dim() != 2 or conv_w.shape[0] != dim:
        raise ValueError("conv_w must have shape (dim, K), got %s" % (tuple(conv_w.shape),))
    K = int(conv_w.shape[1])
    dims = make_dims(batch, L, dim, 16, _io_code(x))
    with _launch_on(dev, stream) as sp:
        if out is None:
            out = torch.empty_like(x)
        rc = lib.ssm_causal_conv1d_silu(
            _ptr(x, "x", x.dtype, (batch, L, dim), dev),
            _ptr(conv_w, "conv_w", torch.float32, (dim, K), dev),
            _ptr(conv_b, "conv_b", torch.float32, (dim,), dev), K,
            _ptr(out, "out", x.dtype, (batch, L, dim), dev),
            ctypes.byref(dims), sp)
    _check(rc, "ssm_causal_conv1d_silu")
    return out


def ssm_causal_conv1d_silu_bwd(x, conv_w, du, conv_b=None, want_dbias=True, stream=None):
    """Gradients of the input stage for dLoss/du = du (include/ssm.h): returns
    (dx [batch, L, dim] like x, dconv_w [dim, K] fp32, dconv_b [dim] fp32 or
    None)."""
    torch = _torch()
    batch, L, dim = x.shape
    dev = _device_of(x, "x")
    if conv_w.dim() != 2 or conv_w.shape[0] != dim:
        raise ValueError("conv_w must have shape (dim, K), got %s" % (tuple(conv_w.shape),))
    K = int(conv_w.shape[1])
    dims = make_dims(batch, L, dim, 16, _io_code(x))
    n = int(lib.ssm_causal_conv1d_silu_bwd_workspace_bytes(ctypes.byref(dims), K))
    with _launch_on(dev, stream) as sp:
        dx = torch.empty_like(x)
        dw = torch.empty((dim, K), dtype=torch.float32, device=dev)
        db = torch.empty((dim,), dtype=torch.float32, device=dev) if want_dbias else None
        ws = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
        dims = make_dims(batch, L, dim, 16, _io_code(x), ws.data_ptr(), n)
        rc = lib.ssm_causal_conv1d_silu_bwd(
            _ptr(x, "x", x.dtype, (batch, L, dim), dev),
            _ptr(conv_w, "conv_w", torch.float32, (dim, K), dev),
            _ptr(conv_b, "conv_b", torch.float32, (dim,), dev), K,
            _ptr(du, "du", x.dtype, (batch, L, dim), dev), _ptr(dx, "dx", x.dtype, None, dev),
            _ptr(dw, "dconv_w", torch.float32, None, dev),
            _ptr(db, "dconv_b", torch.float32, None, dev), ctypes.byref(dims), sp)
    _check(rc, "ssm_causal_conv1d_silu_bwd")
    return dx, dw, db


def ssm_selective_scan_fwd_static(x, delta, A, B, C, D=None, z=None, delta_bias=None,
                                  delta_softplus=False, out=None, final_state=None,
                                  return_final_state=True, chunk_len_hint=0,
                                  tile_config_hint=0, stream=None):
    """ssm_selective_scan_fwd without a workspace: the scan's scratch is the
    library's own fixed array (include/ssm.h), for callers that cannot allocate.
    Calls that overlap on the GPU share that array and must be serialized."""
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    with _launch_on(dev, stream) as sp:
        if out is None:
            out = torch.empty_like(x)
        if final_state is None and return_final_state:
            final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
        rc = _static_call(x, delta, A, B, C, D, z, delta_bias, delta_softplus, out, final_state,
                          chunk_len_hint, tile_config_hint, sp)
    _check(rc, "ssm_selective_scan_fwd_static")
    return out, final_state


def _static_call(x, delta, A, B, C, D, z, delta_bias, delta_softplus, out, final_state,
                 chunk_len_hint, tile_config_hint, sp):
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    dims = make_dims(batch, L, dim, N, _io_code(x), None, 0, chunk_len_hint, tile_config_hint)
    args = (
        _ptr(x, "x", io, (batch, L, dim), dev),
        _ptr(delta, "delta", io, (batch, L, dim), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", io, (batch, L, N), dev),
        _ptr(C, "C", io, (batch, L, N), dev),
        _ptr(D, "D", torch.float32, (dim,), dev),
        _ptr(z, "z", io, (batch, L, dim), dev),
        _ptr(delta_bias, "delta_bias", torch.float32, (dim,), dev),
        1 if delta_softplus else 0,
        _ptr(out, "out", io, (batch, L, dim), dev),
        _ptr(final_state, "final_state", torch.float32, (batch, dim, N), dev),
    )
    return lib.ssm_selective_scan_fwd_static(*args, ctypes.byref(dims), sp)


def ssm_state_update(state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                     delta_softplus=False, out=None, stream=None, zoh=False):
    """One recurrent step; ``state`` [batch, dim, N] fp32 is updated in place.
    x, delta, z: [batch, dim]; B, C: [batch, N], or [batch, dim, N] (one row
    per channel: SSM_FLAG_BC_PER_CHANNEL). Returns out [batch, dim].
    ``zoh=True`` takes the exact zero-order-hold Bbar."""
    torch = _torch()
    batch, dim, N = state.shape
    io = x.dtype
    dev = _device_of(state, "state")
    if out is None:
        with _launch_on(dev, stream):
            out = torch.empty_like(x)
    bcd = B.dim() == 3
    flags = (SSM_FLAG_ZOH if zoh else 0) | (SSM_FLAG_BC_PER_CHANNEL if bcd else 0)
    rows = (batch, dim, N) if bcd else (batch, N)
    dims = make_dims(batch, 1, dim, N, _io_code(x), flags=flags)
    args = (
        _ptr(state, "state", torch.float32, (batch, dim, N), dev),
        _ptr(x, "x", io, (batch, dim), dev),
        _ptr(delta, "delta", io, (batch, dim), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev),
        _ptr(B, "B", io, rows, dev),
        _ptr(C, "C", io, rows, dev),
        _ptr(D, "D", torch.float32, (dim,), dev),
        _ptr(z, "z", io, (batch, dim), dev),
        _ptr(delta_bias, "delta_bias", torch.float32, (dim,), dev),
        1 if delta_softplus else 0,
        _ptr(out, "out", io, (batch, dim), dev),
    )
    with _launch_on(dev, stream) as sp:
        rc = lib.ssm_state_update(*args, ctypes.byref(dims), sp)
    _check(rc, "ssm_state_update")
    return out


def ssm_get_device_status(batch, seqlen, dim, dstate, io, workspace, chunk_len_hint=0,
                          stream=None, tile_config_hint=0) -> int:
    """Synchronize the stream and return the workspace's device status code."""
    torch = _torch()
    ws_ptr = workspace.data_ptr() if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    dims = make_dims(batch, seqlen, dim, dstate, io, ws_ptr, ws_bytes, chunk_len_hint,
                     tile_config_hint)
    dev = _device_of(workspace, "workspace") if workspace is not None else torch.device("cuda")
    with _launch_on(dev, stream) as sp:
        return int(lib.ssm_get_device_status(ctypes.byref(dims), sp))


def ssm_scan_checkpoint_bytes(batch, seqlen, dim, dstate, io) -> int:
    d = make_dims(batch, seqlen, dim, dstate, io)
    return int(lib.ssm_scan_checkpoint_bytes(ctypes.byref(d)))


def ssm_scan_bwd_workspace_bytes(batch, seqlen, dim, dstate, io, chunk_len_hint=0,
                                 tile_config_hint=0, flags=0) -> int:
    d = make_dims(batch, seqlen, dim, dstate, io, chunk_len_hint=chunk_len_hint,
                  tile_config_hint=tile_config_hint, flags=flags)
    return int(lib.ssm_scan_bwd_workspace_bytes(ctypes.byref(d)))


def ssm_selective_scan_fwd_ckpt(x, delta, A, B, C, D=None, z=None, delta_bias=None,
                                delta_softplus=False, h0=None, out=None, final_state=None,
                                ckpt=None, workspace=None, chunk_len_hint=0, stream=None,
                                zoh=False):
    """The scan that also saves the state before every 8th token for the
    backward. Returns (out, final_state, ckpt); ckpt is [batch, ceil(L/8), dim,
    16] fp32. ``zoh=True`` scans with the exact zero-order-hold Bbar; B and C of
    shape [batch, L, dim, 16] select per-channel rows."""
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    bcd = B.dim() == 4
    bc_shape = (batch, L, dim, N) if bcd else (batch, L, N)
    flags = (SSM_FLAG_ZOH if zoh else 0) | (SSM_FLAG_BC_PER_CHANNEL if bcd else 0)
    with _launch_on(dev, stream) as sp:
        if out is None:
            out = torch.empty_like(x)
        if final_state is None:
            final_state = torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
        if ckpt is None:
            ckpt = torch.empty((batch, (L + 7) // 8, dim, N), dtype=torch.float32, device=dev)
        if workspace is None:
            workspace = alloc_workspace(batch, L, dim, N, _io_code(x), dev, chunk_len_hint,
                                        flags=flags)
        ws_ptr = _ptr(workspace, "workspace", torch.uint8, device=dev)
        ws_bytes = workspace.numel() if workspace is not None else 0
        dims = make_dims(batch, L, dim, N, _io_code(x), ws_ptr, ws_bytes, chunk_len_hint,
                         flags=flags)
        rc = lib.ssm_selective_scan_fwd_ckpt(
            _ptr(x, "x", io, (batch, L, dim), dev), _ptr(delta, "delta", io, (batch, L, dim), dev),
            _ptr(A, "A", torch.float32, (dim, N), dev), _ptr(B, "B", io, bc_shape, dev),
            _ptr(C, "C", io, bc_shape, dev), _ptr(D, "D", torch.float32, (dim,), dev),
            _ptr(z, "z", io, (batch, L, dim), dev),
            _ptr(delta_bias, "delta_bias", torch.float32, (dim,), dev),
            1 if delta_softplus else 0, _ptr(h0, "h0", torch.float32, (batch, dim, N), dev),
            _ptr(out, "out", io, (batch, L, dim), dev),
            _ptr(final_state, "final_state", torch.float32, (batch, dim, N), dev),
            _ptr(ckpt, "ckpt", torch.float32, (batch, (L + 7) // 8, dim, N), dev),
            ctypes.byref(dims), sp)
    _check(rc, "ssm_selective_scan_fwd_ckpt")
    return out, final_state, ckpt


def ssm_selective_scan_bwd(x, delta, A, B, C, ckpt, dout, D=None, z=None, delta_bias=None,
                           delta_softplus=False, dfinal_state=None, want_dD=True,
                           want_ddelta_bias=True, want_dh0=False, workspace=None,
                           chunk_len_hint=0, stream=None, zoh=False) -> dict:
    """Gradients of the scan (include/ssm.h). Returns a dict with dx, ddelta,
    dA, dB, dC and, when asked for / defined, dD, dz, ddelta_bias, dh0.
    ``zoh=True`` differentiates the exact zero-order-hold scan (the checkpoints
    must come from a ``zoh=True`` checkpointing forward). B and C of shape
    [batch, L, dim, 16] differentiate the per-channel scan (dB, dC then have
    that shape too)."""
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    with _launch_on(dev, stream) as sp:
        rc, g = _bwd_call(x, delta, A, B, C, ckpt, dout, D, z, delta_bias, delta_softplus,
                          dfinal_state, want_dD, want_ddelta_bias, want_dh0, workspace,
                          chunk_len_hint, sp, zoh)
    _check(rc, "ssm_selective_scan_bwd")
    return g


def _bwd_call(x, delta, A, B, C, ckpt, dout, D, z, delta_bias, delta_softplus, dfinal_state,
              want_dD, want_ddelta_bias, want_dh0, workspace, chunk_len_hint, sp, zoh=False):
    torch = _torch()
    batch, L, dim = x.shape
    N = A.shape[1]
    io = x.dtype
    dev = _device_of(x, "x")
    bcd = B.dim() == 4
    bc_shape = (batch, L, dim, N) if bcd else (batch, L, N)
    flags = (SSM_FLAG_ZOH if zoh else 0) | (SSM_FLAG_BC_PER_CHANNEL if bcd else 0)
    g = {"dx": torch.empty_like(x), "ddelta": torch.empty_like(x),
         "dA": torch.empty((dim, N), dtype=torch.float32, device=dev),
         "dB": torch.empty(bc_shape, dtype=io, device=dev),
         "dC": torch.empty(bc_shape, dtype=io, device=dev),
         "dD": torch.empty(dim, dtype=torch.float32, device=dev) if want_dD else None,
         "dz": torch.empty_like(x) if z is not None else None,
         "ddelta_bias": (torch.empty(dim, dtype=torch.float32, device=dev)
                         if want_ddelta_bias else None),
         "dh0": (torch.empty((batch, dim, N), dtype=torch.float32, device=dev)
                 if want_dh0 else None)}
    if workspace is None:
        n = ssm_scan_bwd_workspace_bytes(batch, L, dim, N, _io_code(x), chunk_len_hint,
                                         flags=flags)
        workspace = torch.empty(max(n, 1), dtype=torch.uint8, device=dev)
    dims = make_dims(batch, L, dim, N, _io_code(x), _ptr(workspace, "workspace", torch.uint8,
                                                         device=dev),
                     workspace.numel(), chunk_len_hint, flags=flags)
    rc = lib.ssm_selective_scan_bwd(
        _ptr(x, "x", io, (batch, L, dim), dev), _ptr(delta, "delta", io, (batch, L, dim), dev),
        _ptr(A, "A", torch.float32, (dim, N), dev), _ptr(B, "B", io, bc_shape, dev),
        _ptr(C, "C", io, bc_shape, dev), _ptr(D, "D", torch.float32, (dim,), dev),
        _ptr(z, "z", io, (batch, L, dim), dev),
        _ptr(delta_bias, "delta_bias", torch.float32, (dim,), dev),
        1 if delta_softplus else 0,
        _ptr(ckpt, "ckpt", torch.float32, (batch, (L + 7) // 8, dim, N), dev),
        _ptr(dout, "dout", io, (batch, L, dim), dev),
        _ptr(dfinal_state, "dfinal_state", torch.float32, (batch, dim, N), dev),
        _ptr(g["dx"], "dx"), _ptr(g["ddelta"], "ddelta"), _ptr(g["dA"], "dA"),
        _ptr(g["dB"], "dB"), _ptr(g["dC"], "dC"), _ptr(g["dD"], "dD"), _ptr(g["dz"], "dz"),
        _ptr(g["ddelta_bias"], "ddelta_bias"), _ptr(g["dh0"], "dh0"),
        ctypes.byref(dims), sp)
    return rc, g


# Short aliases.
selective_scan_fwd = ssm_selective_scan_fwd
state_update = ssm_state_update
causal_conv1d_silu = ssm_causal_conv1d_silu


# ---------------------------------------------------------------------------
# Mamba-2 SSD
# ---------------------------------------------------------------------------
def make_ssd_dims(batch, seqlen, nheads, headdim, ngroups, dstate, workspace=None,
                  workspace_bytes=0) -> ssm_ssd_dims:
    return ssm_ssd_dims(int(batch), int(seqlen), int(nheads), int(headdim), int(ngroups),
                        int(dstate), SSM_BF16, 0, workspace, int(workspace_bytes))


def ssm_ssd_fwd(x, dt, A, B, C, D=None, dt_bias=None, dt_softplus=False, h0=None, y=None,
                final_state=None, return_final_state=True, workspace=None, stream=None):
    """Mamba-2's SSD layer (see include/ssm.h): x [batch, L, H, 64] bf16, dt
    [batch, L, H] bf16, A, D, dt_bias [H] fp32, B, C [batch, L, G, 128] bf16,
    h0 [batch, H, 64, 128] fp32 or None. Returns (y, final_state or None)."""
    torch = _torch()
    device = _device_of(x, "x")
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    with _launch_on(device, stream) as sp:
        if y is None:
            y = torch.empty_like(x)
        if final_state is None and return_final_state:
            final_state = torch.empty((batch, H, P, N), dtype=torch.float32, device=device)
        if workspace is None:
            workspace = torch.zeros(256, dtype=torch.uint8, device=device)
        dims = make_ssd_dims(batch, L, H, P, G, N, workspace.data_ptr(), workspace.numel())
        bf, f32 = torch.bfloat16, torch.float32
        rc = lib.ssm_ssd_fwd(
            _ptr(x, "x", bf, device=device), _ptr(dt, "dt", bf, (batch, L, H), device),
            _ptr(A, "A", f32, (H,), device), _ptr(B, "B", bf, (batch, L, G, N), device),
            _ptr(C, "C", bf, (batch, L, G, N), device), _ptr(D, "D", f32, (H,), device),
            _ptr(dt_bias, "dt_bias", f32, (H,), device), 1 if dt_softplus else 0,
            _ptr(h0, "h0", f32, (batch, H, P, N), device), _ptr(y, "y", bf, x.shape, device),
            _ptr(final_state, "final_state", f32, (batch, H, P, N), device),
            ctypes.byref(dims), sp)
    _check(rc, "ssm_ssd_fwd")
    return y, final_state


def ssm_ssd_get_device_status(batch, seqlen, nheads, ngroups, workspace, stream=None) -> int:
    torch = _torch()
    dims = make_ssd_dims(batch, seqlen, nheads, 64, ngroups, 128, workspace.data_ptr(),
                         workspace.numel())
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    return int(lib.ssm_ssd_get_device_status(ctypes.byref(dims), ctypes.c_void_p(s.cuda_stream)))
