"""float64 CPU oracle for the selective state space scan (S6).

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The CUDA library and
its Python binding never import it, and it imports nothing from them.

The arithmetic lives in ``ssm_oracle.c`` (plain float64 C, compiled with gcc
``-O2`` and no fast-math). This module only compiles it, marshals numpy
float64 arrays through ctypes, and returns numpy arrays. It adds no arithmetic
of its own.

What it computes (page title, section):
  * "State Space Models -- Mamba, S4, and Beyond", "Mamba (S6 -- Selective
    State Space)", ``_selective_scan``: dA = exp(delta*A), dB = delta*B, the
    sequential loop h = dA*h + dB*u, y = C.h, plus D*u.
  * "Mamba: State Space Models Challenge Transformers", "Selective Scan
    Algorithm" and "Mamba's Innovation: Selection": A of shape [D, N],
    delta = softplus(delta), gate y * silu(z).
  * "State-space models (Mamba, S4)", "Training vs Inference Modes": the
    O(1)-per-token recurrent step on a cached state, and training through the
    scan (its gradients: ``selective_scan_bwd``).
  * The variants: the exact zero-order hold (``zoh=True``; "State-space models
    (Mamba, S4)", "From Continuous to Discrete: The Key Step"), per-channel B, C
    (``selective_scan_bcd``, ``state_update_bcd``; the docstring shapes of
    "Mamba: State Space Models Challenge Transformers", "Selective Scan
    Algorithm") and their gradients (``selective_scan_bwd(zoh=True)``,
    ``selective_scan_bcd_bwd``).
  * The block's input stage, causal conv1d + SiLU, and its gradient
    (``causal_conv1d_silu``, ``causal_conv1d_silu_bwd``, chained onto the scan by
    ``selective_scan_conv_bwd``).
  * Mamba-2's SSD layer (``ssd``; "Mamba: State Space Models Challenge
    Transformers", "Mamba-2: Improved Architecture", and "State Space Models and
    Mamba", "Mamba 2 and Hybrid Architectures").
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ssm_oracle.c")
_LIB_PATH = os.path.join(_HERE, "libssm_oracle.so")
_lock = threading.Lock()
_default = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def compile_source(src: str, out_path: str) -> str:
    """Compile an oracle C source into a shared library with gcc (no fast-math,
    no FMA contraction)."""
    tmp = out_path + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
           "-ffp-contract=off", "-pthread", src, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out_path)
    return out_path


def build(force: bool = False) -> str:
    """Compile ssm_oracle.c into oracle/libssm_oracle.so (only when stale)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    return compile_source(_SRC, _LIB_PATH)


def _bind(lib):
    lib.oracle_softplus.restype = ctypes.c_double
    lib.oracle_softplus.argtypes = [ctypes.c_double]
    lib.oracle_silu.restype = ctypes.c_double
    lib.oracle_silu.argtypes = [ctypes.c_double]
    lib.oracle_recurrence.restype = None
    lib.oracle_recurrence.argtypes = [_i64, _i64, _dp, _dp, _dp, _dp, _dp, _dp]
    for name in ("oracle_selective_scan", "oracle_selective_scan_zoh"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = (
            [_i64] * 4 + [_dp] * 8 + [ctypes.c_int] + [_dp] * 3 + [ctypes.c_int])
    for name in ("oracle_state_update", "oracle_state_update_zoh"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = [_i64] * 3 + [_dp] * 9 + [ctypes.c_int] + [_dp]
    for name in ("oracle_phi", "oracle_phi_prime"):
        getattr(lib, name).restype = ctypes.c_double
        getattr(lib, name).argtypes = [ctypes.c_double]
    lib.oracle_causal_conv1d_silu.restype = None
    lib.oracle_causal_conv1d_silu.argtypes = [_i64] * 4 + [_dp] * 4
    lib.oracle_ssd.restype = ctypes.c_int
    lib.oracle_ssd.argtypes = [_i64] * 6 + [_dp] * 7 + [ctypes.c_int] + [_dp] * 3 + [ctypes.c_int]
    lib.oracle_causal_conv1d_silu_bwd.restype = None
    lib.oracle_causal_conv1d_silu_bwd.argtypes = [_i64] * 4 + [_dp] * 7
    for name in ("oracle_selective_scan_bwd", "oracle_selective_scan_bwd_zoh"):
        getattr(lib, name).restype = ctypes.c_int
        getattr(lib, name).argtypes = (
            [_i64] * 4 + [_dp] * 8 + [ctypes.c_int] + [_dp] * 12 + [ctypes.c_int])
    return lib


def _f64(a, shape=None):
    """Contiguous float64 copy (or view) of a, checked against shape."""
    if a is None:
        return None
    arr = np.ascontiguousarray(np.asarray(a, dtype=np.float64))
    if shape is not None and tuple(arr.shape) != tuple(shape):
        raise ValueError("expected shape %s, got %s" % (tuple(shape), arr.shape))
    return arr


def _ptr(a):
    return None if a is None else a.ctypes.data_as(_dp)


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


class Oracle:
    """ctypes front end of one compiled oracle library."""

    def __init__(self, lib_path: str):
        self.path = lib_path
        self._lib = _bind(ctypes.CDLL(lib_path))

    def softplus(self, v: float) -> float:
        return self._lib.oracle_softplus(float(v))

    def silu(self, z: float) -> float:
        return self._lib.oracle_silu(float(z))

    def recurrence(self, Abar, Bbar, C, x, h0):
        """Discretized recurrence for one channel.

        Abar, Bbar, C: [L, N]; x: [L]; h0: [N]. Returns (y [L], h_L [N]).
        """
        Abar = _f64(Abar)
        L, N = Abar.shape
        Bbar, C = _f64(Bbar, (L, N)), _f64(C, (L, N))
        x, h = _f64(x, (L,)), _f64(h0, (N,)).copy()
        y = np.zeros(L, dtype=np.float64)
        self._lib.oracle_recurrence(L, N, _ptr(Abar), _ptr(Bbar), _ptr(C), _ptr(x), _ptr(h), _ptr(y))
        return y, h

    def phi(self, z: float) -> float:
        return self._lib.oracle_phi(float(z))

    def phi_prime(self, z: float) -> float:
        return self._lib.oracle_phi_prime(float(z))

    def selective_scan(self, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                       delta_softplus=False, h0=None, nthreads=None, zoh=False):
        """Selective scan over [batch, L, dim] with a [dim, N] diagonal A;
        zoh=True takes the exact zero-order-hold Bbar = dt * phi(dt A) * B.

        Returns (out [batch, L, dim], final_state [batch, dim, N]), both float64.
        """
        x = _f64(x)
        batch, L, dim = x.shape
        A = _f64(A)
        N = A.shape[1]
        delta = _f64(delta, (batch, L, dim))
        A = _f64(A, (dim, N))
        B, C = _f64(B, (batch, L, N)), _f64(C, (batch, L, N))
        D = _f64(D, (dim,))
        z = _f64(z, (batch, L, dim))
        delta_bias = _f64(delta_bias, (dim,))
        h0 = _f64(h0, (batch, dim, N))
        out = np.zeros((batch, L, dim), dtype=np.float64)
        fs = np.zeros((batch, dim, N), dtype=np.float64)
        fn = self._lib.oracle_selective_scan_zoh if zoh else self._lib.oracle_selective_scan
        rc = fn(
            batch, L, dim, N, _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(out),
            _ptr(fs), int(nthreads or default_threads()))
        if rc != 0:
            raise RuntimeError("oracle_selective_scan failed (%d)" % rc)
        return out, fs

    def state_update(self, state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                     delta_softplus=False, zoh=False):
        """One recurrent step. state: [batch, dim, N] (not modified; a new array is
        returned). x, delta, z: [batch, dim]; B, C: [batch, N].

        Returns (out [batch, dim], new_state [batch, dim, N]).
        """
        st = _f64(state).copy()
        batch, dim, N = st.shape
        x, delta = _f64(x, (batch, dim)), _f64(delta, (batch, dim))
        A = _f64(A, (dim, N))
        B, C = _f64(B, (batch, N)), _f64(C, (batch, N))
        D, z = _f64(D, (dim,)), _f64(z, (batch, dim))
        delta_bias = _f64(delta_bias, (dim,))
        out = np.zeros((batch, dim), dtype=np.float64)
        fn = self._lib.oracle_state_update_zoh if zoh else self._lib.oracle_state_update
        rc = fn(
            batch, dim, N, _ptr(st), _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D),
            _ptr(z), _ptr(delta_bias), int(bool(delta_softplus)), _ptr(out))
        if rc != 0:
            raise RuntimeError("oracle_state_update failed (%d)" % rc)
        return out, st


def _conv_method(self, x, w, bias=None):
    """Causal depthwise conv1d + SiLU. x: [batch, L, dim]; w: [dim, K];
    bias: [dim] or None. Returns u [batch, L, dim] float64."""
    x = _f64(x)
    batch, L, dim = x.shape
    w = _f64(w)
    K = w.shape[1]
    w = _f64(w, (dim, K))
    bias = _f64(bias, (dim,))
    u = np.zeros((batch, L, dim), dtype=np.float64)
    self._lib.oracle_causal_conv1d_silu(batch, L, dim, K, _ptr(x), _ptr(w), _ptr(bias), _ptr(u))
    return u


Oracle.causal_conv1d_silu = _conv_method


def _conv_bwd_method(self, x, w, du, bias=None):
    """Gradients of the input stage for dLoss/du = du [batch, L, dim]. Returns a
    dict of float64 arrays: dx [batch, L, dim], dw [dim, K], dbias [dim] (the
    gradient at zero when bias is None)."""
    x = _f64(x)
    batch, L, dim = x.shape
    w = _f64(w)
    K = w.shape[1]
    w = _f64(w, (dim, K))
    bias = _f64(bias, (dim,))
    du = _f64(du, (batch, L, dim))
    g = {"dx": np.zeros((batch, L, dim)), "dw": np.zeros((dim, K)), "dbias": np.zeros(dim)}
    self._lib.oracle_causal_conv1d_silu_bwd(batch, L, dim, K, _ptr(x), _ptr(w), _ptr(bias),
                                            _ptr(du), _ptr(g["dx"]), _ptr(g["dw"]),
                                            _ptr(g["dbias"]))
    return g


Oracle.causal_conv1d_silu_bwd = _conv_bwd_method


def _ssd_method(self, x, dt, A, B, C, D=None, dt_bias=None, dt_softplus=False, h0=None,
                nthreads=None):
    """Mamba-2's SSD layer: x [batch, L, H, P]; dt [batch, L, H]; A, D, dt_bias
    [H]; B, C [batch, L, G, N] (head hd reads group hd // (H // G)); h0
    [batch, H, P, N]. Returns (y [batch, L, H, P], final_state [batch, H, P, N])."""
    x = _f64(x)
    batch, L, H, P = x.shape
    B = _f64(B)
    G, N = B.shape[2], B.shape[3]
    B, C = _f64(B, (batch, L, G, N)), _f64(C, (batch, L, G, N))
    dt, A = _f64(dt, (batch, L, H)), _f64(A, (H,))
    D, dt_bias = _f64(D, (H,)), _f64(dt_bias, (H,))
    h0 = _f64(h0, (batch, H, P, N))
    y = np.zeros((batch, L, H, P))
    fs = np.zeros((batch, H, P, N))
    rc = self._lib.oracle_ssd(batch, L, H, P, G, N, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C),
                              _ptr(D), _ptr(dt_bias), int(bool(dt_softplus)), _ptr(h0), _ptr(y),
                              _ptr(fs), int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_ssd failed (%d)" % rc)
    return y, fs


Oracle.ssd = _ssd_method


def _conv_scan_bwd_method(self, x, delta, A, B, C, conv_w, dout, conv_bias=None, D=None, z=None,
                          delta_bias=None, delta_softplus=False, h0=None, dh_final=None,
                          nthreads=None):
    """Gradients of the input stage followed by the scan (the scan reads
    u = silu(conv(x)) where it would read x, the D skip included): the scan's
    gradients at x = u, then dx, dconv_w, dconv_bias from the input stage's
    backward fed du = the scan's dx. Returns the dict of selective_scan_bwd
    (dx now the gradient of the stage's input) plus dconv_w, dconv_bias."""
    u = self.causal_conv1d_silu(x, conv_w, conv_bias)
    g = self.selective_scan_bwd(u, delta, A, B, C, dout, D=D, z=z, delta_bias=delta_bias,
                                delta_softplus=delta_softplus, h0=h0, dh_final=dh_final,
                                nthreads=nthreads)
    gc = self.causal_conv1d_silu_bwd(x, conv_w, g["dx"], bias=conv_bias)
    g["dx"], g["dconv_w"], g["dconv_bias"] = gc["dx"], gc["dw"], gc["dbias"]
    return g


Oracle.selective_scan_conv_bwd = _conv_scan_bwd_method


def _bwd_method(self, x, delta, A, B, C, dout, D=None, z=None, delta_bias=None,
                delta_softplus=False, h0=None, dh_final=None, nthreads=None, zoh=False):
    """Gradients of the selective scan for the loss sum(dout * out) (+ sum(dh_final
    * final_state)); zoh=True differentiates the exact zero-order-hold scan.
    Returns a dict of float64 arrays: dx, ddelta, dz (None without z)
    [batch, L, dim]; dA [dim, N]; dB, dC [batch, L, N]; dD, ddelta_bias [dim]
    (None without D / delta_bias); dh0 [batch, dim, N]."""
    x = _f64(x)
    batch, L, dim = x.shape
    A = _f64(A)
    N = A.shape[1]
    delta = _f64(delta, (batch, L, dim))
    A = _f64(A, (dim, N))
    B, C = _f64(B, (batch, L, N)), _f64(C, (batch, L, N))
    D, z = _f64(D, (dim,)), _f64(z, (batch, L, dim))
    delta_bias = _f64(delta_bias, (dim,))
    h0, dh_final = _f64(h0, (batch, dim, N)), _f64(dh_final, (batch, dim, N))
    dout = _f64(dout, (batch, L, dim))
    g = {"dx": np.zeros((batch, L, dim)), "ddelta": np.zeros((batch, L, dim)),
         "dA": np.zeros((dim, N)), "dB": np.zeros((batch, L, N)), "dC": np.zeros((batch, L, N)),
         "dD": np.zeros(dim) if D is not None else None,
         "dz": np.zeros((batch, L, dim)) if z is not None else None,
         "ddelta_bias": np.zeros(dim) if delta_bias is not None else None,
         "dh0": np.zeros((batch, dim, N))}
    fn = self._lib.oracle_selective_scan_bwd_zoh if zoh else self._lib.oracle_selective_scan_bwd
    rc = fn(
        batch, L, dim, N, _ptr(x), _ptr(delta), _ptr(A), _ptr(B), _ptr(C), _ptr(D), _ptr(z),
        _ptr(delta_bias), int(bool(delta_softplus)), _ptr(h0), _ptr(dout), _ptr(dh_final),
        _ptr(g["dx"]), _ptr(g["ddelta"]), _ptr(g["dA"]), _ptr(g["dB"]), _ptr(g["dC"]),
        _ptr(g["dD"]), _ptr(g["dz"]), _ptr(g["ddelta_bias"]), _ptr(g["dh0"]),
        int(nthreads or default_threads()))
    if rc != 0:
        raise RuntimeError("oracle_selective_scan_bwd failed (%d)" % rc)
    return g


Oracle.selective_scan_bwd = _bwd_method


def _bcd_method(self, x, delta, A, B, C, D=None, z=None, delta_bias=None, delta_softplus=False,
                h0=None, nthreads=None, zoh=False):
    """The scan with per-channel B, C [batch, L, dim, N]: every channel d is the
    one-channel scan of the oracle with its own rows B[:, :, d], C[:, :, d]
    (channels are independent). Returns (out, final_state) like selective_scan."""
    x = _f64(x)
    batch, L, dim = x.shape
    B, C = _f64(B), _f64(C)
    N = B.shape[3]
    out = np.zeros((batch, L, dim))
    fs = np.zeros((batch, dim, N))
    A = _f64(A, (dim, N))
    for d in range(dim):
        sl = (slice(None), slice(None), slice(d, d + 1))
        o, f = self.selective_scan(
            x[sl], _f64(delta)[sl], A[d:d + 1], B[:, :, d], C[:, :, d],
            D=None if D is None else _f64(D)[d:d + 1], z=None if z is None else _f64(z)[sl],
            delta_bias=None if delta_bias is None else _f64(delta_bias)[d:d + 1],
            delta_softplus=delta_softplus, h0=None if h0 is None else _f64(h0)[:, d:d + 1],
            nthreads=1, zoh=zoh)
        out[:, :, d] = o[:, :, 0]
        fs[:, d] = f[:, 0]
    return out, fs


Oracle.selective_scan_bcd = _bcd_method


def _bcd_step_method(self, state, x, delta, A, B, C, D=None, z=None, delta_bias=None,
                     delta_softplus=False, zoh=False):
    """One recurrent step with per-channel B, C [batch, dim, N]: channel d is the
    one-channel step of the oracle with its own rows B[:, d], C[:, d]. state
    [batch, dim, N] is not modified. Returns (out [batch, dim], new_state)."""
    st = _f64(state)
    batch, dim, N = st.shape
    B, C = _f64(B, (batch, dim, N)), _f64(C, (batch, dim, N))
    x, delta = _f64(x, (batch, dim)), _f64(delta, (batch, dim))
    A = _f64(A, (dim, N))
    out = np.zeros((batch, dim))
    new = np.zeros((batch, dim, N))
    col = lambda a, d: None if a is None else _f64(a)[:, d:d + 1]
    vec = lambda a, d: None if a is None else _f64(a)[d:d + 1]
    for d in range(dim):
        o, h = self.state_update(st[:, d:d + 1], x[:, d:d + 1], delta[:, d:d + 1], A[d:d + 1],
                                 B[:, d], C[:, d], D=vec(D, d), z=col(z, d),
                                 delta_bias=vec(delta_bias, d), delta_softplus=delta_softplus,
                                 zoh=zoh)
        out[:, d] = o[:, 0]
        new[:, d] = h[:, 0]
    return out, new


Oracle.state_update_bcd = _bcd_step_method


def _bcd_bwd_method(self, x, delta, A, B, C, dout, D=None, z=None, delta_bias=None,
                    delta_softplus=False, h0=None, dh_final=None, nthreads=None, zoh=False):
    """Gradients of the per-channel B, C scan: channel d is the one-channel scan
    with rows B[:, :, d], C[:, :, d], so its gradients are those of that scan
    (dB, dC of a one-channel problem sum over that channel alone). Returns the
    dict of selective_scan_bwd with dB, dC of shape [batch, L, dim, N]."""
    x = _f64(x)
    batch, L, dim = x.shape
    B, C = _f64(B), _f64(C)
    N = B.shape[3]
    A = _f64(A, (dim, N))
    sl3 = lambda a, d: None if a is None else _f64(a)[:, :, d:d + 1]
    sl1 = lambda a, d: None if a is None else _f64(a)[d:d + 1]
    sl2 = lambda a, d: None if a is None else _f64(a)[:, d:d + 1]
    g = {"dx": np.zeros((batch, L, dim)), "ddelta": np.zeros((batch, L, dim)),
         "dA": np.zeros((dim, N)), "dB": np.zeros((batch, L, dim, N)),
         "dC": np.zeros((batch, L, dim, N)),
         "dD": np.zeros(dim) if D is not None else None,
         "dz": np.zeros((batch, L, dim)) if z is not None else None,
         "ddelta_bias": np.zeros(dim) if delta_bias is not None else None,
         "dh0": np.zeros((batch, dim, N))}
    for d in range(dim):
        gd = self.selective_scan_bwd(
            sl3(x, d), sl3(delta, d), A[d:d + 1], B[:, :, d], C[:, :, d], sl3(dout, d),
            D=sl1(D, d), z=sl3(z, d), delta_bias=sl1(delta_bias, d),
            delta_softplus=delta_softplus, h0=sl2(h0, d), dh_final=sl2(dh_final, d),
            nthreads=1, zoh=zoh)
        for k in ("dx", "ddelta", "dz"):
            if g[k] is not None:
                g[k][:, :, d] = gd[k][:, :, 0]
        g["dA"][d] = gd["dA"][0]
        g["dB"][:, :, d] = gd["dB"]
        g["dC"][:, :, d] = gd["dC"]
        for k in ("dD", "ddelta_bias"):
            if g[k] is not None:
                g[k][d] = gd[k][0]
        g["dh0"][:, d] = gd["dh0"][:, 0]
    return g


Oracle.selective_scan_bcd_bwd = _bcd_bwd_method


def default() -> Oracle:
    """The oracle built from ssm_oracle.c (compiled on first use)."""
    global _default
    with _lock:
        if _default is None:
            _default = Oracle(build())
    return _default


def softplus(v):
    return default().softplus(v)


def silu(z):
    return default().silu(z)


def phi(z):
    return default().phi(z)


def phi_prime(z):
    return default().phi_prime(z)


def recurrence(*a, **k):
    return default().recurrence(*a, **k)


def selective_scan(*a, **k):
    return default().selective_scan(*a, **k)


def state_update(*a, **k):
    return default().state_update(*a, **k)


def causal_conv1d_silu(*a, **k):
    return default().causal_conv1d_silu(*a, **k)


def causal_conv1d_silu_bwd(*a, **k):
    return default().causal_conv1d_silu_bwd(*a, **k)


def ssd(*a, **k):
    return default().ssd(*a, **k)


def selective_scan_conv_bwd(*a, **k):
    return default().selective_scan_conv_bwd(*a, **k)


def selective_scan_bwd(*a, **k):
    return default().selective_scan_bwd(*a, **k)


def state_update_bcd(*a, **k):
    return default().state_update_bcd(*a, **k)


def selective_scan_bcd(*a, **k):
    return default().selective_scan_bcd(*a, **k)


def selective_scan_bcd_bwd(*a, **k):
    return default().selective_scan_bcd_bwd(*a, **k)
