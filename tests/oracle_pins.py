"""Checks that pin the float64 oracle to facts the pages and mathematics fix.

Each ``pin_*`` function takes a compiled oracle (``oracle.Oracle``) and raises
AssertionError when the oracle disagrees with a fact that does not come from
the oracle itself: a value printed on the pages, a closed form, a library
routine, or an invariant of the recurrence. ``test_oracle_pins.py`` runs them
on the real oracle; ``test_oracle_mutants.py`` runs them on copies of the
oracle with planted mistakes and requires that every mistake trips one.

Sources (page title, section):
  * "State-space models (Mamba, S4)", "Worked Example: 2D SSM Step" (the
    printed 2-D step) and "The Convolution View" (time-invariant case: y is the
    causal convolution of x with K = (C Bbar, C Abar Bbar, C Abar^2 Bbar, ...),
    from h_0 = 0).
  * "State Space Models -- Mamba, S4, and Beyond", "Mamba (S6 -- Selective
    State Space)" (dA = exp(delta A), dB = delta B, y + D u) and its
    "Verification Checklist" (recurrent inference must reproduce the scan).
  * "Mamba: State Space Models Challenge Transformers", "Mamba's Innovation:
    Selection" (softplus on delta, output gate y * silu(z)).
  * The gradients of the scan (training through it: "State-space models
    (Mamba, S4)", "Training vs Inference Modes") are pinned to finite
    differences of the forward and to PyTorch autograd through a plain loop;
    so are those of the variants and of the input stage (autograd through
    torch.nn.functional.conv1d).
  * The exact zero-order hold ("State-space models (Mamba, S4)", "From
    Continuous to Discrete: The Key Step") is pinned to its closed form, to ODE
    integration (scipy solve_ivp) and to scipy.signal.cont2discrete.
  * Mamba-2's SSD layer ("State Space Models and Mamba", "Mamba 2 and Hybrid
    Architectures": a structured matrix multiplication) is pinned to the scan
    with tied parameters, to the masked matrix form and to its chunked form.
"""
from __future__ import annotations

import os

import numpy as np
from scipy.special import expit

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name="worked_example_2d.txt"):
    vals = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = line.split("=", 1)
            vals[k.strip()] = np.array([float(t) for t in v.split()], dtype=np.float64)
    return vals


def _rng(seed):
    return np.random.Generator(np.random.PCG64(seed))


def _close(a, b, rtol, atol=0.0, what=""):
    a, b = np.asarray(a, np.float64), np.asarray(b, np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    lim = atol + rtol * np.abs(b)
    assert np.all(err <= lim), "%s: max err %.3e (worst at %s)" % (
        what, float(err.max()), np.unravel_index(int(np.argmax(err - lim)), err.shape))


# --------------------------------------------------------------------------
# 1. the worked example
# --------------------------------------------------------------------------
def pin_worked_example_core(orc):
    g = load_golden()
    N = int(g["N"][0])
    y, h = orc.recurrence(g["Abar"].reshape(1, N), g["Bbar"].reshape(1, N),
                          g["C"].reshape(1, N), g["x1"], g["h0"])
    _close(h, g["h1"], 0, 1e-12, "h1")
    _close(y, g["y1"], 0, 1e-12, "y1")
    # the page's intermediate terms: Abar h0 alone (x = 0), Bbar x alone (h0 = 0)
    _, h_a = orc.recurrence(g["Abar"].reshape(1, N), g["Bbar"].reshape(1, N),
                            g["C"].reshape(1, N), [0.0], g["h0"])
    _close(h_a, g["Abar_h0"], 0, 1e-12, "Abar h0")
    _, h_b = orc.recurrence(g["Abar"].reshape(1, N), g["Bbar"].reshape(1, N),
                            g["C"].reshape(1, N), g["x1"], np.zeros(N))
    _close(h_b, g["Bbar_x1"], 0, 1e-12, "Bbar x1")


def pin_worked_example_selective_path(orc):
    """The same step through the full selective path: delta = 1 and
    A = [ln 0.9, ln 0.5] give Abar = exp(delta A) = diag(0.9, 0.5) and
    Bbar = delta B = B; no D, no gate."""
    g = load_golden()
    N = int(g["N"][0])
    x = g["x1"].reshape(1, 1, 1)
    delta = np.ones((1, 1, 1))
    A = np.log(g["Abar"]).reshape(1, N)
    B = g["Bbar"].reshape(1, 1, N)
    C = g["C"].reshape(1, 1, N)
    out, fs = orc.selective_scan(x, delta, A, B, C, h0=g["h0"].reshape(1, 1, N))
    _close(fs.reshape(N), g["h1"], 0, 1e-12, "h1 (selective path)")
    _close(out.reshape(1), g["y1"], 0, 1e-12, "y1 (selective path)")
    # as a decode step from the same cached state
    o2, st = orc.state_update(g["h0"].reshape(1, 1, N), g["x1"].reshape(1, 1),
                              np.ones((1, 1)), A, g["Bbar"].reshape(1, N),
                              g["C"].reshape(1, N))
    _close(st.reshape(N), g["h1"], 0, 1e-12, "h1 (decode step)")
    _close(o2.reshape(1), g["y1"], 0, 1e-12, "y1 (decode step)")


# --------------------------------------------------------------------------
# 2. time-invariant case == causal convolution with K
# --------------------------------------------------------------------------
def pin_lti_convolution(orc, seed=11):
    r = _rng(seed)
    batch, L, dim, N = 2, 48, 3, 5
    A = -np.exp(r.standard_normal((dim, N)) * 0.5)
    dd = np.exp(r.uniform(np.log(1e-2), np.log(0.5), dim))      # one step per channel
    B0, C0 = r.standard_normal(N), r.standard_normal(N)
    D = r.uniform(0.5, 1.5, dim)
    x = r.standard_normal((batch, L, dim))
    delta = np.broadcast_to(dd, (batch, L, dim)).copy()
    B = np.broadcast_to(B0, (batch, L, N)).copy()
    C = np.broadcast_to(C0, (batch, L, N)).copy()
    out, _ = orc.selective_scan(x, delta, A, B, C, D=D)
    k = np.arange(L)
    for d in range(dim):
        Abar = np.exp(dd[d] * A[d])                                   # [N]
        Bbar = dd[d] * B0
        K = (C0[None, :] * Abar[None, :] ** k[:, None] * Bbar[None, :]).sum(1)  # [L]
        for b in range(batch):
            ref = np.convolve(x[b, :, d], K)[:L] + D[d] * x[b, :, d]
            _close(out[b, :, d], ref, 1e-12, 1e-12, "LTI conv (b=%d, d=%d)" % (b, d))


# --------------------------------------------------------------------------
# 3. selective case == brute-force unrolled sum
# --------------------------------------------------------------------------
def _unrolled(x, delta, A, B, C, D, z, bias, softplus, h0):
    """y_k = sum_{i<=k} C_k (prod_{j=i+1..k} Abar_j) Bbar_i x_i
             + C_k (prod_{j<=k} Abar_j) h0 + D x_k, gated by silu(z_k).
    Independent of the oracle's loop: explicit products, one term at a time."""
    batch, L, dim = x.shape
    N = A.shape[1]
    dt = delta + (bias if bias is not None else 0.0)
    if softplus:
        dt = np.logaddexp(0.0, dt)                        # log(1 + e^v)
    Abar = np.exp(dt[..., None] * A[None, None])          # [b, L, d, N]
    Bbar = dt[..., None] * B[:, :, None, :]               # [b, L, d, N]
    y = np.zeros((batch, L, dim))
    hL = np.zeros((batch, dim, N))
    for b in range(batch):
        for d in range(dim):
            for kk in range(L):
                s = np.zeros(N)
                for i in range(kk + 1):
                    p = np.ones(N)
                    for j in range(i + 1, kk + 1):
                        p = p * Abar[b, j, d]
                    s = s + p * Bbar[b, i, d] * x[b, i, d]
                p0 = np.ones(N)
                for j in range(kk + 1):
                    p0 = p0 * Abar[b, j, d]
                h = s + (p0 * h0[b, d] if h0 is not None else 0.0)
                yk = float(np.dot(C[b, kk], h))
                if D is not None:
                    yk += D[d] * x[b, kk, d]
                if z is not None:
                    yk *= z[b, kk, d] * expit(z[b, kk, d])
                y[b, kk, d] = yk
                if kk == L - 1:
                    hL[b, d] = h
    return y, hL


def pin_unrolled_sum(orc, seed=12):
    r = _rng(seed)
    batch, L, dim, N = 2, 9, 3, 3
    x = r.standard_normal((batch, L, dim))
    u = r.standard_normal((batch, L, dim)) * 0.5
    bias = np.log(np.expm1(np.exp(r.uniform(np.log(1e-2), np.log(0.5), dim))))
    A = -np.exp(r.standard_normal((dim, N)) * 0.5)
    A[0, 0] = 0.3                                  # one growing mode: sign matters
    B = r.standard_normal((batch, L, N))
    C = r.standard_normal((batch, L, N))
    D = r.uniform(0.5, 1.5, dim)
    z = r.standard_normal((batch, L, dim))
    h0 = r.standard_normal((batch, dim, N))
    for softplus in (True, False):
        d_in = u if softplus else np.abs(u) * 0.2
        out, fs = orc.selective_scan(x, d_in, A, B, C, D=D, z=z, delta_bias=bias,
                                     delta_softplus=softplus, h0=h0)
        ry, rh = _unrolled(x, d_in, A, B, C, D, z, bias, softplus, h0)
        _close(out, ry, 1e-11, 1e-12, "unrolled y (softplus=%s)" % softplus)
        _close(fs, rh, 1e-11, 1e-12, "unrolled h_L (softplus=%s)" % softplus)
    # without D / z / bias / h0
    out, fs = orc.selective_scan(x, np.abs(u) * 0.2, A, B, C)
    ry, rh = _unrolled(x, np.abs(u) * 0.2, A, B, C, None, None, None, False, None)
    _close(out, ry, 1e-11, 1e-12, "unrolled y (bare)")
    _close(fs, rh, 1e-11, 1e-12, "unrolled h_L (bare)")


# --------------------------------------------------------------------------
# 4. invariants
# --------------------------------------------------------------------------
def _random_case(r, batch=2, L=32, dim=4, N=6):
    return dict(
        x=r.standard_normal((batch, L, dim)),
        delta=np.exp(r.uniform(np.log(1e-3), np.log(1e-1), (batch, L, dim))),
        A=-np.exp(r.standard_normal((dim, N)) * 0.5),
        B=r.standard_normal((batch, L, N)),
        C=r.standard_normal((batch, L, N)),
        D=r.uniform(0.5, 1.5, dim),
        z=r.standard_normal((batch, L, dim)),
    )


def pin_linearity(orc, seed=13):
    """Delta, B, C, z fixed: y is linear in x (the gate multiplies y by a
    factor that does not depend on x; D x is linear)."""
    r = _rng(seed)
    c = _random_case(r)
    x1, x2 = c.pop("x"), r.standard_normal(c["delta"].shape)
    a, b = 0.7, -1.9
    y1, h1 = orc.selective_scan(x1, **c)
    y2, h2 = orc.selective_scan(x2, **c)
    y3, h3 = orc.selective_scan(a * x1 + b * x2, **c)
    _close(y3, a * y1 + b * y2, 1e-12, 1e-12, "linearity y")
    _close(h3, a * h1 + b * h2, 1e-12, 1e-12, "linearity h")
    # homogeneity alone also fixes that nothing in y is independent of x
    y0, h0 = orc.selective_scan(np.zeros_like(x1), **c)
    assert np.all(y0 == 0.0) and np.all(h0 == 0.0), "x = 0 must give y = 0, h = 0"


def pin_delta_zero(orc, seed=14):
    """delta = 0: Abar = 1, Bbar = 0, so h stays h0 exactly and
    y = (C h0 + D x) * silu(z)."""
    r = _rng(seed)
    c = _random_case(r)
    batch, L, dim = c["x"].shape
    N = c["A"].shape[1]
    h0 = r.standard_normal((batch, dim, N))
    c["delta"] = np.zeros_like(c["delta"])
    out, fs = orc.selective_scan(h0=h0, **c)
    assert np.array_equal(fs, h0), "delta = 0 must leave the state bit-identical"
    ref = (np.einsum("btn,bdn->btd", c["C"], h0) + c["D"] * c["x"]) * (c["z"] * expit(c["z"]))
    _close(out, ref, 1e-12, 1e-12, "delta = 0 output")


def pin_delta_large(orc, seed=15):
    """delta -> infinity with A < 0: Abar -> 0 (exactly 0 in float64 for
    delta A < -745), so the state resets every step: h_t = delta B_t x_t."""
    r = _rng(seed)
    c = _random_case(r)
    c["delta"] = np.full_like(c["delta"], 1e4)
    c["A"] = -np.abs(c["A"]) - 0.1
    out, fs = orc.selective_scan(**c)
    ht = c["delta"][..., None] * c["B"][:, :, None, :] * c["x"][..., None]   # [b,L,d,N]
    _close(fs, ht[:, -1], 1e-14, 0, "reset state")
    ref = ((c["C"][:, :, None, :] * ht).sum(-1) + c["D"] * c["x"]) * (c["z"] * expit(c["z"]))
    _close(out, ref, 1e-12, 1e-9, "reset output")


def pin_n1_closed_form(orc, seed=16):
    """N = 1, constant delta, B, x: a = e^{delta A}, c = delta B x and
    h_L = a^L h0 + c (1 - a^L) / (1 - a) (geometric series)."""
    r = _rng(seed)
    L = 300
    for dt, Aval, Bv, xv, h0 in [(0.01, -1.0, 0.8, 1.3, 0.4), (0.2, -3.0, -1.1, 0.5, -2.0),
                                 (0.05, 0.5, 0.3, -0.7, 1.0)]:
        x = np.full((1, L, 1), xv)
        delta = np.full((1, L, 1), dt)
        A = np.array([[Aval]])
        B = np.full((1, L, 1), Bv)
        C = np.full((1, L, 1), 1.0)
        out, fs = orc.selective_scan(x, delta, A, B, C, h0=np.array([[[h0]]]))
        a, c = np.exp(dt * Aval), dt * Bv * xv
        t = np.arange(1, L + 1)
        ref = a ** t * h0 + c * (1 - a ** t) / (1 - a)
        _close(out.reshape(L), ref, 1e-11, 1e-13, "geometric series")
        _close(fs.reshape(1), ref[-1:], 1e-11, 1e-13, "geometric series h_L")
    del r


def pin_split_resume(orc, seed=17):
    """scan over [0, L) == scan over [L1, L) started from the state that the
    scan over [0, L1) ends in (the chunk-carry identity)."""
    r = _rng(seed)
    c = _random_case(r, L=40)
    c["delta_bias"] = r.standard_normal(c["A"].shape[0]) * 0.1
    full, fs = orc.selective_scan(delta_softplus=True, **c)
    L1 = 17
    head = {k: (v[:, :L1] if k in ("x", "delta", "B", "C", "z") else v) for k, v in c.items()}
    tail = {k: (v[:, L1:] if k in ("x", "delta", "B", "C", "z") else v) for k, v in c.items()}
    y1, h1 = orc.selective_scan(delta_softplus=True, **head)
    y2, h2 = orc.selective_scan(delta_softplus=True, h0=h1, **tail)
    assert np.array_equal(np.concatenate([y1, y2], axis=1), full), "split output"
    assert np.array_equal(h2, fs), "split final state"


def pin_decode_equals_scan(orc, seed=18):
    """Recurrent inference (one step per token on a cached state) reproduces
    the scan token by token, from the same initial state."""
    r = _rng(seed)
    c = _random_case(r, L=12)
    batch, L, dim = c["x"].shape
    N = c["A"].shape[1]
    h0 = r.standard_normal((batch, dim, N))
    bias = r.standard_normal(dim) * 0.1
    full, fs = orc.selective_scan(h0=h0, delta_bias=bias, delta_softplus=True, **c)
    st = h0
    for t in range(L):
        y, st = orc.state_update(st, c["x"][:, t], c["delta"][:, t], c["A"], c["B"][:, t],
                                 c["C"][:, t], D=c["D"], z=c["z"][:, t], delta_bias=bias,
                                 delta_softplus=True)
        _close(y, full[:, t], 1e-14, 1e-14, "decode step %d" % t)
    _close(st, fs, 1e-14, 1e-14, "decode final state")


def pin_softplus_silu(orc):
    """softplus and silu against library routines at float64."""
    vs = [-800.0, -40.0, -20.0, -3.0, -1e-3, 0.0, 1e-8, 0.5, 3.0, 20.0, 40.0, 700.0]
    for v in vs:
        ref = float(np.logaddexp(0.0, v))
        got = orc.softplus(v)
        assert abs(got - ref) <= 1e-15 * max(1.0, abs(ref)) + 1e-300, ("softplus", v, got, ref)
        refs = v * float(expit(v))
        gots = orc.silu(v)
        assert abs(gots - refs) <= 1e-15 * max(1.0, abs(refs)) + 1e-300, ("silu", v, gots, refs)
    # very negative arguments: softplus(v) = e^v - e^{2v}/2 + O(e^{3v}); the
    # relative accuracy there is what keeps small steps exact
    for v in (-30.0, -50.0, -300.0):
        ev = np.exp(v)
        assert abs(orc.softplus(v) / (ev - ev * ev / 2) - 1.0) < 1e-15, v


def pin_thread_invariance(orc, seed=19):
    r = _rng(seed)
    c = _random_case(r, batch=3, L=20, dim=7)
    y1, h1 = orc.selective_scan(nthreads=1, **c)
    y8, h8 = orc.selective_scan(nthreads=8, **c)
    assert np.array_equal(y1, y8) and np.array_equal(h1, h8)


def _conv_case(r, K, batch=2, L=40, dim=5):
    x = r.standard_normal((batch, L, dim))
    w = r.standard_normal((dim, K))
    bias = r.standard_normal(dim)
    return x, w, bias


def _silu(v):
    return v * expit(v)


def pin_conv_library(orc, seed=21):
    """Causal depthwise conv1d + SiLU ("State Space Models -- Mamba, S4, and
    Beyond", MambaBlock: nn.Conv1d(kernel_size=d_conv, padding=d_conv - 1,
    groups=d_inner) cut to seq_len, then silu): the pre-activation of channel d
    is numpy's full convolution of x[:, d] with the reversed kernel (Conv1d is
    a cross-correlation), truncated to the first L outputs, plus the bias."""
    r = _rng(seed)
    for K in (1, 2, 3, 4):
        x, w, bias = _conv_case(r, K)
        got = orc.causal_conv1d_silu(x, w, bias)
        batch, L, dim = x.shape
        for b in range(batch):
            for d in range(dim):
                pre = np.convolve(x[b, :, d], w[d, ::-1])[:L] + bias[d]
                _close(got[b, :, d], _silu(pre), 1e-13, 1e-14, "conv K=%d b=%d d=%d" % (K, b, d))


def pin_conv_taps(orc, seed=22):
    """Single-tap kernels: the last tap is the identity (u = silu(x + bias));
    the first tap of a width-4 kernel delays by three tokens, with zeros
    (silu(bias)) before the sequence start -- the causal left padding."""
    r = _rng(seed)
    x, _, bias = _conv_case(r, 4)
    w = np.zeros((x.shape[2], 4))
    w[:, 3] = 1.0
    _close(orc.causal_conv1d_silu(x, w, bias), _silu(x + bias), 1e-15, 1e-15, "identity tap")
    w = np.zeros((x.shape[2], 4))
    w[:, 0] = 1.0
    want = np.empty_like(x)
    want[:, :3] = _silu(bias)
    want[:, 3:] = _silu(x[:, :-3] + bias)
    _close(orc.causal_conv1d_silu(x, w, bias), want, 1e-15, 1e-15, "delay tap")
    nob = np.zeros_like(x)                  # no bias: silu(0) = 0 before the start
    nob[:, 3:] = _silu(x[:, :-3])
    _close(orc.causal_conv1d_silu(x, w), nob, 1e-15, 1e-15, "delay tap, no bias")


def pin_conv_causal(orc, seed=23):
    """Changing x at token t0 changes no output before t0 and, for a width-K
    kernel, none after t0 + K - 1."""
    r = _rng(seed)
    x, w, bias = _conv_case(r, 4, batch=1, L=30, dim=3)
    base = orc.causal_conv1d_silu(x, w, bias)
    x2 = x.copy()
    x2[0, 12] += 1.0
    moved = orc.causal_conv1d_silu(x2, w, bias)
    assert np.array_equal(moved[0, :12], base[0, :12]), "conv reads the future"
    assert np.array_equal(moved[0, 16:], base[0, 16:]), "conv reaches beyond its width"
    assert np.all(moved[0, 12:16] != base[0, 12:16]), "conv misses a tap"


def _torch_conv_silu(x, w, bias):
    """The input stage with PyTorch's own depthwise conv1d: [batch, L, dim] in,
    left padding K - 1 on both sides cut back to the first L outputs."""
    import torch
    K = w.shape[1]
    pre = torch.nn.functional.conv1d(x.transpose(1, 2), w[:, None, :], bias=bias, padding=K - 1,
                                     groups=w.shape[0])[:, :, :x.shape[1]]
    return torch.nn.functional.silu(pre).transpose(1, 2)


def pin_conv_bwd(orc, seed=24):
    """The input stage's gradients (dx, dw, dbias) equal central differences of
    the oracle's own forward and PyTorch autograd through
    torch.nn.functional.conv1d, for K = 1..4, with and without a bias."""
    import torch
    r = _rng(seed)
    for K in (1, 2, 3, 4):
        x, w, bias = _conv_case(r, K, batch=2, L=9, dim=3)
        du = r.standard_normal(x.shape)
        for b_ in (bias, None):
            g = orc.causal_conv1d_silu_bwd(x, w, du, bias=b_)
            tx, tw = torch.tensor(x, requires_grad=True), torch.tensor(w, requires_grad=True)
            tb = torch.tensor(b_ if b_ is not None else np.zeros(3), requires_grad=True)
            (_torch_conv_silu(tx, tw, tb) * torch.tensor(du)).sum().backward()
            for name, t in (("dx", tx), ("dw", tw), ("dbias", tb)):
                _close(g[name], t.grad.numpy(), 1e-12, 1e-13, "conv %s vs autograd, K=%d" % (name, K))
        eps = 1e-6
        for name, arr in (("x", x), ("w", w), ("bias", bias)):
            fd = np.zeros_like(arr)
            for i in np.ndindex(arr.shape):
                p, m = arr.copy(), arr.copy()
                p[i] += eps
                m[i] -= eps
                a = {"x": x, "w": w, "bias": bias}
                lp = (orc.causal_conv1d_silu(**dict(a, **{name: p})) * du).sum()
                lm = (orc.causal_conv1d_silu(**dict(a, **{name: m})) * du).sum()
                fd[i] = (lp - lm) / (2 * eps)
            g = orc.causal_conv1d_silu_bwd(x, w, du, bias=bias)
            _close(g["d" + name], fd, 1e-6, 1e-7, "conv d%s vs finite differences, K=%d" % (name, K))


def pin_conv_scan_bwd(orc, seed=25):
    """The input stage followed by the scan: every gradient, the conv's weights
    and bias included, equals PyTorch autograd through conv1d + SiLU and the
    plain float64 loop of the scan."""
    import torch
    r = _rng(seed)
    c, dout, dhf = _bwd_case(r, 2, 8, 3, 4, True, True)
    w = r.standard_normal((3, 4)) * 0.5
    cb = r.standard_normal(3) * 0.2
    g = orc.selective_scan_conv_bwd(c["x"], c["delta"], c["A"], c["B"], c["C"], w, dout,
                                    conv_bias=cb, D=c["D"], z=c["z"],
                                    delta_bias=c["delta_bias"], delta_softplus=True, h0=c["h0"],
                                    dh_final=dhf)
    tens = {k: torch.tensor(v, requires_grad=True) for k, v in c.items()}
    tw, tcb = torch.tensor(w, requires_grad=True), torch.tensor(cb, requires_grad=True)
    u = _torch_conv_silu(tens["x"], tw, tcb)
    out, fs = _torch_scan(u, tens["delta"], tens["A"], tens["B"], tens["C"], tens["D"],
                          tens["z"], tens["delta_bias"], True, tens["h0"])
    ((out * torch.tensor(dout)).sum() + (fs * torch.tensor(dhf)).sum()).backward()
    for name, t in tens.items():
        _close(g[_GRAD_OF[name]], t.grad.numpy(), 1e-10, 1e-12, "conv+scan d%s vs autograd" % name)
    _close(g["dconv_w"], tw.grad.numpy(), 1e-10, 1e-12, "conv+scan dconv_w vs autograd")
    _close(g["dconv_bias"], tcb.grad.numpy(), 1e-10, 1e-12, "conv+scan dconv_bias vs autograd")


# --------------------------------------------------------------------------
# gradients (the backward of the scan)
# --------------------------------------------------------------------------
def _bwd_case(r, batch, L, dim, N, softplus, full):
    """A small random problem; full=True gives every optional input."""
    c = {"x": r.standard_normal((batch, L, dim)),
         "delta": (r.standard_normal((batch, L, dim)) * 0.5 if softplus
                   else r.uniform(0.05, 0.5, (batch, L, dim))),
         "A": -np.exp(r.standard_normal((dim, N)) * 0.5),
         "B": r.standard_normal((batch, L, N)), "C": r.standard_normal((batch, L, N)),
         "D": r.uniform(0.5, 1.5, dim) if full else None,
         "z": r.standard_normal((batch, L, dim)) if full else None,
         "delta_bias": r.standard_normal(dim) * 0.3 if full else None,
         "h0": r.standard_normal((batch, dim, N)) if full else None}
    dout = r.standard_normal((batch, L, dim))
    dhf = r.standard_normal((batch, dim, N)) if full else None
    return c, dout, dhf


_GRAD_OF = {"x": "dx", "delta": "ddelta", "A": "dA", "B": "dB", "C": "dC", "D": "dD",
            "z": "dz", "delta_bias": "ddelta_bias", "h0": "dh0"}


def pin_bwd_finite_differences(orc, seed=31):
    """Every gradient equals the central difference of the oracle's own loss
    sum(dout * out) + sum(dh_final * final_state) (step 1e-6, truncation error
    ~1e-12): the backward is the derivative of the forward."""
    r = _rng(seed)
    for softplus, full, shape in ((True, True, (2, 5, 3, 4)), (False, False, (1, 6, 2, 1)),
                                  (True, False, (2, 4, 2, 2))):
        c, dout, dhf = _bwd_case(r, *shape, softplus, full)
        g = orc.selective_scan_bwd(c["x"], c["delta"], c["A"], c["B"], c["C"], dout, D=c["D"],
                                   z=c["z"], delta_bias=c["delta_bias"],
                                   delta_softplus=softplus, h0=c["h0"], dh_final=dhf)

        def loss(**kw):
            a = dict(c)
            a.update(kw)
            out, fs = orc.selective_scan(a["x"], a["delta"], a["A"], a["B"], a["C"], D=a["D"],
                                         z=a["z"], delta_bias=a["delta_bias"],
                                         delta_softplus=softplus, h0=a["h0"])
            return float((out * dout).sum() + (0.0 if dhf is None else (fs * dhf).sum()))

        eps = 1e-6
        for name, arr in c.items():
            if arr is None:
                continue
            fd = np.zeros_like(arr)
            for i in np.ndindex(arr.shape):
                p, m = arr.copy(), arr.copy()
                p[i] += eps
                m[i] -= eps
                fd[i] = (loss(**{name: p}) - loss(**{name: m})) / (2 * eps)
            _close(g[_GRAD_OF[name]], fd, 1e-6, 1e-7, "d%s vs finite differences" % name)
        for name in ("D", "z", "delta_bias"):
            if c[name] is None:
                assert g[_GRAD_OF[name]] is None


def _torch_scan(x, delta, A, B, C, D, z, bias, softplus, h0, zoh=False):
    """The scan as a plain PyTorch float64 loop (autograd records it). B, C of
    shape [batch, L, dim, N] are per channel; zoh=True takes the input term
    (e^{dt A} - 1)/A B x of the exact zero-order hold (A must be nonzero)."""
    import torch
    batch, L, dim = x.shape
    N = A.shape[1]
    h = h0 if h0 is not None else torch.zeros(batch, dim, N, dtype=torch.float64)
    ys = []
    for t in range(L):
        v = delta[:, t] + (bias if bias is not None else 0.0)
        dt = torch.nn.functional.softplus(v) if softplus else v
        Bt = B[:, t] if B.dim() == 4 else B[:, t, None, :]
        Ct = C[:, t] if C.dim() == 4 else C[:, t, None, :]
        step = torch.expm1(dt[..., None] * A) / A if zoh else dt[..., None]
        h = torch.exp(dt[..., None] * A) * h + step * x[:, t, :, None] * Bt
        y = (h * Ct).sum(-1)
        if D is not None:
            y = y + D * x[:, t]
        if z is not None:
            y = y * torch.nn.functional.silu(z[:, t])
        ys.append(y)
    return torch.stack(ys, 1), h


def pin_bwd_autograd(orc, seed=32):
    """The oracle's gradients equal PyTorch autograd through a plain float64
    loop of the same recurrence (an independent derivation)."""
    import torch
    r = _rng(seed)
    for softplus, full, shape in ((True, True, (2, 9, 5, 4)), (False, True, (1, 7, 3, 8)),
                                  (True, False, (3, 6, 2, 2))):
        c, dout, dhf = _bwd_case(r, *shape, softplus, full)
        tens = {k: (None if v is None else torch.tensor(v, requires_grad=True))
                for k, v in c.items()}
        out, fs = _torch_scan(tens["x"], tens["delta"], tens["A"], tens["B"], tens["C"],
                              tens["D"], tens["z"], tens["delta_bias"], softplus, tens["h0"])
        loss = (out * torch.tensor(dout)).sum()
        if dhf is not None:
            loss = loss + (fs * torch.tensor(dhf)).sum()
        loss.backward()
        g = orc.selective_scan_bwd(c["x"], c["delta"], c["A"], c["B"], c["C"], dout, D=c["D"],
                                   z=c["z"], delta_bias=c["delta_bias"],
                                   delta_softplus=softplus, h0=c["h0"], dh_final=dhf)
        for name, t in tens.items():
            if t is not None:
                _close(g[_GRAD_OF[name]], t.grad.numpy(), 1e-10, 1e-12,
                       "d%s vs autograd" % name)


def pin_bwd_channel_sums(orc, seed=33):
    """dB and dC sum the channels' contributions and dA, dD, dbias sum the
    batch rows': the gradient of a multi-channel problem equals the sum over
    one-channel (and one-row) problems; per-channel gradients are unchanged."""
    r = _rng(seed)
    c, dout, dhf = _bwd_case(r, 2, 8, 3, 4, True, True)
    kw = dict(delta_softplus=True, nthreads=1)
    g = orc.selective_scan_bwd(c["x"], c["delta"], c["A"], c["B"], c["C"], dout, D=c["D"],
                               z=c["z"], delta_bias=c["delta_bias"], h0=c["h0"], dh_final=dhf,
                               **kw)
    dB, dC = np.zeros_like(c["B"]), np.zeros_like(c["C"])
    for b in range(2):
        for d in range(3):
            sl = lambda a: None if a is None else a[b:b + 1, :, d:d + 1]
            gd = orc.selective_scan_bwd(sl(c["x"]), sl(c["delta"]), c["A"][d:d + 1],
                                        c["B"][b:b + 1], c["C"][b:b + 1], sl(dout),
                                        D=c["D"][d:d + 1], z=sl(c["z"]),
                                        delta_bias=c["delta_bias"][d:d + 1],
                                        h0=c["h0"][b:b + 1, d:d + 1],
                                        dh_final=dhf[b:b + 1, d:d + 1], **kw)
            dB[b] += gd["dB"][0]
            dC[b] += gd["dC"][0]
            _close(gd["dx"][0, :, 0], g["dx"][b, :, d], 1e-12, 1e-14, "dx per channel")
            _close(gd["ddelta"][0, :, 0], g["ddelta"][b, :, d], 1e-12, 1e-14, "ddelta per channel")
            _close(gd["dh0"][0, 0], g["dh0"][b, d], 1e-12, 1e-14, "dh0 per channel")
    _close(dB, g["dB"], 1e-12, 1e-14, "dB = sum over channels")
    _close(dC, g["dC"], 1e-12, 1e-14, "dC = sum over channels")
    g4 = orc.selective_scan_bwd(c["x"], c["delta"], c["A"], c["B"], c["C"], dout, D=c["D"],
                                z=c["z"], delta_bias=c["delta_bias"], h0=c["h0"],
                                dh_final=dhf, delta_softplus=True, nthreads=4)
    for k in g:
        if g[k] is not None:
            _close(g4[k], g[k], 1e-12, 1e-14, "%s, 4 threads vs 1" % k)


# --------------------------------------------------------------------------
# exact zero-order hold ("State-space models (Mamba, S4)", "From Continuous to
# Discrete: The Key Step": exact for an input held constant over each step)
# --------------------------------------------------------------------------
def pin_phi(orc):
    """phi(z) = (e^z - 1)/z: 1 at 0, its Taylor series near 0, numpy elsewhere."""
    assert orc.phi(0.0) == 1.0
    for zz in (1e-9, -1e-7, 3e-5):
        series = 1 + zz / 2 + zz * zz / 6
        _close(orc.phi(zz), series, 1e-15, 0.0, "phi series at %g" % zz)
    for zz in (-20.0, -1.5, -0.3, 0.7, 2.0):
        _close(orc.phi(zz), np.expm1(zz) / zz, 1e-15, 0.0, "phi at %g" % zz)


def pin_zoh_closed_form(orc, seed=41):
    """Constant dt, x, B: L ZOH steps land exactly on the continuous solution
    h(T) = e^{AT} h0 + (e^{AT} - 1)/A B x at T = L dt, for any L; y reads it."""
    r = _rng(seed)
    N, L = 4, 37
    A = -np.exp(r.standard_normal((1, N)))
    B = r.standard_normal(N)
    C = r.standard_normal(N)
    h0 = r.standard_normal((1, 1, N))
    dt, xv, Dv = 0.07, 0.8, 1.3
    x = np.full((1, L, 1), xv)
    out, fs = orc.selective_scan(x, np.full((1, L, 1), dt), A, np.tile(B, (1, L, 1)),
                                 np.tile(C, (1, L, 1)), D=np.array([Dv]), h0=h0, zoh=True)
    for k in (1, 5, L):
        T = k * dt
        hk = np.exp(A[0] * T) * h0[0, 0] + np.expm1(A[0] * T) / A[0] * B * xv
        if k == L:
            _close(fs[0, 0], hk, 1e-12, 1e-14, "ZOH final state vs continuous solution")
        _close(out[0, k - 1, 0], C @ hk + Dv * xv, 1e-12, 1e-14, "ZOH y_%d" % k)


def pin_zoh_ode(orc, seed=42):
    """Per-token inputs: each ZOH step equals integrating h' = A h + B_t x_t over
    [0, dt_t] numerically (scipy solve_ivp, rtol 1e-12); first-order dt B does not."""
    from scipy.integrate import solve_ivp
    r = _rng(seed)
    N, L = 3, 12
    A = -np.exp(r.standard_normal((1, N)) * 0.7)
    B = r.standard_normal((1, L, N))
    C = r.standard_normal((1, L, N))
    x = r.standard_normal((1, L, 1))
    dt = r.uniform(0.05, 0.6, (1, L, 1))
    h = r.standard_normal(N)
    out, fs = orc.selective_scan(x, dt, A, B, C, h0=h[None, None, :], zoh=True)
    for t in range(L):
        sol = solve_ivp(lambda _, y: A[0] * y + B[0, t] * x[0, t, 0], (0.0, dt[0, t, 0]), h,
                        rtol=1e-12, atol=1e-14, method="DOP853")
        h = sol.y[:, -1]
        _close(out[0, t, 0], C[0, t] @ h, 1e-9, 1e-11, "ZOH y_%d vs ODE" % t)
    _close(fs[0, 0], h, 1e-9, 1e-11, "ZOH final state vs ODE")
    out1, _ = orc.selective_scan(x, dt, A, B, C, h0=None)
    outz, _ = orc.selective_scan(x, dt, A, B, C, h0=None, zoh=True)
    assert np.abs(out1 - outz).max() > 1e-3, "first-order and ZOH must differ at these steps"


def pin_zoh_library(orc, seed=46):
    """One ZOH step equals SciPy's zero-order-hold discretization of the
    continuous system (scipy.signal.cont2discrete, method "zoh", which takes the
    matrix exponential of the augmented [[A, B], [0, 0]] dt): h1 = Ad h0 + Bd x."""
    from scipy.signal import cont2discrete
    r = _rng(seed)
    N = 5
    for dt in (1e-3, 0.07, 0.9):
        A = -np.exp(r.standard_normal(N))
        B = r.standard_normal(N)
        h0 = r.standard_normal(N)
        xv = r.standard_normal()
        Ad, Bd, _, _, _ = cont2discrete((np.diag(A), B[:, None], np.ones((1, N)), np.zeros((1, 1))),
                                        dt, method="zoh")
        _, fs = orc.selective_scan(np.full((1, 1, 1), xv), np.full((1, 1, 1), dt), A[None, :],
                                   B[None, None, :], np.zeros((1, 1, N)), h0=h0[None, None, :],
                                   zoh=True)
        _close(fs[0, 0], Ad @ h0 + Bd[:, 0] * xv, 1e-11, 1e-13, "ZOH step vs cont2discrete, dt=%g" % dt)


def pin_zoh_small_step(orc, seed=43):
    """As dt -> 0, ZOH tends to the first-order form: the difference per step is
    dt B x (phi(dt A) - 1) ~ dt^2 A B x / 2."""
    r = _rng(seed)
    c = _random_case(r, batch=1, L=16, dim=3, N=4)
    small = np.full_like(c["delta"], 1e-6)
    o1, f1 = orc.selective_scan(c["x"], small, c["A"], c["B"], c["C"], D=c["D"])
    oz, fz = orc.selective_scan(c["x"], small, c["A"], c["B"], c["C"], D=c["D"], zoh=True)
    _close(oz, o1, 1e-5, 1e-12, "ZOH -> first order as dt -> 0")
    assert np.abs(fz - f1).max() > 0.0


def pin_zoh_decode(orc, seed=44):
    """The ZOH decode step is one token of the ZOH scan from the same state."""
    r = _rng(seed)
    c = _random_case(r, batch=2, L=1, dim=3, N=4)
    st = r.standard_normal((2, 3, 4))
    oz, fz = orc.selective_scan(c["x"], c["delta"], c["A"], c["B"], c["C"], D=c["D"], z=c["z"],
                                h0=st, zoh=True)
    od, sd = orc.state_update(st, c["x"][:, 0], c["delta"][:, 0], c["A"], c["B"][:, 0],
                              c["C"][:, 0], D=c["D"], z=c["z"][:, 0], zoh=True)
    _close(od, oz[:, 0], 1e-14, 1e-15, "ZOH decode y")
    _close(sd, fz, 1e-14, 1e-15, "ZOH decode state")


# --------------------------------------------------------------------------
# per-channel B, C ("Mamba: State Space Models Challenge Transformers",
# "Selective Scan Algorithm": B, C of shape [B, L, D, N] in its docstring)
# --------------------------------------------------------------------------
def pin_bc_per_channel(orc, seed=45):
    """Per-channel B, C: each channel equals the explicit unrolled sum with its
    own rows; rows equal across channels give the shared-B, C scan exactly."""
    r = _rng(seed)
    c = _random_case(r, batch=2, L=10, dim=3, N=4)
    B4 = r.standard_normal((2, 10, 3, 4))
    C4 = r.standard_normal((2, 10, 3, 4))
    bias = r.standard_normal(3) * 0.2
    h0 = r.standard_normal((2, 3, 4))
    out, fs = orc.selective_scan_bcd(c["x"], c["delta"], c["A"], B4, C4, D=c["D"], z=c["z"],
                                     delta_bias=bias, delta_softplus=True, h0=h0)
    for d in range(3):
        sl = slice(d, d + 1)
        y, hL = _unrolled(c["x"][:, :, sl], c["delta"][:, :, sl], c["A"][sl], B4[:, :, d],
                          C4[:, :, d], c["D"][sl], c["z"][:, :, sl], bias[sl], True, h0[:, sl])
        _close(out[:, :, sl], y, 1e-12, 1e-13, "per-channel y, channel %d" % d)
        _close(fs[:, sl], hL, 1e-12, 1e-13, "per-channel final state, channel %d" % d)
    Bs = np.repeat(c["B"][:, :, None, :], 3, 2)   # the shared rows, once per channel
    Cs = np.repeat(c["C"][:, :, None, :], 3, 2)
    o1, f1 = orc.selective_scan(c["x"][:, :10], c["delta"][:, :10], c["A"], c["B"][:, :10],
                                c["C"][:, :10], D=c["D"], h0=h0)
    o2, f2 = orc.selective_scan_bcd(c["x"][:, :10], c["delta"][:, :10], c["A"],
                                    Bs[:, :10], Cs[:, :10], D=c["D"], h0=h0)
    assert np.array_equal(o1, o2) and np.array_equal(f1, f2), "shared rows = shared B, C"



# --------------------------------------------------------------------------
# gradients of the variants (exact zero-order hold, per-channel B, C)
# --------------------------------------------------------------------------
def pin_phi_prime(orc):
    """phi'(z) = integral_0^1 s e^{zs} ds, since phi(z) is the mean of e^{zs}
    over s in [0, 1]: 1/2 at 0; adaptive quadrature on both sides of |z| = 1
    (where the oracle switches from its series to the closed form); and the
    central difference of numpy's expm1(z)/z."""
    from scipy.integrate import quad
    assert orc.phi_prime(0.0) == 0.5
    for zz in (-30.0, -4.0, -1.2, -1.0, -0.999, -0.3, -1e-4, 1e-6, 0.5, 1.0, 1.001, 3.0):
        val, _ = quad(lambda sv: sv * np.exp(zz * sv), 0.0, 1.0, epsabs=0.0, epsrel=1e-13)
        _close(orc.phi_prime(zz), val, 1e-12, 0.0, "phi' at %g vs quadrature" % zz)
    for zz in (-2.5, -0.7, 0.4):
        hh = 1e-5
        fd = (np.expm1(zz + hh) / (zz + hh) - np.expm1(zz - hh) / (zz - hh)) / (2 * hh)
        _close(orc.phi_prime(zz), fd, 1e-8, 0.0, "phi' at %g vs central difference" % zz)


def _variant_case(r, shape, softplus, full, per_channel):
    c, dout, dhf = _bwd_case(r, *shape, softplus, full)
    if per_channel:
        batch, L, dim, N = shape
        c["B"] = r.standard_normal((batch, L, dim, N))
        c["C"] = r.standard_normal((batch, L, dim, N))
    return c, dout, dhf


def _variant_grads(orc, c, dout, dhf, softplus, zoh, per_channel):
    fn = orc.selective_scan_bcd_bwd if per_channel else orc.selective_scan_bwd
    return fn(c["x"], c["delta"], c["A"], c["B"], c["C"], dout, D=c["D"], z=c["z"],
              delta_bias=c["delta_bias"], delta_softplus=softplus, h0=c["h0"], dh_final=dhf,
              zoh=zoh)


def pin_bwd_variants_finite_differences(orc, seed=51):
    """The gradients of the zero-order-hold scan and of the per-channel B, C scan
    equal the central differences of the oracle's own forward of that variant
    (itself pinned to the ODE and to the unrolled sum)."""
    r = _rng(seed)
    for zoh, per_channel, softplus, full, shape in ((True, False, True, True, (2, 4, 2, 3)),
                                                    (True, False, False, False, (1, 5, 2, 2)),
                                                    (False, True, True, True, (1, 4, 3, 2)),
                                                    (True, True, True, True, (1, 3, 2, 3))):
        c, dout, dhf = _variant_case(r, shape, softplus, full, per_channel)
        g = _variant_grads(orc, c, dout, dhf, softplus, zoh, per_channel)
        fwd = orc.selective_scan_bcd if per_channel else orc.selective_scan

        def loss(**kw):
            a = dict(c)
            a.update(kw)
            out, fs = fwd(a["x"], a["delta"], a["A"], a["B"], a["C"], D=a["D"], z=a["z"],
                          delta_bias=a["delta_bias"], delta_softplus=softplus, h0=a["h0"],
                          zoh=zoh)
            return float((out * dout).sum() + (0.0 if dhf is None else (fs * dhf).sum()))

        eps = 1e-6
        for name, arr in c.items():
            if arr is None:
                continue
            fd = np.zeros_like(arr)
            for i in np.ndindex(arr.shape):
                p, m = arr.copy(), arr.copy()
                p[i] += eps
                m[i] -= eps
                fd[i] = (loss(**{name: p}) - loss(**{name: m})) / (2 * eps)
            _close(g[_GRAD_OF[name]], fd, 1e-6, 1e-7,
                   "d%s vs finite differences (zoh=%s, per-channel=%s)" % (name, zoh, per_channel))


def pin_bwd_variants_autograd(orc, seed=52):
    """The gradients of both variants equal PyTorch autograd through a plain
    float64 loop (the zero-order hold written with torch.expm1)."""
    import torch
    r = _rng(seed)
    for zoh, per_channel, softplus, full, shape in ((True, False, True, True, (2, 7, 3, 4)),
                                                    (True, False, False, True, (1, 6, 2, 5)),
                                                    (False, True, True, True, (2, 6, 3, 4)),
                                                    (True, True, False, False, (1, 5, 2, 3))):
        c, dout, dhf = _variant_case(r, shape, softplus, full, per_channel)
        tens = {k: (None if v is None else torch.tensor(v, requires_grad=True))
                for k, v in c.items()}
        out, fs = _torch_scan(tens["x"], tens["delta"], tens["A"], tens["B"], tens["C"],
                              tens["D"], tens["z"], tens["delta_bias"], softplus, tens["h0"],
                              zoh=zoh)
        loss = (out * torch.tensor(dout)).sum()
        if dhf is not None:
            loss = loss + (fs * torch.tensor(dhf)).sum()
        loss.backward()
        g = _variant_grads(orc, c, dout, dhf, softplus, zoh, per_channel)
        for name, t in tens.items():
            if t is not None:
                _close(g[_GRAD_OF[name]], t.grad.numpy(), 1e-10, 1e-12,
                       "d%s vs autograd (zoh=%s, per-channel=%s)" % (name, zoh, per_channel))


def pin_bwd_per_channel_shared_rows(orc, seed=53):
    """Per-channel rows that repeat the shared B, C rows give the shared scan's
    gradients: dB, dC summed over channels equal the shared dB, dC, and every
    other gradient is unchanged (with and without the zero-order hold)."""
    r = _rng(seed)
    for zoh in (False, True):
        c, dout, dhf = _bwd_case(r, 2, 6, 3, 4, True, True)
        g = orc.selective_scan_bwd(c["x"], c["delta"], c["A"], c["B"], c["C"], dout, D=c["D"],
                                   z=c["z"], delta_bias=c["delta_bias"], delta_softplus=True,
                                   h0=c["h0"], dh_final=dhf, zoh=zoh)
        B4 = np.repeat(c["B"][:, :, None, :], 3, 2)
        C4 = np.repeat(c["C"][:, :, None, :], 3, 2)
        g4 = orc.selective_scan_bcd_bwd(c["x"], c["delta"], c["A"], B4, C4, dout, D=c["D"],
                                        z=c["z"], delta_bias=c["delta_bias"],
                                        delta_softplus=True, h0=c["h0"], dh_final=dhf, zoh=zoh)
        _close(g4["dB"].sum(2), g["dB"], 1e-12, 1e-13, "per-channel dB summed (zoh=%s)" % zoh)
        _close(g4["dC"].sum(2), g["dC"], 1e-12, 1e-13, "per-channel dC summed (zoh=%s)" % zoh)
        for k in ("dx", "ddelta", "dz", "dA", "dD", "ddelta_bias", "dh0"):
            _close(g4[k], g[k], 1e-12, 1e-13, "%s per-channel vs shared (zoh=%s)" % (k, zoh))



# --------------------------------------------------------------------------
# Mamba-2's SSD layer ("Mamba: State Space Models Challenge Transformers",
# "Mamba-2: Improved Architecture"; "State Space Models and Mamba", "Mamba 2 and
# Hybrid Architectures": the SSM as a structured matrix multiplication)
# --------------------------------------------------------------------------
def _ssd_case(r, batch, L, H, P, G, N, full):
    return {"x": r.standard_normal((batch, L, H, P)),
            "dt": (r.standard_normal((batch, L, H)) * 0.5 if full
                   else r.uniform(0.02, 0.3, (batch, L, H))),
            "A": -np.exp(r.standard_normal(H) * 0.5),
            "B": r.standard_normal((batch, L, G, N)), "C": r.standard_normal((batch, L, G, N)),
            "D": r.uniform(0.5, 1.5, H) if full else None,
            "dt_bias": r.standard_normal(H) * 0.3 if full else None,
            "h0": r.standard_normal((batch, H, P, N)) if full else None}


def pin_ssd_as_selective_scan(orc, seed=61):
    """SSD is the selective scan with one decay per head: channel d = hd * P + p
    of a per-channel-B, C scan with A[d, :] = A[hd], delta = dt of its head and
    the rows of its head's group gives the same y and final state; with one
    group the shared-B, C scan does."""
    r = _rng(seed)
    for (batch, L, H, P, G, N), full in (((2, 9, 4, 3, 2, 5), True), ((1, 7, 2, 4, 1, 3), False)):
        c = _ssd_case(r, batch, L, H, P, G, N, full)
        y, fs = orc.ssd(c["x"], c["dt"], c["A"], c["B"], c["C"], D=c["D"], dt_bias=c["dt_bias"],
                        dt_softplus=full, h0=c["h0"])
        head = np.repeat(np.arange(H), P)             # head of channel d
        grp = head // (H // G)
        x = c["x"].reshape(batch, L, H * P)
        delta = c["dt"][:, :, head]
        A = np.repeat(c["A"][head][:, None], N, 1)
        rep = lambda a: None if a is None else a[head]
        h0 = None if c["h0"] is None else c["h0"].reshape(batch, H * P, N)
        out, f = orc.selective_scan_bcd(x, delta, A, c["B"][:, :, grp], c["C"][:, :, grp],
                                        D=rep(c["D"]), delta_bias=rep(c["dt_bias"]),
                                        delta_softplus=full, h0=h0)
        _close(y.reshape(batch, L, H * P), out, 1e-12, 1e-13, "SSD y vs per-channel scan")
        _close(fs.reshape(batch, H * P, N), f, 1e-12, 1e-13, "SSD state vs per-channel scan")
        if G == 1:
            o1, f1 = orc.selective_scan(x, delta, A, c["B"][:, :, 0], c["C"][:, :, 0],
                                        D=rep(c["D"]), delta_bias=rep(c["dt_bias"]),
                                        delta_softplus=full, h0=h0)
            _close(y.reshape(batch, L, H * P), o1, 1e-12, 1e-13, "SSD y vs shared-B scan")


def pin_ssd_matrix_form(orc, seed=62):
    """The dual form: per batch row and head, y = M X + D X (+ the decayed h0
    read by C) with the masked matrix M[t, s] = (C_t . B_s) e^{A (S_t - S_s)}
    dt_s for s <= t and 0 above the diagonal, S the running sum of dt; the final
    state is e^{A S_L} h0 + sum_s e^{A (S_L - S_s)} dt_s x_s B_s^T."""
    r = _rng(seed)
    for (batch, L, H, P, G, N), full in (((2, 12, 4, 3, 2, 6), True), ((1, 10, 3, 2, 3, 4), False),
                                         ((1, 8, 2, 5, 1, 3), True)):
        c = _ssd_case(r, batch, L, H, P, G, N, full)
        y, fs = orc.ssd(c["x"], c["dt"], c["A"], c["B"], c["C"], D=c["D"], dt_bias=c["dt_bias"],
                        dt_softplus=full, h0=c["h0"])
        for b in range(batch):
            for hd in range(H):
                g = hd // (H // G)
                v = c["dt"][b, :, hd] + (c["dt_bias"][hd] if c["dt_bias"] is not None else 0.0)
                dt = np.logaddexp(0.0, v) if full else v
                S = np.cumsum(dt)
                Bm, Cm, X = c["B"][b, :, g], c["C"][b, :, g], c["x"][b, :, hd]
                M = np.tril((Cm @ Bm.T) * np.exp(c["A"][hd] * (S[:, None] - S[None, :]))
                            * dt[None, :])
                want = M @ X
                hL = (np.exp(c["A"][hd] * (S[-1] - S)) * dt)[:, None, None] \
                    * (X[:, :, None] * Bm[:, None, :])
                hL = hL.sum(0)
                if c["h0"] is not None:
                    want += np.exp(c["A"][hd] * S)[:, None] * (Cm @ c["h0"][b, hd].T)
                    hL += np.exp(c["A"][hd] * S[-1]) * c["h0"][b, hd]
                if c["D"] is not None:
                    want += c["D"][hd] * X
                _close(y[b, :, hd], want, 1e-10, 1e-12, "SSD y vs matrix form, b=%d head=%d" % (b, hd))
                _close(fs[b, hd], hL, 1e-10, 1e-12, "SSD state vs matrix form, b=%d head=%d" % (b, hd))



def pin_bc_per_channel_decode(orc, seed=47):
    """The per-channel decode step is one token of the per-channel scan from the
    same state (with and without the zero-order hold), and with rows equal
    across channels it is the shared-B, C step exactly."""
    r = _rng(seed)
    c = _random_case(r, batch=2, L=1, dim=3, N=4)
    st = r.standard_normal((2, 3, 4))
    B4 = r.standard_normal((2, 1, 3, 4))
    C4 = r.standard_normal((2, 1, 3, 4))
    bias = r.standard_normal(3) * 0.2
    for zoh in (False, True):
        oz, fz = orc.selective_scan_bcd(c["x"], c["delta"], c["A"], B4, C4, D=c["D"], z=c["z"],
                                        delta_bias=bias, delta_softplus=True, h0=st, zoh=zoh)
        od, sd = orc.state_update_bcd(st, c["x"][:, 0], c["delta"][:, 0], c["A"], B4[:, 0],
                                      C4[:, 0], D=c["D"], z=c["z"][:, 0], delta_bias=bias,
                                      delta_softplus=True, zoh=zoh)
        _close(od, oz[:, 0], 1e-14, 1e-15, "per-channel decode y (zoh=%s)" % zoh)
        _close(sd, fz, 1e-14, 1e-15, "per-channel decode state (zoh=%s)" % zoh)
    Bs = np.repeat(c["B"][:, 0, None, :], 3, 1)
    Cs = np.repeat(c["C"][:, 0, None, :], 3, 1)
    o1, s1 = orc.state_update(st, c["x"][:, 0], c["delta"][:, 0], c["A"], c["B"][:, 0],
                              c["C"][:, 0], D=c["D"])
    o2, s2 = orc.state_update_bcd(st, c["x"][:, 0], c["delta"][:, 0], c["A"], Bs, Cs, D=c["D"])
    assert np.array_equal(o1, o2) and np.array_equal(s1, s2), "shared rows = shared B, C step"



def pin_ssd_chunked_form(orc, seed=63):
    """The chunked form of the matrix product: per chunk of Q tokens (the last one
    ragged), y = tril((C Bᵀ) ∘ e^{A (s_t - s_u)} dt_u) X (the chunk's own tokens,
    s the running sum of dt inside the chunk) + e^{A s_t} C_t h_inᵀ (the state
    carried in) + D x, and the state passed on is e^{A s_Q} h_in + Σ_u
    e^{A (s_Q - s_u)} dt_u x_u B_uᵀ. Every chunk size gives the oracle's y and
    final state."""
    r = _rng(seed)
    batch, L, H, P, G, N = 2, 23, 4, 3, 2, 5
    c = _ssd_case(r, batch, L, H, P, G, N, True)
    y, fs = orc.ssd(c["x"], c["dt"], c["A"], c["B"], c["C"], D=c["D"], dt_bias=c["dt_bias"],
                    dt_softplus=True, h0=c["h0"])
    for Q in (1, 4, 7, 23, 32):
        for b in range(batch):
            for hd in range(H):
                g = hd // (H // G)
                a = c["A"][hd]
                dt_all = np.logaddexp(0.0, c["dt"][b, :, hd] + c["dt_bias"][hd])
                h = c["h0"][b, hd].copy()                    # [P, N]
                yc = np.zeros((L, P))
                for t0 in range(0, L, Q):
                    t1 = min(L, t0 + Q)
                    dt = dt_all[t0:t1]
                    sl = np.cumsum(dt)
                    Bm, Cm, X = c["B"][b, t0:t1, g], c["C"][b, t0:t1, g], c["x"][b, t0:t1, hd]
                    M = np.tril((Cm @ Bm.T) * np.exp(a * (sl[:, None] - sl[None, :])) * dt[None, :])
                    yc[t0:t1] = M @ X + np.exp(a * sl)[:, None] * (Cm @ h.T) + c["D"][hd] * X
                    w = np.exp(a * (sl[-1] - sl)) * dt
                    h = np.exp(a * sl[-1]) * h + (X * w[:, None]).T @ Bm
                _close(yc, y[b, :, hd], 1e-10, 1e-12, "SSD chunked y, Q=%d b=%d head=%d" % (Q, b, hd))
                _close(h, fs[b, hd], 1e-10, 1e-12, "SSD chunked state, Q=%d b=%d head=%d" % (Q, b, hd))


ALL_PINS = [
    pin_ssd_as_selective_scan,
    pin_ssd_matrix_form,
    pin_ssd_chunked_form,
    pin_conv_bwd,
    pin_conv_scan_bwd,
    pin_phi_prime,
    pin_bwd_variants_finite_differences,
    pin_bwd_variants_autograd,
    pin_bwd_per_channel_shared_rows,
    pin_bc_per_channel,
    pin_bc_per_channel_decode,
    pin_phi,
    pin_zoh_closed_form,
    pin_zoh_ode,
    pin_zoh_small_step,
    pin_zoh_library,
    pin_zoh_decode,
    pin_bwd_finite_differences,
    pin_bwd_autograd,
    pin_bwd_channel_sums,
    pin_conv_library,
    pin_conv_taps,
    pin_conv_causal,
    pin_worked_example_core,
    pin_worked_example_selective_path,
    pin_lti_convolution,
    pin_unrolled_sum,
    pin_linearity,
    pin_delta_zero,
    pin_delta_large,
    pin_n1_closed_form,
    pin_split_resume,
    pin_decode_equals_scan,
    pin_softplus_silu,
    pin_thread_invariance,
]
