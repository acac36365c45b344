"""Seeded synthetic inputs for the selective scan and the recurrent step.

This module draws random inputs and rounds them to the I/O dtype. It holds none
of the scan's arithmetic. The CUDA-path tests, the oracle tests and the
benchmark all take their inputs from here, so that both sides see bit-identical
values.

Recipe (shapes follow the pages' model sizes: d_state 16, expand 2, d_model
768 / 1024 / 2560, as in "State Space Models -- Mamba, S4, and Beyond",
``MambaBlock`` / ``MambaLanguageModel`` and "Mamba: State Space Models
Challenge Transformers", "Code Example"):

* numpy ``Generator(PCG64(seed))``; every value is drawn in float64 and then
  rounded ONCE, round-to-nearest-even, to its storage type (bf16 or fp32 for
  the I/O tensors x, delta, z, B, C; fp32 for A, D, delta_bias and the state).
* Draw order: x, z, delta (or u), bias, A, B, C, D, state.
* "log-uniform in [lo, hi]" means exp(U(ln lo, ln hi)) per element.
* ``A_kind="s4d"``: A[d, n] = -(n + 1) (the pages' ``A_log = log(arange(1,
  N+1))`` initialisation, A = -exp(A_log)). ``A_kind="lognormal"``:
  A = -exp(N(0, 0.5^2)).
* ``delta_kind="loguniform"``: delta log-uniform in [lo, hi], no softplus.
  ``delta_kind="softplus_bias"``: u ~ N(0, 0.5^2) and bias[d] = log(expm1(s_d))
  with s_d log-uniform in [lo, hi], so that softplus(bias) = s_d; the scan then
  takes delta = softplus(u + bias).
* D = 1, or D ~ U(0.5, 1.5).

bf16 values are carried as uint16 bit patterns (numpy has no bf16); ``widen``
turns any stored array back into float64 exactly.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np

IO_DTYPES = ("f32", "bf16")


# --------------------------------------------------------------------------
# exact rounding and widening
# --------------------------------------------------------------------------
def round_bf16_bits(v: np.ndarray) -> np.ndarray:
    """Round float64 values once, to nearest even, to bf16; return uint16 bits.

    bf16 keeps 8 significant bits, float64 keeps 53, so rounding drops the low
    45 mantissa bits: add 2**44 - 1 plus the lowest kept bit, then clear the
    dropped bits (the usual integer round-half-even; a carry into the exponent
    is the correct result). That holds wherever the result is a normal bf16
    number; the rare values below 2**-126 take the slower exact path, where
    v = m * 2**e and the bf16 value is rint(m * 2**8) * 2**(e - 8) with the
    quantum floored at the smallest bf16 subnormal, 2**-133.
    """
    v = np.ascontiguousarray(np.asarray(v, dtype=np.float64))
    if not np.all(np.isfinite(v)):
        raise ValueError("non-finite input")
    bits = v.view(np.uint64)
    keep_lsb = (bits >> np.uint64(45)) & np.uint64(1)
    rb = (bits + (np.uint64((1 << 44) - 1) + keep_lsb)) & np.uint64(~((1 << 45) - 1) & 0xFFFFFFFFFFFFFFFF)
    r = rb.view(np.float64)
    tiny = np.abs(v) < 2.0 ** -126
    if np.any(tiny):
        vt = v[tiny]
        _, e = np.frexp(vt)
        q = np.maximum(e.astype(np.int64) - 8, -133)
        r = r.copy()
        r[tiny] = np.ldexp(np.rint(np.ldexp(vt, -q)), q)
    if np.any(np.abs(r) > 3.3895313892515355e38):
        raise ValueError("value out of bf16 range")
    bits32 = r.astype(np.float32).view(np.uint32)  # exact: r is a bf16 value
    return (bits32 >> np.uint32(16)).astype(np.uint16)


def _round_bf16_bits_slow(v: np.ndarray) -> np.ndarray:
    """Reference form of round_bf16_bits (frexp / rint / ldexp), for tests."""
    v = np.asarray(v, dtype=np.float64)
    _, e = np.frexp(v)
    q = np.maximum(e.astype(np.int64) - 8, -133)
    r = np.ldexp(np.rint(np.ldexp(v, -q)), q)
    return (r.astype(np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def store(v: np.ndarray, io: str) -> np.ndarray:
    """Round float64 to the storage type of ``io`` ('f32' or 'bf16' bits)."""
    if io == "f32":
        return np.asarray(v, dtype=np.float64).astype(np.float32)
    if io == "bf16":
        return round_bf16_bits(v)
    raise ValueError("io must be 'f32' or 'bf16'")


def widen(a: Optional[np.ndarray]) -> Optional[np.ndarray]:
    """Exact float64 value of a stored array (uint16 = bf16 bits)."""
    if a is None:
        return None
    if a.dtype == np.uint16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a, dtype=np.float64)


# --------------------------------------------------------------------------
# workload descriptions
# --------------------------------------------------------------------------
@dataclasses.dataclass(frozen=True)
class ScanSpec:
    """One selective-scan workload: sizes and the distributions of its inputs."""
    batch: int
    L: int
    dim: int
    N: int = 16
    io: str = "bf16"
    delta_kind: str = "loguniform"      # or "softplus_bias"
    delta_lo: float = 1e-3
    delta_hi: float = 1e-1
    A_kind: str = "s4d"                 # or "lognormal"
    D_kind: str = "one"                 # "one", "uniform" or "none"
    gate: bool = True                   # z given
    final_state: bool = True
    seed: int = 0

    @property
    def delta_softplus(self) -> bool:
        return self.delta_kind == "softplus_bias"

    @property
    def elements(self) -> int:
        return self.batch * self.L * self.dim


@dataclasses.dataclass(frozen=True)
class DecodeSpec:
    """Recurrent decode: `steps` single-token updates of a [batch, dim, N] state."""
    batch: int
    dim: int
    N: int = 16
    steps: int = 64
    io: str = "bf16"
    delta_lo: float = 1e-3
    delta_hi: float = 1e-1
    A_kind: str = "s4d"
    D_kind: str = "one"
    gate: bool = True
    state_init: str = "normal"          # "normal" (N(0,1)) or "zero"
    seed: int = 0


# The five workloads, named by what they are. Seeds are 1000 + position.
WORKLOADS: Dict[str, object] = {
    "scan_f32_b2_L256_d16": ScanSpec(2, 256, 16, io="f32", seed=1001),
    "scan_bf16_b4_L2048_d1536_softplus": ScanSpec(
        4, 2048, 1536, io="bf16", delta_kind="softplus_bias", A_kind="lognormal",
        D_kind="uniform", final_state=False, seed=1002),
    "scan_bf16_b8_L4096_d2048": ScanSpec(8, 4096, 2048, io="bf16", seed=1003),
    "scan_bf16_b1_L131072_d5120": ScanSpec(
        1, 131072, 5120, io="bf16", delta_lo=1e-4, delta_hi=1e-2, seed=1004),
    "decode_bf16_b256_d5120_x64": DecodeSpec(256, 5120, steps=64, seed=1005),
}


@dataclasses.dataclass(frozen=True)
class SsdSpec:
    """One Mamba-2 SSD workload: x [batch, L, H, P], dt [batch, L, H], B, C
    [batch, L, G, N]. dt = softplus(u + bias) with u ~ N(0, 0.5^2) and
    softplus(bias[hd]) log-uniform in [dt_lo, dt_hi]; A[hd] = -U(1, 16); x, B,
    C ~ N(0, 1); D ~ U(0.5, 1.5); h0 (when drawn) ~ N(0, 1)."""
    batch: int
    L: int
    H: int = 8
    P: int = 64
    G: int = 1
    N: int = 128
    dt_lo: float = 1e-3
    dt_hi: float = 1e-1
    seed: int = 0

    @property
    def elements(self) -> int:
        return self.batch * self.L * self.H * self.P


# The SSD layer at the pages' Mamba-2 sizes (8 heads of 64 channels, d_state 128).
SSD_WORKLOADS: Dict[str, SsdSpec] = {
    "ssd_bf16_b16_L8192_h8_p64_n128": SsdSpec(16, 8192, seed=1101),
}


def _loguniform(rng, lo, hi, size):
    return np.exp(np.log(lo) + (np.log(hi) - np.log(lo)) * rng.random(size))


def _normal_chunked(rng, size, scale=1.0, io="bf16", chunk=1 << 24):
    """Draw N(0, scale^2) in float64 and round to io, chunk by chunk (the
    stream is identical to one large draw; only peak memory differs)."""
    n = int(np.prod(size))
    out = np.empty(n, dtype=np.uint16 if io == "bf16" else np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = store(rng.standard_normal(e - s) * scale, io)
    return out.reshape(size)


def _loguniform_chunked(rng, lo, hi, size, io, chunk=1 << 24):
    n = int(np.prod(size))
    out = np.empty(n, dtype=np.uint16 if io == "bf16" else np.float32)
    for s in range(0, n, chunk):
        e = min(n, s + chunk)
        out[s:e] = store(_loguniform(rng, lo, hi, e - s), io)
    return out.reshape(size)


def _A(rng, kind, dim, N):
    if kind == "s4d":
        return np.tile(-(np.arange(N, dtype=np.float64) + 1.0), (dim, 1)).astype(np.float32)
    if kind == "lognormal":
        return (-np.exp(rng.standard_normal((dim, N)) * 0.5)).astype(np.float32)
    raise ValueError(kind)


def _D(rng, kind, dim):
    if kind == "one":
        return np.ones(dim, dtype=np.float32)
    if kind == "uniform":
        return rng.uniform(0.5, 1.5, dim).astype(np.float32)
    if kind == "none":
        return None
    raise ValueError(kind)


def make_scan_inputs(spec: ScanSpec, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw one set of scan inputs for ``spec``.

    Returns a dict with x, delta, z (or None), B, C (stored I/O dtype), A
    [dim, N] fp32, D [dim] fp32 (or None), delta_bias [dim] fp32 (or None).
    """
    rng = np.random.Generator(np.random.PCG64(spec.seed if seed is None else seed))
    b, L, d, N, io = spec.batch, spec.L, spec.dim, spec.N, spec.io
    out: Dict[str, Optional[np.ndarray]] = {}
    out["x"] = _normal_chunked(rng, (b, L, d), 1.0, io)
    out["z"] = _normal_chunked(rng, (b, L, d), 1.0, io) if spec.gate else None
    if spec.delta_kind == "loguniform":
        out["delta"] = _loguniform_chunked(rng, spec.delta_lo, spec.delta_hi, (b, L, d), io)
        out["delta_bias"] = None
    elif spec.delta_kind == "softplus_bias":
        out["delta"] = _normal_chunked(rng, (b, L, d), 0.5, io)
        s = _loguniform(rng, spec.delta_lo, spec.delta_hi, d)
        out["delta_bias"] = np.log(np.expm1(s)).astype(np.float32)
    else:
        raise ValueError(spec.delta_kind)
    out["A"] = _A(rng, spec.A_kind, d, N)
    out["B"] = _normal_chunked(rng, (b, L, N), 1.0, io)
    out["C"] = _normal_chunked(rng, (b, L, N), 1.0, io)
    out["D"] = _D(rng, spec.D_kind, d)
    return out


def make_decode_inputs(spec: DecodeSpec, seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw the inputs of ``spec.steps`` decode steps.

    Per-step tensors carry a leading step axis: x, delta, z [steps, batch, dim];
    B, C [steps, batch, N] (stored I/O dtype). A [dim, N], D [dim] fp32;
    state0 [batch, dim, N] fp32.
    """
    rng = np.random.Generator(np.random.PCG64(spec.seed if seed is None else seed))
    S, b, d, N, io = spec.steps, spec.batch, spec.dim, spec.N, spec.io
    out: Dict[str, Optional[np.ndarray]] = {}
    out["x"] = _normal_chunked(rng, (S, b, d), 1.0, io)
    out["z"] = _normal_chunked(rng, (S, b, d), 1.0, io) if spec.gate else None
    out["delta"] = _loguniform_chunked(rng, spec.delta_lo, spec.delta_hi, (S, b, d), io)
    out["delta_bias"] = None
    out["A"] = _A(rng, spec.A_kind, d, N)
    out["B"] = _normal_chunked(rng, (S, b, N), 1.0, io)
    out["C"] = _normal_chunked(rng, (S, b, N), 1.0, io)
    out["D"] = _D(rng, spec.D_kind, d)
    if spec.state_init == "normal":
        out["state0"] = rng.standard_normal((b, d, N)).astype(np.float32)
    else:
        out["state0"] = np.zeros((b, d, N), dtype=np.float32)
    return out


def make_conv_weights(dim: int, K: int = 4, bias: bool = True,
                      seed: int = 0) -> Tuple[np.ndarray, Optional[np.ndarray]]:
    """Taps [dim, K] and bias [dim] (or None) of a depthwise causal conv1d,
    fp32, drawn uniform in +-1/sqrt(K): the default initialisation range of a
    Conv1d whose fan-in is K (one input channel per group)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    bound = 1.0 / np.sqrt(K)
    w = rng.uniform(-bound, bound, (dim, K)).astype(np.float32)
    b = rng.uniform(-bound, bound, dim).astype(np.float32) if bias else None
    return w, b


def algorithmic_bytes_conv(batch: int, L: int, dim: int, K: int, io: str,
                           bias: bool = True) -> int:
    """Bytes the standalone conv1d + SiLU must move at least once: x read and u
    written per element, the taps (and bias) once."""
    es = 2 if io == "bf16" else 4
    return 2 * batch * L * dim * es + dim * K * 4 + (dim * 4 if bias else 0)


def make_bc_per_channel(spec: ScanSpec, seed: Optional[int] = None):
    """Per-channel B, C [batch, L, dim, N] ~ N(0, 1) in the stored I/O dtype
    (the rows a scan with per-channel B, C reads instead of the shared ones)."""
    rng = np.random.Generator(np.random.PCG64((spec.seed if seed is None else seed) + 500))
    shape = (spec.batch, spec.L, spec.dim, spec.N)
    return _normal_chunked(rng, shape, 1.0, spec.io), _normal_chunked(rng, shape, 1.0, spec.io)


def algorithmic_bytes_scan_bcd(spec: ScanSpec) -> int:
    """Bytes of the scan with per-channel B, C: x, delta, z, y per element and
    B, C rows per element (2 N values), A, D, bias once, the final state."""
    es = 2 if spec.io == "bf16" else 4
    per_elem = (4 if spec.gate else 3) * es + 2 * spec.N * es
    extra = spec.dim * spec.N * 4 + 2 * spec.dim * 4
    if spec.final_state:
        extra += spec.batch * spec.dim * spec.N * 4
    return spec.elements * per_elem + extra


def algorithmic_bytes_scan_bcd_bwd(spec: ScanSpec) -> int:
    """Bytes of the backward with per-channel B, C: x, delta, (z,) dout and the
    B, C rows read, dx, ddelta, (dz,) and the dB, dC rows written per element;
    the saved state before every 8th token read (16 fp32 per channel and 8
    tokens); A, D, bias read and dA, dD, dbias written once."""
    es = 2 if spec.io == "bf16" else 4
    scalars = (7 if spec.gate else 5) * es
    per_elem = scalars + 4 * spec.N * es + spec.N * 4 / 8
    extra = 2 * (spec.dim * spec.N * 4 + 2 * spec.dim * 4)
    return int(spec.elements * per_elem) + extra


def algorithmic_bytes_scan(spec: ScanSpec) -> int:
    """Bytes the scan must move at least once: x, delta, z read and y written
    per element; B and C per (b, t); A, D, delta_bias once; final_state written."""
    io_b = 4 if spec.io == "f32" else 2
    per_elem = (3 if spec.gate else 2) * io_b + io_b
    total = spec.elements * per_elem
    total += 2 * spec.batch * spec.L * spec.N * io_b
    total += spec.dim * spec.N * 4
    if spec.D_kind != "none":
        total += spec.dim * 4
    if spec.delta_kind == "softplus_bias":
        total += spec.dim * 4
    if spec.final_state:
        total += spec.batch * spec.dim * spec.N * 4
    return total


def algorithmic_bytes_decode_step(spec: DecodeSpec) -> int:
    """Bytes one decode step must move: state read + written, x/delta/z read and
    y written per (b, d), B and C per b, A and D once."""
    io_b = 4 if spec.io == "f32" else 2
    bd = spec.batch * spec.dim
    total = 2 * bd * spec.N * 4
    total += bd * ((3 if spec.gate else 2) * io_b + io_b)
    total += 2 * spec.batch * spec.N * io_b
    total += spec.dim * spec.N * 4
    if spec.D_kind != "none":
        total += spec.dim * 4
    return total


def make_ssd_inputs(spec: SsdSpec, with_h0: bool = False,
                    seed: Optional[int] = None) -> Dict[str, np.ndarray]:
    """Draw one set of SSD inputs (x, dt, B, C as bf16 bits; A, D, dt_bias fp32;
    h0 fp32 or None). Draw order: x, dt (u), bias, A, B, C, D, h0."""
    rng = np.random.Generator(np.random.PCG64(spec.seed if seed is None else seed))
    b, L, H, P, G, N = spec.batch, spec.L, spec.H, spec.P, spec.G, spec.N
    out: Dict[str, Optional[np.ndarray]] = {}
    out["x"] = _normal_chunked(rng, (b, L, H, P), 1.0, "bf16")
    out["dt"] = _normal_chunked(rng, (b, L, H), 0.5, "bf16")
    s = _loguniform(rng, spec.dt_lo, spec.dt_hi, H)
    out["dt_bias"] = np.log(np.expm1(s)).astype(np.float32)
    out["A"] = (-rng.uniform(1.0, 16.0, H)).astype(np.float32)
    out["B"] = _normal_chunked(rng, (b, L, G, N), 1.0, "bf16")
    out["C"] = _normal_chunked(rng, (b, L, G, N), 1.0, "bf16")
    out["D"] = rng.uniform(0.5, 1.5, H).astype(np.float32)
    out["h0"] = rng.standard_normal((b, H, P, N)).astype(np.float32) if with_h0 else None
    return out


def algorithmic_bytes_ssd(spec: SsdSpec, final_state: bool = True) -> int:
    """Bytes the SSD layer must move at least once: x read and y written per
    element, dt per (b, t, head), B and C per (b, t, group), A, D, bias once,
    the final state written."""
    b, L, H, P, G, N = spec.batch, spec.L, spec.H, spec.P, spec.G, spec.N
    total = 2 * b * L * H * P * 2 + b * L * H * 2 + 2 * b * L * G * N * 2 + 3 * H * 4
    if final_state:
        total += b * H * P * N * 4
    return total
