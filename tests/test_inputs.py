"""The seeded input generator: exact bf16 rounding, exact widening, and
reproducible streams."""
import numpy as np

from selective_state_space_119_b300 import inputs as I


def test_bf16_rounding_matches_exact_definition():
    rng = np.random.default_rng(3)
    v = np.concatenate([
        rng.standard_normal(1 << 18) * 3.0,
        np.exp(rng.uniform(np.log(1e-44), np.log(1e37), 1 << 16)) * rng.choice([-1.0, 1.0], 1 << 16),
        [0.0, -0.0, 1.0, -1.0, 2.0 ** -133, 2.0 ** -134, 3 * 2.0 ** -135, 2.0 ** -126],
    ])
    # exact ties halfway between two bf16 neighbours round to the even one
    base = I.bf16_bits_to_f32(np.arange(0x3f00, 0x3f40, dtype=np.uint16)).astype(np.float64)
    _, e = np.frexp(base)
    ties = base + np.ldexp(1.0, e - 9)          # bf16 quantum is 2**(e-8)
    v = np.concatenate([v, ties])
    fast, slow = I.round_bf16_bits(v), I._round_bf16_bits_slow(v)
    assert np.array_equal(fast, slow)
    # ties: the result is the even neighbour
    tb = I.round_bf16_bits(ties)
    assert np.all(tb & 1 == 0)
    lo = np.arange(0x3f00, 0x3f40, dtype=np.uint16)
    assert np.array_equal(tb, np.where(lo & 1, lo + 1, lo).astype(np.uint16))


def test_bf16_is_nearest():
    rng = np.random.default_rng(4)
    v = rng.standard_normal(4096) * 10
    r = I.widen(I.round_bf16_bits(v))
    bits = I.round_bf16_bits(v).astype(np.int32)
    up = I.widen(((bits + 1) & 0xFFFF).astype(np.uint16))
    dn = I.widen(((bits - 1) & 0xFFFF).astype(np.uint16))
    assert np.all(np.abs(r - v) <= np.abs(up - v)) and np.all(np.abs(r - v) <= np.abs(dn - v))


def test_widen_is_exact():
    bits = np.arange(0, 1 << 16, dtype=np.uint16)
    f = I.bf16_bits_to_f32(bits)
    fin = np.isfinite(f)
    assert np.array_equal(I.round_bf16_bits(f[fin].astype(np.float64)), bits[fin])


def test_streams_are_reproducible_and_chunk_invariant():
    spec = I.WORKLOADS["scan_f32_b2_L256_d16"]
    a, b = I.make_scan_inputs(spec), I.make_scan_inputs(spec)
    for k in a:
        if a[k] is not None:
            assert np.array_equal(a[k], b[k]), k
    r1 = np.random.Generator(np.random.PCG64(9))
    r2 = np.random.Generator(np.random.PCG64(9))
    x1 = I._normal_chunked(r1, (3, 1000), 1.0, "bf16", chunk=77)
    x2 = I.round_bf16_bits(r2.standard_normal(3000)).reshape(3, 1000)
    assert np.array_equal(x1, x2)


def test_workload_recipes():
    c2 = I.WORKLOADS["scan_bf16_b4_L2048_d1536_softplus"]
    small = I.ScanSpec(2, 64, 32, io="bf16", delta_kind="softplus_bias", A_kind="lognormal",
                       D_kind="uniform", seed=c2.seed)
    inp = I.make_scan_inputs(small)
    s = np.logaddexp(0.0, inp["delta_bias"].astype(np.float64))   # softplus(bias) = s_d
    assert np.all((s > 0.99e-3) & (s < 1.01e-1))
    assert np.all(inp["A"] < 0)
    assert np.all((inp["D"] >= 0.5) & (inp["D"] <= 1.5))
    c1 = I.make_scan_inputs(I.WORKLOADS["scan_f32_b2_L256_d16"])
    assert np.array_equal(c1["A"], np.tile(-np.arange(1, 17, dtype=np.float32), (16, 1)))
    d = I.widen(c1["delta"])
    assert d.min() >= 1e-3 * (1 - 1e-6) and d.max() <= 1e-1 * (1 + 1e-6)
    assert I.algorithmic_bytes_scan(I.WORKLOADS["scan_f32_b2_L256_d16"]) == 199744
    assert I.algorithmic_bytes_scan(c2) == 101298176
    assert I.algorithmic_bytes_scan(I.WORKLOADS["scan_bf16_b8_L4096_d2048"]) == 540155904
    assert I.algorithmic_bytes_scan(I.WORKLOADS["scan_bf16_b1_L131072_d5120"]) == 5377773568
    assert I.algorithmic_bytes_decode_step(I.WORKLOADS["decode_bf16_b256_d5120_x64"]) == 178622464
