"""Pins of the oracle's SwiGLU activation (CPU only).

The activation between the gate+up and down projections, h = SiLU(g) * u
with SiLU(g) = g / (1 + e^-g), runs in FP32 on the BF16 outputs of the gate
and up projections and is rounded to BF16.  Its exponential is a Cody-Waite
reduction with a Taylor polynomial.  The pins compare with float64
mathematics (numpy's exp), not with the oracle's own formulas, and check
the special cases that fix each term: the sign of the exponent, the factor
u, the final rounding, the range limits."""
import numpy as np

import oracle

F32_ULP = lambda v: np.spacing(np.abs(v).astype(np.float32)).astype(np.float64)  # noqa: E731


def bf16_bits_of(v: np.ndarray) -> np.ndarray:
    """float64 -> BF16 bits, round to nearest even (via the exact FP32 value
    when it is one; the values here are)."""
    f = np.asarray(v, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lower = u & 0xFFFF
    upper = u >> 16
    up = (lower > 0x8000) | ((lower == 0x8000) & ((upper & 1) == 1))
    return (upper + up).astype(np.uint16)


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_exp_within_one_ulp_of_float64():
    rng = np.random.default_rng(5)
    x = np.concatenate([np.linspace(-87.0, 88.0, 400001), rng.uniform(-87, 88, 100000),
                        rng.normal(0, 3, 100000).clip(-87, 88)]).astype(np.float32)
    got = oracle.exp_cw(x).astype(np.float64)
    ref = np.exp(x.astype(np.float64))
    assert np.all(np.abs(got - ref) <= F32_ULP(ref)), "more than 1 ulp off e^x"


def test_exp_special_values_and_range():
    e = oracle.exp_cw(np.array([0.0, -0.0, 88.5, 1e30, -87.5, -1e30], np.float32))
    assert e[0] == 1.0 and e[1] == 1.0                      # r = 0 and n = 0 give exactly 1
    assert np.isinf(e[2]) and np.isinf(e[3]) and e[2] > 0  # above the range
    assert e[4] == 0.0 and e[5] == 0.0                      # below it
    # exact powers of two where the polynomial is evaluated at r = 0
    n = np.arange(-120, 121, dtype=np.float64)
    x = (n * np.log(2.0)).astype(np.float32)
    ref = np.exp(x.astype(np.float64))
    assert np.all(np.abs(oracle.exp_cw(x) - ref) <= F32_ULP(ref))


def test_silu_mul_within_one_bf16_ulp_of_float64():
    # every finite BF16 g in [-24, 24] against several u, both signs
    all_bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    gvals = bf16_to_f64(all_bits)
    g = all_bits[np.isfinite(gvals) & (np.abs(gvals) <= 24.0)]
    for uval in (1.0, -1.0, 0.3359375, -2.75, 1e-3, 96.0):
        u = np.full(g.shape, bf16_bits_of(np.array([uval]))[0], np.uint16)
        h = oracle.silu_mul(g, u)
        gf, uf = bf16_to_f64(g), bf16_to_f64(u)
        ref = gf / (1.0 + np.exp(-gf)) * uf
        got = bf16_to_f64(h)
        ulp = np.maximum(bf16_to_f64(bf16_bits_of(np.abs(ref)) + 1) - bf16_to_f64(bf16_bits_of(np.abs(ref))),
                         2.0 ** -133)
        assert np.all(np.abs(got - ref) <= ulp), f"u = {uval}"
        assert np.all((np.sign(got) == np.sign(ref)) | (got == 0) | (np.abs(ref) < 1e-30))


def test_silu_mul_special_cases():
    b = lambda v: bf16_bits_of(np.array(v, dtype=np.float64))  # noqa: E731
    # g = 0: zero, with the sign of u
    h = oracle.silu_mul(b([0.0, 0.0]), b([3.0, -3.0]))
    assert np.all(bf16_to_f64(h) == 0.0)
    assert h[0] == 0x0000 and h[1] == 0x8000
    # u = 0: zero
    assert np.all(bf16_to_f64(oracle.silu_mul(b([1.5, -7.0]), b([0.0, 0.0]))) == 0.0)
    # g >= 17: 1 + e^-g rounds to 1 in FP32, so h = bf16(g * u) exactly
    g = np.linspace(17.0, 80.0, 64)
    u = np.linspace(-3.0, 3.0, 64)
    gb, ub = b(g), b(u)
    exp = bf16_bits_of(bf16_to_f64(gb).astype(np.float32) * bf16_to_f64(ub).astype(np.float32))
    assert np.array_equal(oracle.silu_mul(gb, ub), exp)
    # g < -88: e^-g overflows, SiLU(g) = g / Inf = -0
    h = oracle.silu_mul(b([-100.0, -100.0]), b([2.0, -2.0]))
    assert np.all(bf16_to_f64(h) == 0.0)
    # SiLU(1) * 1 = 1 / (1 + 1/e) = 0.7310585..., BF16 0.73046875 (0x3F3B)
    assert oracle.silu_mul(b([1.0]), b([1.0]))[0] == 0x3F3B
    # SiLU(-1) * 1 = -0.2689414..., BF16 -0.26953125 (0xBE8A)
    assert oracle.silu_mul(b([-1.0]), b([1.0]))[0] == 0xBE8A
