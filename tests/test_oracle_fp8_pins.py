"""Pins of the 8-bit oracle (``oracle/fp8.py``) to facts outside it, and
planted mistakes that those pins must catch.

* Decoding: the values the OCP 8-bit floating point specification lists for
  E4M3 (largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9,
  the NaN codes), and strict monotonicity over the positive codes.
* Encoding: a brute-force nearest-value search over the 127 non-negative
  finite values, with ties going to the even mantissa, on random values, on
  every midpoint between neighbours and one fp32 ulp either side of it;
  PyTorch's own float8_e4m3fn cast (a library routine) for |v| <= 448; and
  saturation beyond 448.
* Quantisation: the element of largest magnitude maps onto 448 and every
  dequantised value is within half a quantum of its input.
* The GEMM: exact rational arithmetic (``fractions.Fraction``) on tiny sizes,
  which also fixes which operand is transposed and how the scales enter.
"""
from fractions import Fraction

import numpy as np
import pytest

from oracle import fp8 as F

torch = pytest.importorskip("torch")

POS_CODES = np.arange(0x7F, dtype=np.uint8)          # 0x00 .. 0x7e: every non-negative finite value


def test_decode_specification_values():
    d = F.e4m3_decode
    assert d(0x7E) == 448.0
    assert d(0xFE) == -448.0
    assert d(0x08) == 2.0 ** -6
    assert d(0x07) == 7 * 2.0 ** -9
    assert d(0x01) == 2.0 ** -9
    assert d(0x38) == 1.0 and d(0xB8) == -1.0
    assert d(0x40) == 2.0 and d(0x3C) == 1.5
    assert np.isnan(d(0x7F)) and np.isnan(d(0xFF))
    assert d(0x00) == 0.0 and np.signbit(d(0x80))
    vals = d(POS_CODES)
    assert np.all(np.diff(vals) > 0)


def test_round_trip_of_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(F.e4m3_encode(F.e4m3_decode(codes)), codes)


def _brute_force(v):
    """Nearest representable value by exhaustive search; ties to the even code."""
    vals = F.e4m3_decode(POS_CODES)
    out = np.empty(len(v), dtype=np.uint8)
    for i, x in enumerate(np.asarray(v, dtype=np.float64)):
        a = min(abs(x), 448.0)
        dist = np.abs(vals - a)
        best = np.flatnonzero(dist == dist.min())
        c = int(best[0]) if len(best) == 1 else int(best[np.argmin(best % 2)])
        out[i] = c | (0x80 if np.signbit(x) else 0)
    return out


def test_encode_matches_brute_force_nearest_with_ties_to_even():
    rng = np.random.default_rng(5)
    vals = F.e4m3_decode(POS_CODES)
    mids = (vals[1:] + vals[:-1]) / 2                 # exact ties (fp64 and fp32 hold them)
    f32 = mids.astype(np.float32)
    assert np.array_equal(f32.astype(np.float64), mids)
    cases = np.concatenate([
        rng.standard_normal(3000) * 30.0,
        rng.standard_normal(1000) * 1e-2,             # subnormal range
        mids, -mids,
        np.nextafter(f32, np.float32(np.inf)).astype(np.float64),
        np.nextafter(f32, np.float32(-np.inf)).astype(np.float64),
        [0.0, -0.0, 1e-30, -1e-30, 448.0, 460.0, 463.99, 464.0, 500.0, 1e30, -1e30],
    ]).astype(np.float32)
    assert np.array_equal(F.e4m3_encode(cases), _brute_force(cases))


def test_encode_matches_torch_float8_e4m3fn_in_range():
    rng = np.random.default_rng(6)
    v = np.concatenate([rng.uniform(-448, 448, 20000), rng.standard_normal(20000) * 1e-2]).astype(np.float32)
    want = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(F.e4m3_encode(v), want)


def test_saturation():
    v = np.array([449.0, 463.0, 464.0, 480.0, 1e6, -449.0, -1e6], dtype=np.float32)
    assert list(F.e4m3_encode(v)) == [0x7E] * 5 + [0xFE] * 2


def test_quantize_maps_amax_to_448_and_bounds_the_error():
    rng = np.random.default_rng(7)
    x = (rng.standard_normal(5000) * 3.7).astype(np.float32)
    codes, amax, scale, scale_inv = F.quantize(x)
    assert amax == np.max(np.abs(x))
    assert F.e4m3_decode(codes[np.argmax(np.abs(x))]) * np.sign(x[np.argmax(np.abs(x))]) == 448.0
    deq = F.e4m3_decode(codes) * np.float64(scale_inv)
    xs = np.abs(x.astype(np.float64) * np.float64(scale))
    # half a quantum: 2^-4 relative in the normal range, 2^-10 absolute below it (in scaled units);
    # the two fp32 roundings (x * scale, 1 / scale) add a few 2^-24 relative
    bound = np.maximum(2.0 ** -4 * xs, 2.0 ** -10) * (1 + 1e-6) / np.float64(scale)
    assert np.all(np.abs(deq - x) <= bound + 4 * 2.0 ** -24 * np.abs(x))


def test_quantize_degenerate_inputs():
    codes, amax, scale, scale_inv = F.quantize(np.zeros(10, dtype=np.float32))
    assert amax == 0 and scale == 1 and scale_inv == 1 and not codes.any()
    codes, amax, scale, scale_inv = F.quantize(np.zeros(0, dtype=np.float32))
    assert amax == 0 and scale == 1 and codes.size == 0
    # a maximum so small that 448 / amax overflows fp32: the scale falls back to 1
    codes, amax, scale, _ = F.quantize(np.array([1e-40, -5e-41], dtype=np.float32))
    assert scale == 1 and not (codes & 0x7F).any()


def test_gemm_exact_on_tiny_sizes():
    rng = np.random.default_rng(8)
    M, N, K = 3, 4, 16
    a = rng.integers(0, 256, (M, K)).astype(np.uint8)
    b = rng.integers(0, 256, (N, K)).astype(np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x11                      # no NaN codes
    b[(b & 0x7F) == 0x7F] = 0x22
    sa, sb = np.float32(0.375), np.float32(1.0 / 64)
    D = F.gemm(a, b, sa, sb)

    def exact(c):
        c = int(c)
        s = -1 if c >> 7 else 1
        e, m = (c >> 3) & 15, c & 7
        return s * (Fraction(m, 2 ** 9) if e == 0 else Fraction(8 + m, 8) * Fraction(2) ** (e - 7))

    for i in range(M):
        for j in range(N):
            want = Fraction(float(sa)) * Fraction(float(sb)) * sum(exact(a[i, k]) * exact(b[j, k]) for k in range(K))
            assert Fraction(D[i, j]) == want


# ---------------------------------------------------------------- planted mistakes
def _encode_ties_away(v):
    """The oracle's encoder with ties rounded away from zero (a plausible slip)."""
    v = np.asarray(v, dtype=np.float64)
    a = np.abs(v)
    _, ex = np.frexp(a)
    q = np.exp2((np.maximum(ex - 1, -6) - 3).astype(np.float64))
    r = np.floor(a / q + 0.5)
    return F.e4m3_encode(np.copysign(np.minimum(r * q, 448.0), v))


def _encode_no_subnormals(v):
    """Flushes the subnormal range to zero (another plausible slip)."""
    v = np.asarray(v, dtype=np.float64)
    return F.e4m3_encode(np.where(np.abs(v) < 2.0 ** -6, 0.0, v))


@pytest.mark.parametrize("wrong", [_encode_ties_away, _encode_no_subnormals])
def test_planted_encoder_mistakes_are_caught(wrong):
    vals = F.e4m3_decode(POS_CODES)
    cases = np.concatenate([(vals[1:] + vals[:-1]) / 2, [3e-3, 1.1e-3]]).astype(np.float32)
    assert not np.array_equal(wrong(cases), _brute_force(cases))


def test_planted_gemm_transpose_is_caught():
    rng = np.random.default_rng(9)
    a = rng.integers(0, 0x70, (4, 4)).astype(np.uint8)
    b = rng.integers(0, 0x70, (4, 4)).astype(np.uint8)
    A, B = F.e4m3_decode(a), F.e4m3_decode(b)
    good = F.gemm(a, b, 1.0, 1.0)
    assert np.array_equal(good, A @ B.T)
    assert not np.allclose(good, A @ B)
