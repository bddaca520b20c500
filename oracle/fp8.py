"""8-bit floating point (E4M3) quantisation and the scaled 8-bit GEMM.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  It shares no code with
the CUDA path.

What the pages fix: the woshipm nanochat analysis names FP8 among nanochat's
speed levers on Hopper-class tensor cores (§一.2, and §六.2 on the precision
strategy), and nothing more: no format, scaling or placement.

The reading taken here (published definitions):

* Format: E4M3 of the OCP 8-bit floating point specification (OFP8, 2023).
  A code is sign (bit 7), a 4-bit exponent field E with bias 7 (bits 6-3) and
  a 3-bit mantissa M (bits 2-0).  E = 0 holds the subnormals M * 2^-9;
  otherwise the value is (1 + M/8) * 2^(E-7), except E = 15 with M = 7, which
  is NaN.  The largest finite value is 1.75 * 2^8 = 448; there are no
  infinities.
* Conversion of a real value: IEEE round to nearest, ties to even mantissa,
  saturating (a magnitude beyond 448 becomes 448); the sign is kept, so a
  negative value that rounds to zero gives the code 0x80.
* Scaling: one factor per tensor from the tensor's current absolute maximum,
  mapping it onto 448: scale = fl32(448 / amax) (replaced by 1 when that is
  not finite and positive), codes of fl32(x * scale), and the dequantisation
  factor scale_inv = fl32(1 / scale).  The quantised code is an integer
  decided by floating point, so this side takes the decision in the same
  precision as the kernels: fp32 for the scale and the scaled value.
* The GEMM: D = a_scale_inv * b_scale_inv * sum_k A(m, k) B(n, k) over the
  decoded values.  The fp64 sum of E4M3 products is exact for K < 2^17 (each
  product is an 8-bit integer times a power of two in [2^-18, 2^11]).
"""
import numpy as np

E4M3_MAX = 448.0
_MIN_NORMAL_EXP = -6      # smallest normal binade: [2^-6, 2^-5)
_MANT_BITS = 3


def e4m3_decode(codes):
    """fp64 values of E4M3 codes (NaN for 0x7f / 0xff)."""
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    sign = np.where(c >> 7, -1.0, 1.0)
    e = (c >> 3) & 15
    m = (c & 7).astype(np.float64)
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0))
    mag = np.where((e == 15) & (c & 7 == 7), np.nan, mag)
    return sign * mag


def e4m3_encode(v):
    """E4M3 codes of finite values v (rounded to nearest even, saturating)."""
    v = np.asarray(v, dtype=np.float64)
    if not np.all(np.isfinite(v)):
        raise ValueError("E4M3 encoding of a non-finite value is not defined here")
    neg = np.signbit(v)
    a = np.abs(v)
    # binade exponent of a (a in [2^E, 2^(E+1))), the subnormal range sharing
    # the quantum of the smallest normal binade
    _, ex = np.frexp(a)
    E = np.maximum(ex.astype(np.int64) - 1, _MIN_NORMAL_EXP)
    q = np.exp2((E - _MANT_BITS).astype(np.float64))
    r = np.rint(a / q)                                   # half to even; a / q is exact
    val = np.minimum(r * q, E4M3_MAX)                    # saturate
    # code of the (representable) magnitude val
    _, vex = np.frexp(val)
    VE = vex.astype(np.int64) - 1
    normal = val >= 2.0 ** _MIN_NORMAL_EXP
    e_field = np.where(normal, VE + 7, 0)
    m_field = np.where(normal, val / np.exp2(VE.astype(np.float64)) * 8.0 - 8.0, val / 2.0 ** -9)
    code = (e_field << 3) | np.rint(m_field).astype(np.int64)
    code = np.where(val == 0, 0, code)
    return (code | (neg.astype(np.int64) << 7)).astype(np.uint8)


def quantize(x):
    """Per-tensor E4M3 quantisation of x (fp32 values; bf16 inputs as their
    fp32 values).  Returns (codes uint8, amax, scale, scale_inv), the last
    three as float32."""
    x32 = np.asarray(x, dtype=np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0.0)
    with np.errstate(divide="ignore", over="ignore"):
        scale = np.float32(E4M3_MAX) / amax
    if not (np.isfinite(scale) and scale > 0):
        scale = np.float32(1.0)
    scaled = (x32 * scale).astype(np.float32)
    return e4m3_encode(scaled), amax, np.float32(scale), np.float32(np.float32(1.0) / scale)


def gemm(a_codes, b_codes, a_scale_inv, b_scale_inv):
    """D[m, n] = a_scale_inv * b_scale_inv * sum_k A(m, k) B(n, k), fp64."""
    A = e4m3_decode(a_codes)
    B = e4m3_decode(b_codes)
    return (float(a_scale_inv) * float(b_scale_inv)) * (A @ B.T)
