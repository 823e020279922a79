"""bfloat16 encode/decode for the oracle (TEST INFRASTRUCTURE ONLY).

bfloat16 is the IEEE-754 binary32 layout cut to its top 16 bits: 1 sign bit,
8 exponent bits (bias 127) and 7 fraction bits.  The path's inputs are bf16,
its accumulation is at least fp32 and its outputs are bf16 rounded to
nearest, ties to even (the page pair cited in ``oracle/__init__`` fixes only
"bf16 GEMM"; rounding mode RNE is the IEEE default and the one the CUDA path
uses).

Rounding is written from the definition, not by bit tricks: for a finite
value x, the spacing of bf16 numbers around |x| is ulp = 2**(e - 7) with
e = floor(log2|x|) clamped below at the smallest normal exponent -126 (below
it the subnormal spacing 2**-133 stays fixed).  |x| / ulp is exact in fp64
(a power-of-two scale), ``numpy.rint`` rounds it half-to-even, and the result
times ulp is the rounded value; at or above 2**128 it overflows to infinity.
"""
import numpy as np

_MIN_NORMAL_EXP = -126
_round_half_even = np.rint   # numpy's rint rounds halfway cases to even
_FRAC_BITS = 7
_SUBNORMAL_ULP_EXP = _MIN_NORMAL_EXP - _FRAC_BITS  # -133


def bits_to_f64(bits):
    """Decode bf16 bit patterns (uint16 array) to exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_to_bf16(x):
    """Round float values (any float dtype; computed in fp64) to bf16 bits.

    Returns a uint16 array.  NaN maps to the quiet NaN 0x7FC0; +-inf stays
    infinite; overflow past the largest finite bf16 after
    rounding gives infinity, as IEEE round-to-nearest prescribes.
    """
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x)
    a = np.abs(x)
    out = np.zeros(x.shape, dtype=np.uint16)

    finite_nz = np.isfinite(a) & (a > 0)
    af = a[finite_nz]
    # |x| = m * 2**E with m in [0.5, 1)  =>  floor(log2 |x|) = E - 1.
    _, E = np.frexp(af)
    e = np.maximum(E.astype(np.int64) - 1, _MIN_NORMAL_EXP)
    ulp_exp = e - _FRAC_BITS
    q = np.ldexp(af, -ulp_exp)             # exact: power-of-two scaling
    r = _round_half_even(q)
    y = np.ldexp(r, ulp_exp)                # the rounded magnitude

    enc = np.zeros(af.shape, dtype=np.uint32)
    overflow = y >= 2.0 ** 128
    sub = (y < 2.0 ** _MIN_NORMAL_EXP) & ~overflow
    norm = ~sub & ~overflow
    # subnormal (and zero after rounding): exponent field 0, fraction = y / 2**-133
    enc[sub] = np.ldexp(y[sub], -_SUBNORMAL_ULP_EXP).astype(np.uint32)
    # normal: y = (1 + f/128) * 2**ey, exponent field ey + 127
    _, Ey = np.frexp(y[norm])
    ey = Ey.astype(np.int64) - 1
    frac = np.ldexp(y[norm], -ey) - 1.0     # in [0, 1), a multiple of 1/128
    enc[norm] = (((ey + 127).astype(np.uint32) << 7)
                 | (frac * 128.0).astype(np.uint32))   # exact integer
    enc[overflow] = 0xFF << 7
    out[finite_nz] = enc.astype(np.uint16)

    out[np.isinf(a)] = 0xFF << 7
    out[np.isnan(x)] = 0x7FC0
    out = np.where(sign & ~np.isnan(x), out | np.uint16(0x8000), out)
    return out.astype(np.uint16)


def f32_round_to_bf16(x32):
    """fp32 array -> bf16 bits (fp32 is exact in fp64, so one rounding)."""
    return round_to_bf16(np.asarray(x32, dtype=np.float32).astype(np.float64))
