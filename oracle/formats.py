"""16-bit float formats for the oracle (test infrastructure only).

The cache, the queries and the outputs are 16-bit floats (fp16 or bf16).  The oracle
keeps them as raw ``uint16`` bit patterns, decodes them exactly to float64, computes in
float64 and rounds the result back with round-to-nearest-even (ties to even), straight
from float64 -- no intermediate float32 step, so there is no double rounding.

Format parameters (IEEE 754 binary16 and the bfloat16 truncation of binary32):
    fp16: 10 stored mantissa bits, normal exponents -14 .. 15
    bf16:  7 stored mantissa bits, normal exponents -126 .. 127
"""
import numpy as np

FORMATS = {
    "fp16": {"mant": 10, "emin": -14, "emax": 15, "qnan": 0x7E00},
    "bf16": {"mant": 7, "emin": -126, "emax": 127, "qnan": 0x7FC0},
}


def decode_bits(bits, dtype):
    """Exact value (float64) of each 16-bit pattern in ``bits``."""
    bits = np.asarray(bits, dtype=np.uint16)
    if dtype == "fp16":
        return bits.view(np.float16).astype(np.float64)
    if dtype == "bf16":
        with np.errstate(invalid="ignore"):   # signalling-NaN patterns stay NaN
            return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    raise ValueError(dtype)


def round_rne(x, dtype):
    """Round float64 values to the nearest value of ``dtype``, ties to even.

    For |x| in [2^e, 2^(e+1)) the spacing of the format is 2^(max(e, emin) - mant); dividing
    by that power of two is exact in float64, ``np.rint`` rounds half to even, and
    multiplying back is exact.  A result beyond the largest finite value becomes inf
    (the overflow rule of round-to-nearest).  NaN and inf pass through.
    """
    f = FORMATS[dtype]
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0)
    xf = x[finite]
    _, e2 = np.frexp(xf)               # xf = m * 2**e2, 0.5 <= |m| < 1
    e = np.maximum(e2 - 1, f["emin"])  # exponent of the leading bit, clamped for subnormals
    quantum = np.ldexp(1.0, e - f["mant"])
    r = np.rint(xf / quantum) * quantum
    max_finite = (2.0 - 2.0 ** (-f["mant"])) * 2.0 ** f["emax"]
    r = np.where(np.abs(r) > max_finite, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def encode_bits(x, dtype):
    """Bit patterns of ``round_rne(x, dtype)``; NaN becomes the format's quiet NaN."""
    r = round_rne(x, dtype)
    nan = np.isnan(r)
    if dtype == "fp16":
        bits = r.astype(np.float16).view(np.uint16)   # exact: r is already an fp16 value
    elif dtype == "bf16":
        bits = (r.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)  # exact
    else:
        raise ValueError(dtype)
    bits = np.array(bits, dtype=np.uint16)
    bits[nan] = FORMATS[dtype]["qnan"]
    return bits
