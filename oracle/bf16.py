"""bfloat16 rounding for the oracle (test infrastructure only).

The KV pools hold bfloat16.  [Leyline] "Limitations" states that rotation
done in fp32 leaves only the KV *storage* error, i.e. one rounding to bf16
per materialisation.  The oracle models exactly that: values are carried in
float64 and rounded once, round-to-nearest-even, straight from float64 to
bfloat16 (no intermediate float32 step, so there is no double rounding).

bfloat16: 1 sign bit, 8 exponent bits (same range as float32), 8 significant
bits (7 stored).  Normal numbers have 8 significant bits; below 2**-126 the
spacing is fixed at 2**-133 (subnormals).
"""
import numpy as np

BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127


def round_bf16(x):
    """Round float64 values to the nearest bfloat16 (ties to even); returns float64."""
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    xf = x[finite]
    _, e = np.frexp(xf)                   # xf = m * 2**e, 0.5 <= |m| < 1
    q_exp = np.maximum(e - 8, -133)       # spacing of bf16 values near xf
    scaled = np.ldexp(xf, -q_exp)         # exact: power-of-two scaling
    r = np.ldexp(np.rint(scaled), q_exp)  # np.rint rounds half to even
    r = np.where(np.abs(r) > BF16_MAX, np.copysign(np.inf, r), r)
    out[finite] = r
    return out


def to_bits(x):
    """bf16 bit patterns (uint16) of float64 values that are exact bfloat16 numbers."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)              # exact for bf16-representable values
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def from_bits(b):
    """float64 values of bf16 bit patterns (uint16)."""
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def ulp_bf16(x):
    """Spacing of bfloat16 numbers at |x| (the value of one unit in the last place)."""
    x = np.abs(np.asarray(x, dtype=np.float64))
    _, e = np.frexp(np.where(x == 0, 1.0, x))
    return np.ldexp(1.0, np.maximum(e - 8, -133))
