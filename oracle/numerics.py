"""Exact bf16 <-> float64 conversion for the oracle (test infrastructure only).

bf16 is the upper half of an IEEE-754 binary32 word: 1 sign bit, 8 exponent
bits, 7 stored mantissa bits.  Every bf16 value is exactly representable in
float64, so widening is exact.  Narrowing float64 -> bf16 is done here in one
rounding step (round to nearest, ties to even), never through float32, so no
double rounding occurs.
"""
import numpy as np

# bf16 has 8 significant bits (7 stored + the implicit leading one).
_BF16_SIG_BITS = 8
# Smallest normal bf16 exponent (same exponent field as binary32).
_BF16_EMIN = -126
_BF16_MAX = float(np.ldexp(2.0 - 2.0 ** -7, 127))


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) to float64, exactly."""
    b = np.asarray(bits).astype(np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):      # NaN payloads widen to NaN
        return b.view(np.float32).astype(np.float64)


def round_to_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bf16 value (ties to even).

    Returns float64 values that are exactly representable in bf16.  Handles
    subnormals (quantum 2**-133), overflow to +-inf (values at or beyond the
    midpoint above the largest finite bf16), signed zeros and NaN.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    finite = np.isfinite(x)
    out[~finite] = x[~finite]
    xf = x[finite]
    # frexp: xf = m * 2**e with 0.5 <= |m| < 1, so the leading bit has weight 2**(e-1)
    _, e = np.frexp(xf)
    # quantum (weight of the last kept bit) for a normal number with this exponent
    q_exp = (e - 1) - (_BF16_SIG_BITS - 1)
    # subnormal range: the quantum never drops below 2**(EMIN - 7)
    q_exp = np.maximum(q_exp, _BF16_EMIN - (_BF16_SIG_BITS - 1))
    scaled = np.ldexp(xf, -q_exp)          # exact: a power-of-two scaling
    r = np.rint(scaled)                    # round half to even
    y = np.ldexp(r, q_exp)
    # overflow: anything that rounds above the largest finite value becomes inf
    big = np.abs(y) > _BF16_MAX
    y[big] = np.copysign(np.inf, xf[big])
    # keep the sign of zero
    y = np.where(y == 0, np.copysign(0.0, xf), y)
    out[finite] = y
    return out


def f64_to_bf16_bits(x) -> np.ndarray:
    """Round float64 to bf16 (ties to even) and return the raw uint16 bits."""
    y = round_to_bf16(x)
    f32 = y.astype(np.float32)             # exact: y is a bf16 value
    return (f32.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
