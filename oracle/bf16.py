"""bfloat16 rounding written from the format's definition (test infrastructure).

bfloat16 keeps float32's 8-bit exponent and 7 explicit mantissa bits, so a
finite value carries 8 significant bits; float32's subnormal range is kept,
with a quantum of 2**-133 below 2**-126.  Rounding is IEEE 754
round-to-nearest, ties-to-even.  Values at or beyond 2**128 after rounding
overflow to infinity.

Pinned by tests/test_oracle_bf16.py against hand-worked ties and against
PyTorch's float32 -> bfloat16 conversion (a library routine) on float32
inputs, where rounding float64 directly must agree with it.
"""

import numpy as np


def round_bf16(x) -> np.ndarray:
    """Round float64 values to the nearest bfloat16 value (ties to even).

    Returns float64 values that are exactly representable in bfloat16.
    """
    x = np.asarray(x, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        _, e = np.frexp(x)  # x = m * 2**e with 0.5 <= |m| < 1
        qe = np.maximum(e - 8, -133)  # exponent of one unit in the last place
        r = np.ldexp(np.rint(np.ldexp(x, -qe)), qe)  # rint: half to even
        r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, x), r)
    return np.where(np.isfinite(x), r, x)


def bits_to_f64(u16) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> float64 values (exact)."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return u.view(np.float32).astype(np.float64)


def f64_to_bits(x) -> np.ndarray:
    """float64 -> bfloat16 bit patterns (uint16), rounding to nearest even."""
    r = round_bf16(x).astype(np.float32)  # exact: r is bf16-representable
    return (r.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
