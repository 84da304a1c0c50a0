"""bf16 rounding and sign-of-zero canonicalisation (oracle; test infrastructure).

The chains keep their intermediate tensor in bf16 ([cuSync] §II-B and Fig.
``fig:gpt-3:mlp``: the first GeMM's GeLU output is stored and then read by
the second GeMM).  The oracle evaluates every chain in fp64 and rounds the
intermediate to bf16 once, directly from the fp64 value, with IEEE
round-to-nearest, ties-to-even.

bf16 keeps 8 significant bits (1 implicit + 7 stored), the fp32 exponent
range (normal exponents -126..127) and subnormals down to 2**-133.

[CUDA-FGS] §4.6.4.1 (Sentinel Value) and Table 16 make the 16-bit pattern
0x8000 (negative zero) the sentinel for bf16 data, and §4.6.4.3 (Producer
Rules, "Canonicalization") requires a producer to store +0 wherever it
would have stored -0.  ``canonicalize_zero`` is that replacement; it does
not change any value, only the sign of zero.
"""

import numpy as np

_BF16_MIN_QUANTUM_EXP = -133   # spacing of bf16 subnormals: 2**-133
_BF16_SIG_BITS = 8             # significant bits of a normal bf16 number


def round_to_bf16(x):
    """Round fp64 values to the nearest bf16 value, ties to even.

    Returns fp64 values that are exactly representable in bf16.  Values at
    or beyond the overflow threshold become +-inf; NaN stays NaN; the sign of
    zero (and of results that round to zero) is kept.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.array(x, dtype=np.float64, copy=True)
    finite = np.isfinite(x) & (x != 0.0)
    if not np.any(finite):
        return out
    xf = x[finite]
    # x = m * 2**e with 0.5 <= |m| < 1, so the leading bit has weight 2**(e-1)
    # and the last kept bit of a normal bf16 number has weight 2**(e-8).
    _, e = np.frexp(xf)
    q = np.maximum(e - _BF16_SIG_BITS, _BF16_MIN_QUANTUM_EXP)
    scaled = np.ldexp(xf, -q)          # exact: scaling by a power of two
    r = np.ldexp(np.rint(scaled), q)   # np.rint rounds half to even
    r = np.where(r == 0.0, np.copysign(0.0, xf), r)
    # Overflow: anything that rounds to 2**128 or beyond is infinite.
    r = np.where(np.abs(r) >= 2.0 ** 128, np.copysign(np.inf, xf), r)
    out[finite] = r
    return out


def canonicalize_zero(x):
    """Replace -0.0 by +0.0 (bf16 pattern 0x8000 -> 0x0000); other values unchanged."""
    x = np.asarray(x, dtype=np.float64)
    return np.where(x == 0.0, 0.0, x)


def bf16_bits(x):
    """The 16-bit bf16 encodings (uint16) of values already exact in bf16."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)  # exact for bf16-representable values
    return (f.view(np.uint32) >> 16).astype(np.uint16)


def from_bf16_bits(bits):
    """fp64 values of raw bf16 encodings (uint16)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
