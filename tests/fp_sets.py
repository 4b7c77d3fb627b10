"""Structured FP32 input sets for the encoder pins (test infrastructure).

A rounding encoder to a format with ``m`` mantissa bits looks at the FP32
bits above and below the rounding position.  ``structured_f32(top_bits)``
enumerates every pattern of the top ``top_bits`` bits (sign, exponent and
the leading mantissa bits, so every binade and every kept-mantissa pattern)
and pairs each with a handful of low-bit tails: zero (exact ties and exact
values), one (just above), all ones (just below the next), the half-way
pattern and its neighbours, and a random tail.
"""
import numpy as np


def structured_f32(top_bits: int, seed: int = 1234) -> np.ndarray:
    low_bits = 32 - top_bits
    full = (1 << low_bits) - 1
    half = 1 << (low_bits - 1)
    rng = np.random.default_rng(seed)
    hi = np.arange(1 << top_bits, dtype=np.uint64) << np.uint64(low_bits)
    tails = [0, 1, full, half, half - 1, half + 1]
    parts = [hi | np.uint64(t) for t in tails]
    parts.append(hi | rng.integers(0, full + 1, size=hi.size, dtype=np.uint64))
    bits = np.concatenate(parts).astype(np.uint32)
    return bits.view(np.float32)


def random_f32(n: int, seed: int = 99) -> np.ndarray:
    rng = np.random.default_rng(seed)
    return rng.integers(0, 1 << 32, size=n, dtype=np.uint64).astype(np.uint32).view(np.float32)


def finite(x: np.ndarray) -> np.ndarray:
    return x[np.isfinite(x)]
