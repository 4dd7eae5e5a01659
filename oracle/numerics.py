"""bf16 <-> fp32 conversions for the oracle (test infrastructure only).

The pages count parameters and gradients at 16 bits ("Infra: Data Parallel",
ZeRO memory figure: 2 bytes each) and optimizer state at 4 bytes per value
(k = 12: fp32 master weights, first and second moments).  The 16-bit format is
read as bfloat16: the upper half of an IEEE-754 binary32.

* widening bf16 -> fp32 is exact: place the 16 bits in the upper half.
* narrowing fp32 -> bf16 is round-to-nearest, ties-to-even, written here
  from that definition: keep the upper 16 bits, then look at the 16 bits
  that are dropped.  Above half an ulp rounds up, below rounds down, exactly
  half rounds to the neighbour whose last kept bit is 0.  Carrying into the
  exponent field is the correct result (it also turns values beyond the
  largest bf16 into infinity).  NaN stays NaN (quiet bit set).
"""

import numpy as np


def f32_from_bf16(bits):
    """bf16 bit patterns (uint16 array) -> float32 values, exactly."""
    bits = np.asarray(bits, dtype=np.uint16)
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def bf16_rne(x):
    """float32 values -> bf16 bit patterns (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    kept = u >> np.uint32(16)
    dropped = u & np.uint32(0xFFFF)
    half = np.uint32(0x8000)
    last_kept_bit = kept & np.uint32(1)
    round_up = (dropped > half) | ((dropped == half) & (last_kept_bit == 1))
    out = kept + round_up.astype(np.uint32)
    # NaN: exponent all ones and a non-zero fraction -> a quiet NaN with the same sign
    is_nan = ((u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)) & ((u & np.uint32(0x007FFFFF)) != 0)
    out = np.where(is_nan, kept | np.uint32(0x0040), out)
    return out.astype(np.uint16)


def bf16_ulp(bits):
    """Spacing of bf16 numbers at |value| (as float64), for 1-ulp gates."""
    exp_field = (np.asarray(bits, dtype=np.uint16).astype(np.int64) >> 7) & 0xFF
    e = np.where(exp_field == 0, 1, exp_field) - 127
    return np.ldexp(1.0, (e - 7).astype(np.int64))
