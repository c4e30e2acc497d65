"""Counter-based SplitMix64 streams for the synthetic block-sparse inputs.

SplitMix64 is the generator of Steele, Lea and Flood, "Fast splittable
pseudorandom number generators" (OOPSLA 2014): the state advances by the
golden-ratio increment 0x9E3779B97F4A7C15 and each output is the state run
through a fixed 64-bit finaliser (two xor-shift-multiply rounds and a final
xor-shift).  Here the t-th output of a stream whose initial state is `s` is
the finaliser applied to s + (t + 1) * increment, which lets every element of
every block be drawn independently of any storage order.

This module is input infrastructure.  It holds no part of the contraction.
"""
from __future__ import annotations

import math

import numpy as np

GOLDEN = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
_MASK = (1 << 64) - 1


def _mix(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output finaliser, elementwise on a uint64 array."""
    z = (z ^ (z >> np.uint64(30))) * _M1
    z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def mix_scalar(x: int) -> int:
    """The same finaliser on one Python int (kept in 64 bits)."""
    z = x & _MASK
    z = ((z ^ (z >> 30)) * 0xBF58476D1CE4E5B9) & _MASK
    z = ((z ^ (z >> 27)) * 0x94D049BB133111EB) & _MASK
    return z ^ (z >> 31)


class SplitMix64:
    """Sequential SplitMix64 stream (used for the structure draws)."""

    def __init__(self, seed: int):
        self.state = seed & _MASK

    def next_u64(self) -> int:
        self.state = (self.state + 0x9E3779B97F4A7C15) & _MASK
        return mix_scalar(self.state)

    def uniform_int(self, lo: int, hi: int) -> int:
        """Integer uniform on [lo, hi] by rejection-free multiply-shift of the top bits.

        The bias of the multiply-shift map is below 2**-50 for the small ranges
        the workloads use.
        """
        span = hi - lo + 1
        return lo + ((self.next_u64() >> 11) * span >> 53)


def block_key(seed: int, op: int, row_sector: int, col_sector: int) -> int:
    """Initial state of the value stream of one block of one operand."""
    k = mix_scalar(seed ^ (op << 56))
    k = mix_scalar(k ^ (row_sector & _MASK))
    k = mix_scalar(k ^ (col_sector & _MASK))
    return k


def stream_u64(keys: np.ndarray, t: np.ndarray) -> np.ndarray:
    """t-th output of the streams with initial states `keys` (uint64 arrays)."""
    with np.errstate(over="ignore"):
        return _mix(keys + (t + np.uint64(1)) * GOLDEN)


def u64_to_unit(x: np.ndarray) -> np.ndarray:
    """Top 53 bits as a double in [0, 1)."""
    return (x >> np.uint64(11)).astype(np.float64) * (1.0 / 9007199254740992.0)


def uniform_pm1(keys: np.ndarray, t: np.ndarray) -> np.ndarray:
    """Uniform on [-1, 1): 2u - 1 with u the t-th unit draw of each stream."""
    return 2.0 * u64_to_unit(stream_u64(keys, t)) - 1.0


def normal(keys: np.ndarray, t: np.ndarray) -> np.ndarray:
    """Standard normal by the Box-Muller transform on draws 2t and 2t+1."""
    u1 = u64_to_unit(stream_u64(keys, np.uint64(2) * t))
    u2 = u64_to_unit(stream_u64(keys, np.uint64(2) * t + np.uint64(1)))
    return np.sqrt(-2.0 * np.log1p(-u1)) * np.cos(2.0 * math.pi * u2)


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round doubles to the nearest bfloat16 value, ties to even, returned as doubles.

    bfloat16 keeps 8 significant bits.  frexp gives x = m * 2**e with
    0.5 <= |m| < 1, so m * 256 holds the 8 kept bits in its integer part and
    rint (round half to even) does the rounding in one step.  Inputs here are
    far from the bfloat16 subnormal and overflow ranges.
    """
    m, e = np.frexp(x)
    return np.ldexp(np.rint(m * 256.0), e - 8)


def bf16_bits(x_bf16_exact: np.ndarray) -> np.ndarray:
    """Bit pattern (uint16) of doubles that already hold bfloat16 values."""
    f = np.asarray(x_bf16_exact, dtype=np.float32)  # exact: 8 significant bits
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)
