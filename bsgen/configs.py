"""The synthetic block-sparse workloads: sector axes, allowed-charge rules, value draws.

A workload names three sector axes (row, inner, column).  Each sector has an
index (its identity), a U(1) charge, an optional Z2 parity and a dimension.
An operand's allowed-charge rule says which (row sector, column sector) pairs
hold a block: dq_min <= q_row - q_col <= dq_max, and, when `z2` is set, equal
parities.  This module only *describes* the rule; evaluating it, building
layouts and contracting are left to the code under test and to the oracle.

Values are drawn per block from a SplitMix64 stream keyed on
(seed, operand, row sector, column sector), element t of the block being its
row-major index, so any storage layout receives the same numbers.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

from . import rng

OP_A, OP_B = 0, 1


@dataclass
class Axis:
    q: np.ndarray                     # int32 U(1) charge per sector
    d: np.ndarray                     # int32 dimension per sector
    p: Optional[np.ndarray] = None    # uint8 Z2 parity per sector, or None

    @property
    def n(self) -> int:
        return int(self.q.shape[0])

    def __post_init__(self):
        self.q = np.ascontiguousarray(self.q, dtype=np.int32)
        self.d = np.ascontiguousarray(self.d, dtype=np.int32)
        if self.p is not None:
            self.p = np.ascontiguousarray(self.p, dtype=np.uint8)


@dataclass
class Rule:
    dq_min: int
    dq_max: int
    z2: bool = False


@dataclass
class Workload:
    name: str
    dtype: str                 # "f64" or "bf16" (BF16 inputs, FP32 output)
    rows: Axis
    inner: Axis
    cols: Axis
    rule_a: Rule
    rule_b: Rule
    values: str                # uniform | normal | normal_inv_sqrt_dk | int3 | ones
    seed: int
    # layout names of the timed run, and of the run that exercises packing
    layout_a: str = "rowpanel|charge_sorted"
    layout_b: str = "colpanel|charge_sorted"
    layout_c: str = "blockrow"
    pack_layout_a: str = "blockrow"
    pack_layout_b: str = "blockrow"
    pack_layout_c: str = "blockrow"
    notes: str = ""
    extra: dict = field(default_factory=dict)

    # ---- values ---------------------------------------------------------
    def block_scale(self, op: int, rs: np.ndarray, cs: np.ndarray) -> np.ndarray:
        if self.values != "normal_inv_sqrt_dk":
            return np.ones(len(rs))
        k = cs if op == OP_A else rs        # the inner sector of the block
        return 1.0 / np.sqrt(self.inner.d[k].astype(np.float64))

    def draw(self, op: int, rs, cs, rows, cols) -> np.ndarray:
        """Values of the listed blocks, concatenated, each block row-major.

        For bf16 workloads the values are already rounded to bfloat16 (exact
        doubles); `rng.bf16_bits` gives their bit patterns.
        """
        rs = np.asarray(rs, dtype=np.int64)
        cs = np.asarray(cs, dtype=np.int64)
        sizes = np.asarray(rows, dtype=np.int64) * np.asarray(cols, dtype=np.int64)
        total = int(sizes.sum())
        if total == 0:
            return np.zeros(0)
        keys = np.fromiter((rng.block_key(self.seed, op, int(r), int(c)) for r, c in zip(rs, cs)),
                           dtype=np.uint64, count=len(rs))
        starts = np.concatenate([[0], np.cumsum(sizes)[:-1]])
        kk = np.repeat(keys, sizes)
        t = (np.arange(total, dtype=np.int64) - np.repeat(starts, sizes)).astype(np.uint64)
        if self.values == "uniform":
            v = rng.uniform_pm1(kk, t)
        elif self.values in ("normal", "normal_inv_sqrt_dk"):
            v = rng.normal(kk, t) * np.repeat(self.block_scale(op, rs, cs), sizes)
        elif self.values == "int3":
            v = (rng.stream_u64(kk, t) % np.uint64(7)).astype(np.float64) - 3.0
        elif self.values == "ones":
            v = np.ones(total)
        else:
            raise ValueError(self.values)
        if self.dtype == "bf16":
            v = rng.round_to_bf16(v)
        return v


def _dims(qs, fn):
    return np.array([fn(q) for q in qs], dtype=np.int32)


def _round_half_away(x: float) -> int:
    return int(math.floor(abs(x) + 0.5)) * (1 if x >= 0 else -1)


def config1() -> Workload:
    """FP64 toy: 9 charges -4..4, d(q) = 1 + (|q|*7) % 6, bands |dq| <= 1."""
    qs = np.arange(-4, 5)
    d = _dims(qs, lambda q: 1 + (abs(q) * 7) % 6)
    ax = Axis(qs, d)
    return Workload("fp64_toy_9x9x9", "f64", ax, Axis(qs, d), Axis(qs, d), Rule(-1, 1), Rule(-1, 1),
                    "uniform", 0x5EED0000 + 1)


def config2() -> Workload:
    """FP64 tail: 31 charges -15..15, d(q) = max(1, round(64 exp(-q^2/50)))."""
    qs = np.arange(-15, 16)
    d = _dims(qs, lambda q: max(1, _round_half_away(64 * math.exp(-q * q / 50))))
    return Workload("fp64_tail_31x31x31", "f64", Axis(qs, d), Axis(qs, d), Axis(qs, d), Rule(-1, 1),
                    Rule(-1, 1), "normal", 0x5EED0000 + 2)


def config3() -> Workload:
    """FP64 large: 41 charges -20..20, d(q) = max(1, round(512 exp(-q^2/60))), N(0, 1/sqrt(d_k))."""
    qs = np.arange(-20, 21)
    d = _dims(qs, lambda q: max(1, _round_half_away(512 * math.exp(-q * q / 60))))
    return Workload("fp64_large_41x41x41", "f64", Axis(qs, d), Axis(qs, d), Axis(qs, d), Rule(-1, 1),
                    Rule(-1, 1), "normal_inv_sqrt_dk", 0x5EED0000 + 3)


def config4() -> Workload:
    """BF16 in / FP32 out: inner and column axes are BlockSpace charges -12..12 with
    d(q) = max(2, round(256 exp(-q^2/40))); the row axis is that BlockSpace times a
    LocalSpace key s in 0..3, sector (q, s) at index 4*(q+12)+s with dimension d(q).
    A holds |q_row - q_inner| <= 2, B holds |q_inner - q_col| <= 1; the key takes no
    part in either rule."""
    qs = np.arange(-12, 13)
    d = _dims(qs, lambda q: max(2, _round_half_away(256 * math.exp(-q * q / 40))))
    rq = np.repeat(qs, 4)
    rd = np.repeat(d, 4)
    return Workload("bf16_localspace_100x25x25", "bf16", Axis(rq, rd), Axis(qs, d), Axis(qs, d),
                    Rule(-2, 2), Rule(-1, 1), "uniform", 0x5EED0000 + 4,
                    layout_a="rowpanel|charge_sorted|align16", layout_b="colpanel|charge_sorted|align16",
                    layout_c="rowpanel|charge_sorted|align16",
                    pack_layout_a="blockrow", pack_layout_b="blockrow",
                    pack_layout_c="blockrow", extra={"key_dim": 4})


def random_sector_axis(s: rng.SplitMix64, n: int, n_big: int, big_dim: int, qlo: int, qhi: int,
                       dlo: int, dhi: int) -> Axis:
    q = np.empty(n, np.int32)
    p = np.empty(n, np.uint8)
    d = np.empty(n, np.int32)
    for t in range(n):
        q[t] = s.uniform_int(qlo, qhi)
        p[t] = s.uniform_int(0, 1)
        d[t] = s.uniform_int(dlo, dhi)
    perm = list(range(n))
    for t in range(n_big):                   # partial Fisher-Yates: n_big distinct indices
        r = s.uniform_int(t, n - 1)
        perm[t], perm[r] = perm[r], perm[t]
    d[perm[:n_big]] = big_dim
    return Axis(q, d, p)


def config5(seed_offset: int = 0, n: int = 2000, n_big: int = 16, big_dim: int = 1024) -> Workload:
    """FP64 launch-bound stress: 2000 random sectors per axis with Z2 x U(1) charges
    (q uniform in -30..30, parity 0/1), dims uniform 1..8 except 16 sectors of 1024;
    both operands hold |dq| <= 1 with equal parity."""
    seed = 0x5EED0000 + 5 + seed_offset
    s = rng.SplitMix64(seed)
    axes = [random_sector_axis(s, n, n_big, big_dim, -30, 30, 1, 8) for _ in range(3)]
    return Workload("fp64_stress_2000x2000x2000", "f64", axes[0], axes[1], axes[2],
                    Rule(-1, 1, True), Rule(-1, 1, True), "normal", seed)


CONFIGS = {1: config1, 2: config2, 3: config3, 4: config4, 5: config5}


def get(n: int) -> Workload:
    return CONFIGS[n]()


def tiny_random(seed: int, values: str = "int3", max_sectors: int = 12, max_dim: int = 6,
                qrange: int = 3, z2: Optional[bool] = None, dtype: str = "f64") -> Workload:
    """A small random structure for brute-force checks: a few sectors per axis with
    repeated charges allowed, random band rules, optional parity."""
    s = rng.SplitMix64(0xC0FFEE00 + seed)
    use_z2 = bool(s.uniform_int(0, 1)) if z2 is None else z2

    def axis():
        n = s.uniform_int(1, max_sectors)
        q = [s.uniform_int(-qrange, qrange) for _ in range(n)]
        d = [s.uniform_int(1, max_dim) for _ in range(n)]
        p = [s.uniform_int(0, 1) for _ in range(n)] if use_z2 else None
        return Axis(np.array(q), np.array(d), None if p is None else np.array(p))

    def rule():
        lo = s.uniform_int(-2, 1)
        hi = s.uniform_int(lo, 2)
        return Rule(lo, hi, use_z2)

    return Workload(f"tiny_random_{seed}", dtype, axis(), axis(), axis(), rule(), rule(), values,
                    0x7E570000 + seed)


def chain2():
    """A two-stage chain shaped like the R/A/B/C apply: T = A B, then Y = T D.

    Stage 1 is the 31-sector tail workload; D maps its column axis to an output
    axis of the same 31 charges with |dq| <= 1 and N(0,1) values.  Returns the
    stage-1 workload and the stage-2 workload whose `rows`/`inner` are T's axes
    and whose rule_b / values describe D (its rule_a is unused: stage 2's
    left operand is T, whose blocks are stage 1's structural product)."""
    w1 = config2()
    w1.layout_c = "rowpanel|charge_sorted"     # T is laid out for the next stage
    qs = np.arange(-15, 16)
    d = _dims(qs, lambda q: max(1, _round_half_away(64 * math.exp(-q * q / 50))))
    out = Axis(qs, d)
    w2 = Workload("chain_stage2_31x31x31", "f64", w1.rows, w1.cols, out, Rule(-100, 100), Rule(-1, 1),
                  "normal", 0x5EED0000 + 102, layout_a="rowpanel|charge_sorted",
                  layout_b="colpanel|charge_sorted", layout_c="blockrow")
    return w1, w2
