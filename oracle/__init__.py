"""CPU oracle for the block-sparse contraction (test infrastructure only).

Only the tests, the smoke check and the bench's CPU-baseline leg may import
this package.  It wraps the plain-C oracle (bs_oracle.c) through ctypes and
places the seeded values of `bsgen` into buffers laid out by the oracle's own
restatement of the layout rules.  It shares nothing with the CUDA library.

Every function here follows the uni20 design note "block coalescing"
(Summary; "Why single-axis coalescing is hole-free"): the result of any
coalesced lowering equals the plain sum over populated (i, k, j) triples.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np

from . import build as _build

_lib = None

FLAG_BITS = {"blockrow": 0, "rowpanel": 1, "colpanel": 2, "charge_sorted": 4, "align16": 8, "align64": 16}


def load(path: str):
    """Load an oracle shared object and declare its C signatures."""
    L = ctypes.CDLL(path)
    P = ctypes.c_void_p
    i32, i64, u32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    L.bso_rule_mask.argtypes = [i32, P, P, i32, P, P, i32, i32, i32, P]
    L.bso_rule_mask.restype = None
    L.bso_product_mask.argtypes = [i32, i32, i32, P, P, P]
    L.bso_product_mask.restype = None
    L.bso_layout.argtypes = [i32, P, P, P, i32, P, P, P, P, u32, i32, P, P, P]
    L.bso_layout.restype = i32
    L.bso_contract.argtypes = [i32, i32, i32, P, P, P, P, P, P, P, P, P, i32, P, P, P, P, i64, P]
    L.bso_contract.restype = i64
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = load(_build.build())
    return _lib


def use(L):
    """Swap the loaded oracle library (tests load deliberately broken builds this way)."""
    global _lib
    old, _lib = _lib, L
    return old


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def parse_flags(name: str) -> int:
    f = 0
    for part in name.split("|"):
        part = part.strip()
        if part:
            f |= FLAG_BITS[part]
    return f


def rule_mask(ax_r, ax_c, rule) -> np.ndarray:
    """Populated-block mask (nr x nc, uint8) of an allowed-charge rule."""
    m = np.zeros((ax_r.n, ax_c.n), np.uint8)
    rp = ax_r.p if ax_r.p is not None else np.zeros(ax_r.n, np.uint8)
    cp = ax_c.p if ax_c.p is not None else np.zeros(ax_c.n, np.uint8)
    lib().bso_rule_mask(ax_r.n, _p(ax_r.q), _p(rp), ax_c.n, _p(ax_c.q), _p(cp), rule.dq_min,
                        rule.dq_max, 1 if rule.z2 else 0, _p(m))
    return m


def product_mask(ma: np.ndarray, mb: np.ndarray) -> np.ndarray:
    ni, nk = ma.shape
    nj = mb.shape[1]
    mc = np.zeros((ni, nj), np.uint8)
    lib().bso_product_mask(ni, nk, nj, _p(np.ascontiguousarray(ma)), _p(np.ascontiguousarray(mb)), _p(mc))
    return mc


@dataclass
class Layout:
    off: np.ndarray      # int64 nr x nc, -1 where absent
    ld: np.ndarray       # int64 nr x nc
    nelems: int
    rows: np.ndarray     # d of the row axis
    cols: np.ndarray     # d of the column axis

    def blocks(self):
        """(row, col, offset, rows, cols, ld) of every populated block, by (row, col)."""
        r, c = np.nonzero(self.off >= 0)
        return np.stack([r, c, self.off[r, c], self.rows[r], self.cols[c], self.ld[r, c]], 1).astype(np.int64)


def layout(ax_r, ax_c, mask: np.ndarray, flags: str, elem_bytes: int) -> Layout:
    off = np.empty(mask.shape, np.int64)
    ld = np.empty(mask.shape, np.int64)
    ne = np.zeros(1, np.int64)
    rp = ax_r.p if ax_r.p is not None else None
    cp = ax_c.p if ax_c.p is not None else None
    rc = lib().bso_layout(ax_r.n, _p(ax_r.q), _p(rp), _p(ax_r.d), ax_c.n, _p(ax_c.q), _p(cp), _p(ax_c.d),
                          _p(np.ascontiguousarray(mask)), parse_flags(flags), elem_bytes, _p(off), _p(ld), _p(ne))
    if rc != 0:
        raise RuntimeError(f"bso_layout failed: {rc}")
    return Layout(off, ld, int(ne[0]), ax_r.d.copy(), ax_c.d.copy())


def place(values: np.ndarray, lay: Layout, nelems_dtype=np.float64, fill=0.0) -> np.ndarray:
    """Scatter block-row-major concatenated values (in (row, col) block order) into a buffer."""
    buf = np.full(lay.nelems, fill, dtype=nelems_dtype)
    pos = 0
    for (r, c, off, nr, nc, ld) in lay.blocks():
        n = nr * nc
        blk = values[pos:pos + n].reshape(nr, nc)
        idx = off + np.arange(nr)[:, None] * ld + np.arange(nc)[None, :]
        buf[idx] = blk
        pos += n
    return buf


def operand(w, op: int, ax_r, ax_c, mask, flags: str):
    """Buffer of operand `op` of workload `w` (doubles, or bf16 bit patterns)."""
    eb = 2 if w.dtype == "bf16" else 8
    lay = layout(ax_r, ax_c, mask, flags, eb)
    b = lay.blocks()
    vals = w.draw(op, b[:, 0], b[:, 1], b[:, 3], b[:, 4])
    buf = place(vals, lay)
    if w.dtype == "bf16":
        from bsgen import rng
        buf = rng.bf16_bits(buf)
    return buf, lay


@dataclass
class Problem:
    w: object
    ma: np.ndarray
    mb: np.ndarray
    mc: np.ndarray
    la: Layout
    lb: Layout
    lc: Layout
    A: np.ndarray
    B: np.ndarray


def problem(w, la_flags=None, lb_flags=None, lc_flags=None) -> Problem:
    """Masks, layouts and operand buffers of a workload, built by the oracle's own code."""
    la_flags = w.layout_a if la_flags is None else la_flags
    lb_flags = w.layout_b if lb_flags is None else lb_flags
    lc_flags = w.layout_c if lc_flags is None else lc_flags
    ma = rule_mask(w.rows, w.inner, w.rule_a)
    mb = rule_mask(w.inner, w.cols, w.rule_b)
    mc = product_mask(ma, mb)
    A, la = operand(w, 0, w.rows, w.inner, ma, la_flags)
    B, lb = operand(w, 1, w.inner, w.cols, mb, lb_flags)
    lc = layout(w.rows, w.cols, mc, lc_flags, 4 if w.dtype == "bf16" else 8)
    return Problem(w, ma, mb, mc, la, lb, lc, A, B)


def contract(pr: Problem, sel=None):
    """(C, S) in C's layout as doubles; with `sel` (array of (i, j)) only those blocks."""
    w = pr.w
    C = np.zeros(pr.lc.nelems, np.float64)
    S = np.zeros(pr.lc.nelems, np.float64)
    dt = 1 if w.dtype == "bf16" else 0
    if sel is None:
        nsel, selp = 0, None
    else:
        sel = np.ascontiguousarray(np.asarray(sel, dtype=np.int32).reshape(-1, 2))
        nsel, selp = len(sel), sel
    lib().bso_contract(w.rows.n, w.inner.n, w.cols.n, _p(w.rows.d), _p(w.inner.d), _p(w.cols.d),
                       _p(pr.la.off), _p(pr.la.ld), _p(pr.lb.off), _p(pr.lb.ld), _p(pr.lc.off), _p(pr.lc.ld),
                       dt, _p(pr.A), _p(pr.B), _p(C), _p(S), nsel, _p(selp))
    return C, S


def block_view(buf: np.ndarray, lay: Layout, r: int, c: int) -> np.ndarray:
    off, ld = lay.off[r, c], lay.ld[r, c]
    nr, nc = lay.rows[r], lay.cols[c]
    idx = off + np.arange(nr)[:, None] * ld + np.arange(nc)[None, :]
    return buf[idx]


def chain_stage2(pr1: Problem, T: np.ndarray, w2, lb_flags=None, lc_flags=None) -> Problem:
    """Second stage of a chain Y = T D, T being stage 1's C (values in stage 1's C layout).

    T's populated blocks are stage 1's structural product; D follows w2's rule_b
    and values (drawn as operand 1 of w2).  The contraction is the same plain
    per-triple sum ("Two coalescing modes" does not change what is computed).
    """
    ma = pr1.mc
    mb = rule_mask(w2.inner, w2.cols, w2.rule_b)
    mc = product_mask(ma, mb)
    B, lb = operand(w2, 1, w2.inner, w2.cols, mb, lb_flags or w2.layout_b)
    lc = layout(w2.rows, w2.cols, mc, lc_flags or w2.layout_c, 8)
    return Problem(w2, ma, mb, mc, pr1.lc, lb, lc, T, B)
