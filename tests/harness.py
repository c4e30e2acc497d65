"""Test-side helpers for running the library on seeded workloads and comparing with the oracle.

Placement of seeded values into the library's layouts is written here, apart
from the oracle's own placement code; the two meet only through `bsgen`.
"""
from __future__ import annotations

import numpy as np

import bsgen
import oracle

TOL = {"f64": 1e-12, "bf16": 5e-3}
KAPPA_MAX = 1e4


def element_index(blocks: np.ndarray) -> np.ndarray:
    """Buffer index of every element of every block (row-major within a block, blocks in the given order)."""
    if len(blocks) == 0:
        return np.zeros(0, np.int64)
    rows, cols = blocks[:, 3], blocks[:, 4]
    sizes = rows * cols
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]])
    rep = np.repeat(np.arange(len(blocks)), sizes)
    local = np.arange(int(sizes.sum()), dtype=np.int64) - starts[rep]
    c = cols[rep]
    return blocks[rep, 2] + (local // c) * blocks[rep, 5] + local % c


def operand_host(w: bsgen.Workload, op: int, blocks: np.ndarray, nelems: int) -> np.ndarray:
    """Host buffer of one operand in a library layout: doubles, or bf16 bit patterns."""
    vals = w.draw(op, blocks[:, 0], blocks[:, 1], blocks[:, 3], blocks[:, 4])
    buf = np.zeros(nelems, np.float64)
    buf[element_index(blocks)] = vals
    if w.dtype == "bf16":
        return bsgen.rng.bf16_bits(buf)
    return buf


def sort_rc(blocks: np.ndarray) -> np.ndarray:
    return blocks[np.lexsort((blocks[:, 1], blocks[:, 0]))]


def block_errors(c_got: np.ndarray, c_ref: np.ndarray, s_ref: np.ndarray, blocks: np.ndarray):
    """Per block: ||got - ref||_F, ||ref||_F, ||S||_F (S = sum of |a||b|)."""
    idx = element_index(blocks)
    sizes = blocks[:, 3] * blocks[:, 4]
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    d2 = (c_got[idx].astype(np.float64) - c_ref[idx]) ** 2
    r2 = c_ref[idx] ** 2
    s2 = s_ref[idx] ** 2
    red = lambda x: np.sqrt(np.add.reduceat(x, starts)) if len(x) else np.zeros(0)
    return red(d2), red(r2), red(s2)


def check_blocks(c_got, c_ref, s_ref, blocks, tol):
    """Max per-block relative Frobenius error; blocks whose sum cancels (||S|| / ||C|| > 1e4)
    are judged against ||S|| instead.  Returns (ok, worst, n_cancelling)."""
    err, ref, sc = block_errors(c_got, c_ref, s_ref, blocks)
    kappa = sc / np.maximum(ref, 1e-300)
    cancel = kappa > KAPPA_MAX
    rel = np.where(cancel, err / np.maximum(sc, 1e-300), err / np.maximum(ref, 1e-300))
    rel = np.where((ref == 0) & (sc == 0), err, rel)
    worst = float(rel.max()) if len(rel) else 0.0
    return worst <= tol, worst, int(cancel.sum())


# ---------------------------------------------------------------- the oracle over every host core
_POOL_PR = None


def _pool_init(w, flags):
    global _POOL_PR
    _POOL_PR = oracle.problem(w, *flags)


def _pool_blocks(sel):
    """Oracle C and S values of the listed (i, j) blocks, concatenated block after
    block (row-major inside a block), in the order of `sel`."""
    C, S = oracle.contract(_POOL_PR, sel=sel)
    lc = _POOL_PR.lc
    blk = np.array([[i, j, lc.off[i, j], lc.rows[i], lc.cols[j], lc.ld[i, j]] for i, j in sel], np.int64)
    idx = element_index(blk)
    return C[idx], S[idx]


def oracle_all_blocks(w, la, lb, lc, workers: int = 0):
    """(C, S, problem) of the whole workload, its C blocks dealt longest-first by
    flops over spawned worker processes (spawned, so none inherits a CUDA context);
    each worker runs the plain oracle on its blocks."""
    import multiprocessing as mp
    import os
    pr = oracle.problem(w, la, lb, lc)
    ij = np.argwhere(pr.mc)
    if len(ij) == 0:
        return np.zeros(pr.lc.nelems), np.zeros(pr.lc.nelems), pr
    kd = pr.ma.astype(np.float64) * w.inner.d[None, :].astype(np.float64)    # d_k where A[i,k]
    ksum = kd @ pr.mb.astype(np.float64)                                      # sum of d_k over shared k
    cost = w.rows.d[ij[:, 0]].astype(np.float64) * w.cols.d[ij[:, 1]] * ksum[ij[:, 0], ij[:, 1]]
    n = max(1, min(workers or len(os.sched_getaffinity(0)), len(ij)))
    load = np.zeros(n)
    parts = [[] for _ in range(n)]
    for t in np.argsort(-cost, kind="stable"):
        b = int(np.argmin(load))
        load[b] += cost[t]
        parts[b].append(ij[t])
    parts = [np.asarray(p, np.int32).reshape(-1, 2) for p in parts if p]
    C = np.zeros(pr.lc.nelems)
    S = np.zeros(pr.lc.nelems)
    with mp.get_context("spawn").Pool(len(parts), initializer=_pool_init, initargs=(w, (la, lb, lc))) as pool:
        for sel, (cv, sv) in zip(parts, pool.map(_pool_blocks, parts, chunksize=1)):
            lcb = pr.lc
            blk = np.array([[i, j, lcb.off[i, j], lcb.rows[i], lcb.cols[j], lcb.ld[i, j]] for i, j in sel], np.int64)
            idx = element_index(blk)
            C[idx] = cv
            S[idx] = sv
    return C, S, pr
