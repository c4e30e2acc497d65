"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each pin checks the oracle against something fixed by the pages or by
mathematics: hand-derived golden fixtures (tests/golden), a dense embedding
multiplied by numpy's matmul (for C, and for the conditioning scale S, which
must equal the dense product of the elementwise magnitudes |A| |B|), charge
conservation, closed forms for all-ones inputs, the one-sector case that is a
textbook GEMM, and exactness of integer arithmetic.  The last test plants mistakes in copies of the oracle's C source
and requires that every planted mistake trips at least one pin.
"""
import json
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest

import bsgen
import oracle
from bsgen import Axis, Rule

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def rule_np(ax_r, ax_c, rule):
    """The allowed-charge rule of the workload description, in numpy."""
    dq = ax_r.q[:, None].astype(np.int64) - ax_c.q[None, :].astype(np.int64)
    m = (dq >= rule.dq_min) & (dq <= rule.dq_max)
    if rule.z2:
        m &= ax_r.p[:, None] == ax_c.p[None, :]
    return m


def dense_operand(w, op, ax_r, ax_c, rule):
    """Scatter the seeded blocks of one operand into a dense matrix (sector index order)."""
    rs = np.concatenate([[0], np.cumsum(ax_r.d)])
    cs = np.concatenate([[0], np.cumsum(ax_c.d)])
    D = np.zeros((rs[-1], cs[-1]))
    for r, c in zip(*np.nonzero(rule_np(ax_r, ax_c, rule))):
        v = w.draw(op, [r], [c], [ax_r.d[r]], [ax_c.d[c]]).reshape(ax_r.d[r], ax_c.d[c])
        D[rs[r]:rs[r + 1], cs[c]:cs[c + 1]] = v
    return D, rs, cs


def check_dense_embedding(w, la=None, lb=None, lc=None, exact=False, rtol=1e-14):
    """Oracle C against the dense product; returns a list of failure strings."""
    fails = []
    pr = oracle.problem(w, la, lb, lc)
    C, S = oracle.contract(pr)
    DA, ri, ki = dense_operand(w, 0, w.rows, w.inner, w.rule_a)
    DB, _, cj = dense_operand(w, 1, w.inner, w.cols, w.rule_b)
    DC = DA @ DB
    # the conditioning scale: S = sum over the same terms of |a| |b|, i.e. the
    # dense product of the elementwise magnitudes, restricted to populated C
    DS = np.abs(DA) @ np.abs(DB)
    # the oracle's operand buffers hold exactly the seeded blocks
    for (r, c) in zip(*np.nonzero(pr.ma)):
        blk = oracle.block_view(pr.A, pr.la, r, c)
        if w.dtype == "bf16":
            blk = (blk.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        if not np.array_equal(blk, DA[ri[r]:ri[r + 1], ki[c]:ki[c + 1]]):
            fails.append(f"A block {r},{c} misplaced")
            break
    for i in range(w.rows.n):
        for j in range(w.cols.n):
            ref = DC[ri[i]:ri[i + 1], cj[j]:cj[j + 1]]
            if not pr.mc[i, j]:
                if np.any(ref != 0.0):
                    fails.append(f"C block {i},{j} absent from the oracle but nonzero in the dense product")
                continue
            got = oracle.block_view(C, pr.lc, i, j)
            s = oracle.block_view(S, pr.lc, i, j)
            sref = DS[ri[i]:ri[i + 1], cj[j]:cj[j + 1]]
            if exact:
                if not np.array_equal(got, ref):
                    fails.append(f"C block {i},{j} differs (exact)")
                if not np.array_equal(s, sref):
                    fails.append(f"S block {i},{j} differs from |A| |B| (exact)")
            else:
                if np.linalg.norm(got - ref) > rtol * max(np.linalg.norm(s), 1e-300):
                    fails.append(f"C block {i},{j} differs beyond {rtol} of its scale")
                if np.linalg.norm(s - sref) > rtol * max(np.linalg.norm(sref), 1e-300):
                    fails.append(f"S block {i},{j} differs from |A| |B| beyond {rtol}")
    return fails


def count_triples(ma, mb):
    return int((ma.astype(np.int64) @ mb.astype(np.int64)).sum())


# ---------------------------------------------------------------- golden fixtures
def check_layout_golden():
    fails = []
    g = json.load(open(os.path.join(GOLDEN, "layout_small.json")))
    rows = Axis(np.array(g["rows"]["q"]), np.array(g["rows"]["d"]))
    cols = Axis(np.array(g["cols"]["q"]), np.array(g["cols"]["d"]))
    mask = np.zeros((rows.n, cols.n), np.uint8)
    for r, c in g["populated"]:
        mask[r, c] = 1
    for case in g["cases"]:
        lay = oracle.layout(rows, cols, mask, case["flags"], g["elem_bytes"])
        if lay.nelems != case["nelems"]:
            fails.append(f"{case['flags']}: nelems {lay.nelems} != {case['nelems']}")
        for r, c, off, ld in case["blocks"]:
            if lay.off[r, c] != off or lay.ld[r, c] != ld:
                fails.append(f"{case['flags']}: block {r},{c} at ({lay.off[r, c]},{lay.ld[r, c]}) not ({off},{ld})")
        if int((lay.off >= 0).sum()) != len(case["blocks"]):
            fails.append(f"{case['flags']}: wrong block count")
    return fails


def check_band_golden():
    fails = []
    g = json.load(open(os.path.join(GOLDEN, "band_structure.json")))
    for n, want in g["configs"].items():
        w = bsgen.get(int(n))
        ma = oracle.rule_mask(w.rows, w.inner, w.rule_a)
        mb = oracle.rule_mask(w.inner, w.cols, w.rule_b)
        mc = oracle.product_mask(ma, mb)
        got = {"a_blocks": int(ma.sum()), "b_blocks": int(mb.sum()), "c_blocks": int(mc.sum()),
               "triples": count_triples(ma, mb)}
        if "a_elems" in want:
            got["a_elems"] = oracle.layout(w.rows, w.inner, ma, "blockrow", 8).nelems
            got["c_elems"] = oracle.layout(w.rows, w.cols, mc, "blockrow", 8).nelems
        for key, v in got.items():
            if want.get(key, v) != v:
                fails.append(f"config {n}: {key} = {v}, closed form {want[key]}")
    return fails


def test_layout_golden():
    assert check_layout_golden() == []


def test_band_structure_golden():
    assert check_band_golden() == []


# ---------------------------------------------------------------- dense embedding
LAYOUT_VARIANTS = [
    (None, None, None),
    ("blockrow", "blockrow", "blockrow"),
    ("rowpanel", "colpanel", "rowpanel|align16"),
    ("colpanel|charge_sorted", "rowpanel|charge_sorted", "colpanel|charge_sorted"),
]


@pytest.mark.parametrize("cfg", [1, 2])
@pytest.mark.parametrize("lay", LAYOUT_VARIANTS)
def test_dense_embedding_band_configs(cfg, lay):
    assert check_dense_embedding(bsgen.get(cfg), *lay) == []


@pytest.mark.parametrize("seed", range(12))
def test_dense_embedding_tiny_random_integer_exact(seed):
    w = bsgen.tiny_random(seed, values="int3")
    lay = LAYOUT_VARIANTS[seed % len(LAYOUT_VARIANTS)]
    assert check_dense_embedding(w, *lay, exact=True) == []


@pytest.mark.parametrize("seed", range(4))
def test_dense_embedding_tiny_random_normal(seed):
    w = bsgen.tiny_random(100 + seed, values="normal", max_sectors=20, max_dim=9)
    assert check_dense_embedding(w) == []


def test_dense_embedding_bf16_inputs():
    """bfloat16 operands are widened exactly: integer inputs give an exact product."""
    w = bsgen.tiny_random(7, values="int3", dtype="bf16")
    w.layout_a, w.layout_b, w.layout_c = "rowpanel|align16", "colpanel|align16", "rowpanel|align16"
    assert check_dense_embedding(w, exact=True) == []
    w2 = bsgen.tiny_random(8, values="uniform", dtype="bf16", max_sectors=16, max_dim=12)
    assert check_dense_embedding(w2) == []


# ---------------------------------------------------------------- invariants
@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_charge_conservation(cfg):
    """Every populated C block obeys the composed rule; on the band workloads every
    pair obeying it is populated (a witness k exists)."""
    w = bsgen.get(cfg)
    ma = oracle.rule_mask(w.rows, w.inner, w.rule_a)
    mb = oracle.rule_mask(w.inner, w.cols, w.rule_b)
    mc = oracle.product_mask(ma, mb).astype(bool)
    composed = Rule(w.rule_a.dq_min + w.rule_b.dq_min, w.rule_a.dq_max + w.rule_b.dq_max,
                    w.rule_a.z2 and w.rule_b.z2)
    allowed = rule_np(w.rows, w.cols, composed)
    assert not np.any(mc & ~allowed)
    if cfg in (1, 2, 3, 4):
        assert np.array_equal(mc, allowed)


def test_closed_form_ones_unit_dims():
    """All dims 1 and all values 1: C[i,j] counts the k allowed by both rules, which on
    consecutive charges -4..4 with bands of 1 is the length of
    [max(qi,qj)-1, min(qi,qj)+1] clipped to [-4, 4]."""
    qs = np.arange(-4, 5)
    ax = Axis(qs, np.ones(9))
    w = bsgen.Workload("ones", "f64", ax, Axis(qs, np.ones(9)), Axis(qs, np.ones(9)), Rule(-1, 1),
                       Rule(-1, 1), "ones", 1, layout_a="blockrow", layout_b="blockrow", layout_c="blockrow")
    pr = oracle.problem(w)
    C, _ = oracle.contract(pr)
    for i, qi in enumerate(qs):
        for j, qj in enumerate(qs):
            lo, hi = max(qi, qj) - 1, min(qi, qj) + 1
            want = max(0, min(hi, 4) - max(lo, -4) + 1)
            if want == 0:
                assert pr.lc.off[i, j] < 0
            else:
                assert C[pr.lc.off[i, j]] == want
    assert C[pr.lc.off[4, 4]] == 3 and C[pr.lc.off[4, 6]] == 1


def test_closed_form_ones_real_dims():
    """All values 1: every element of C[i,j] equals the sum of d_k over shared k."""
    w = bsgen.config2()
    w.values = "ones"
    pr = oracle.problem(w)
    C, _ = oracle.contract(pr)
    q, d = w.inner.q, w.inner.d
    for i in range(w.rows.n):
        for j in range(w.cols.n):
            ks = [k for k in range(len(q)) if abs(w.rows.q[i] - q[k]) <= 1 and abs(q[k] - w.cols.q[j]) <= 1]
            if not ks:
                continue
            blk = oracle.block_view(C, pr.lc, i, j)
            assert np.all(blk == sum(int(d[k]) for k in ks))


def test_single_sector_is_a_dense_gemm():
    """One sector per axis reduces to one dense GEMM: compare with numpy and with a naive loop."""
    for (m, k, n) in [(1, 1, 1), (7, 5, 3), (17, 33, 9)]:
        w = bsgen.Workload("one", "f64", Axis([0], [m]), Axis([0], [k]), Axis([0], [n]), Rule(0, 0),
                           Rule(0, 0), "normal", 99, layout_a="blockrow", layout_b="blockrow", layout_c="blockrow")
        pr = oracle.problem(w)
        C, _ = oracle.contract(pr)
        A = pr.A.reshape(m, k)
        B = pr.B.reshape(k, n)
        np.testing.assert_allclose(C.reshape(m, n), A @ B, rtol=1e-13, atol=1e-13)
        naive = np.zeros((m, n))
        for r in range(m):
            for c in range(n):
                s = 0.0
                for p in range(k):
                    s = s + A[r, p] * B[p, c]
                naive[r, c] = s
        assert np.array_equal(C.reshape(m, n), naive)   # same order, same roundings


def test_selected_blocks_match_full_run():
    w = bsgen.config2()
    pr = oracle.problem(w)
    C, S = oracle.contract(pr)
    sel = np.argwhere(pr.mc)[::7]
    C2, S2 = oracle.contract(pr, sel)
    for i, j in sel:
        assert np.array_equal(oracle.block_view(C2, pr.lc, i, j), oracle.block_view(C, pr.lc, i, j))


# ---------------------------------------------------------------- planted mistakes
MUTANTS = {
    "sign_of_product": ("acc = acc + prod;", "acc = acc - prod;"),
    "dropped_inner_term": ("for (int32_t p = 0; p < dk[k]; ++p) {", "for (int32_t p = 1; p < dk[k]; ++p) {"),
    "reversed_a_index": ("ao + (int64_t)r * al + p", "ao + (int64_t)r * al + (dk[k] - 1 - p)"),
    "mirrored_b_column": ("bo + (int64_t)p * bl + c", "bo + (int64_t)p * bl + (dj[j] - 1 - c)"),
    "product_mask_misses_first_column": ("if (mb[(size_t)k * nj + j]) mc", "if (j > 0 && mb[(size_t)k * nj + j]) mc"),
    "rule_lower_bound_strict": ("int ok = dq >= dq_min && dq <= dq_max;", "int ok = dq > dq_min && dq <= dq_max;"),
    "rowpanel_ignores_alignment": ("col += round_up(cd[c], al);", "col += cd[c];"),
    "charge_order_reversed": ("int before = q[v] < q[w]", "int before = q[v] > q[w]"),
    "bf16_widening_shift": ("<< 16;", "<< 15;"),
    "parity_ignored": ("if (z2 && ok) ok = rp[r] == cp[c];", "(void)rp; (void)cp;"),
    "scale_drops_magnitude": ("mag = mag + (prod < 0 ? -prod : prod);", "mag = mag + prod;"),
    "scale_skips_first_term": ("mag = mag + (prod < 0 ? -prod : prod);", "if (u + p > 0) mag = mag + (prod < 0 ? -prod : prod);"),
}


def run_pins():
    fails = check_layout_golden() + check_band_golden()
    for seed in range(6):
        fails += check_dense_embedding(bsgen.tiny_random(seed, values="int3", z2=True), *LAYOUT_VARIANTS[seed % 4],
                                       exact=True)
    wb = bsgen.tiny_random(7, values="int3", dtype="bf16")
    fails += check_dense_embedding(wb, exact=True)
    wc = bsgen.config1()
    fails += check_dense_embedding(wc, "rowpanel|align16", "colpanel|charge_sorted", "blockrow")
    return fails


def test_pins_pass_on_the_real_oracle():
    assert run_pins() == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name):
    old, new = MUTANTS[name]
    src = open(oracle._build.SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not unique"
    tmp = tempfile.mkdtemp()
    try:
        path = os.path.join(tmp, "mut.c")
        open(path, "w").write(src.replace(old, new))
        so = os.path.join(tmp, "libmut.so")
        subprocess.run(["gcc", "-O1", "-ffp-contract=off", "-fPIC", "-shared", "-o", so, path], check=True)
        prev = oracle.use(oracle.load(so))
        try:
            fails = run_pins()
        finally:
            oracle.use(prev)
        assert fails, f"planted mistake {name} went unnoticed"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)


def test_chain_matches_dense_triple_product():
    """The two-stage chain Y = (A B) D equals the dense product of the three embeddings."""
    w1, w2 = bsgen.chain2()
    pr1 = oracle.problem(w1)
    T, _ = oracle.contract(pr1)
    pr2 = oracle.chain_stage2(pr1, T, w2)
    Y, S = oracle.contract(pr2)
    DA, ri, ki = dense_operand(w1, 0, w1.rows, w1.inner, w1.rule_a)
    DB, _, cj = dense_operand(w1, 1, w1.inner, w1.cols, w1.rule_b)
    DD, _, oj = dense_operand(w2, 1, w2.inner, w2.cols, w2.rule_b)
    DY = (DA @ DB) @ DD
    for i in range(w2.rows.n):
        for j in range(w2.cols.n):
            ref = DY[ri[i]:ri[i + 1], oj[j]:oj[j + 1]]
            if not pr2.mc[i, j]:
                assert np.all(ref == 0.0)
                continue
            got = oracle.block_view(Y, pr2.lc, i, j)
            s = oracle.block_view(S, pr2.lc, i, j)
            assert np.linalg.norm(got - ref) <= 1e-13 * max(np.linalg.norm(s), 1e-300)
