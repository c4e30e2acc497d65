"""Host-side checks of libbs.so that need no GPU.

- the shared library loads and exports every entry point include/bs.h declares;
- layouts built by the library equal the oracle's layouts bit for bit;
- host-only plans cover every populated triple exactly once, with hole-free
  single-axis groups, and build the same C layout as the oracle;
- argument errors come back as status codes.
"""
import os
import re

import numpy as np
import pytest

import bsgen
import oracle

bs = pytest.importorskip("block_sparse_tensor_gb300")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_library_exports_every_declared_symbol():
    header = open(os.path.join(ROOT, "include", "bs.h")).read()
    declared = set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]*?\b(bs_\w+)\s*\(", header, re.M))
    assert len(declared) >= 15
    for name in declared:
        assert hasattr(bs.lib, name), f"{name} declared but not exported"
    assert set(bs.EXPORTED) <= declared
    assert bs.version().startswith("bs ")


LAYOUT_FLAGS = ["blockrow", "rowpanel", "colpanel", "blockrow|charge_sorted", "rowpanel|charge_sorted",
                "colpanel|charge_sorted", "rowpanel|align16", "colpanel|charge_sorted|align16", "blockrow|align16",
                "rowpanel|charge_sorted|align64", "colpanel|align64", "blockrow|align16|align64"]


def lib_blocks_by_rc(layout):
    b = layout.blocks()
    order = np.lexsort((b[:, 1], b[:, 0]))
    return b[order]


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
@pytest.mark.parametrize("flags", LAYOUT_FLAGS)
def test_layout_matches_oracle(cfg, flags):
    w = bsgen.get(cfg)
    eb = 2 if w.dtype == "bf16" else 8
    for ax_r, ax_c, rule in [(w.rows, w.inner, w.rule_a), (w.inner, w.cols, w.rule_b)]:
        L = bs.Layout(ax_r, ax_c, rule, flags, eb)
        mask = oracle.rule_mask(ax_r, ax_c, rule)
        ol = oracle.layout(ax_r, ax_c, mask, flags, eb)
        assert L.nelems == ol.nelems
        assert np.array_equal(lib_blocks_by_rc(L), ol.blocks())


def test_layout_matches_oracle_config5():
    w = bsgen.config5()
    for flags in ["blockrow", "rowpanel|charge_sorted", "colpanel|charge_sorted"]:
        L = bs.Layout(w.rows, w.inner, w.rule_a, flags, 8)
        ol = oracle.layout(w.rows, w.inner, oracle.rule_mask(w.rows, w.inner, w.rule_a), flags, 8)
        assert L.nelems == ol.nelems
        assert np.array_equal(lib_blocks_by_rc(L), ol.blocks())


def host_plan(w, la=None, lb=None, **opts):
    eb = 2 if w.dtype == "bf16" else 8
    A = bs.Layout(w.rows, w.inner, w.rule_a, la or w.layout_a, eb)
    B = bs.Layout(w.inner, w.cols, w.rule_b, lb or w.layout_b, eb)
    dt = bs.BF16_F32 if w.dtype == "bf16" else bs.F64
    opts.setdefault("c_layout_flags", w.layout_c)
    return bs.Plan(A, B, dt, host_only=1, **opts), A, B


def oracle_triples(w):
    ma = oracle.rule_mask(w.rows, w.inner, w.rule_a).astype(bool)
    mb = oracle.rule_mask(w.inner, w.cols, w.rule_b).astype(bool)
    out = set()
    for i, k in zip(*np.nonzero(ma)):
        for j in np.nonzero(mb[k])[0]:
            out.add((int(i), int(k), int(j)))
    return out, ma, mb


POLICIES = [dict(axis_policy=bs.AXIS_CONTRACTION), dict(axis_policy=bs.AXIS_FREE), dict(axis_policy=bs.AXIS_NONE),
            dict(axis_policy=bs.AXIS_AUTO), dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS),
            dict(axis_policy=bs.AXIS_FREE, pack_policy=bs.PACK_ALWAYS)]


@pytest.mark.parametrize("cfg", [1, 2, 3])
@pytest.mark.parametrize("pol", range(len(POLICIES)))
@pytest.mark.parametrize("lay", [(None, None), ("blockrow", "blockrow")])
def test_plan_covers_each_triple_once_and_is_hole_free(cfg, pol, lay):
    w = bsgen.get(cfg)
    P, A, B = host_plan(w, *lay, **POLICIES[pol])
    want, ma, mb = oracle_triples(w)
    ptr, tr = P.triples()
    got = [tuple(int(x) for x in t) for t in tr]
    assert len(got) == len(set(got)) == len(want)
    assert set(got) == want
    st = P.stats()
    assert st["triples"] == len(want)
    # every group is one axis: a contraction group has one (i, j) (or stacked i's
    # with the same k list); a free group has one (k, j); nothing else
    for g in range(len(ptr) - 1):
        t = tr[ptr[g]:ptr[g + 1]]
        ks = {int(x) for x in t[:, 1]}
        js = {int(x) for x in t[:, 2]}
        is_ = {int(x) for x in t[:, 0]}
        assert len(js) == 1
        if st["axis"] == bs.AXIS_CONTRACTION:
            # hole-free: every (i, k) pair of the rectangle exists
            for i in is_:
                for k in ks:
                    assert ma[i, k] and mb[k, next(iter(js))]
        elif st["axis"] == bs.AXIS_FREE:
            assert len(ks) == 1
        else:
            assert len(t) == 1
    flops = sum(2 * int(w.rows.d[i]) * int(w.inner.d[k]) * int(w.cols.d[j]) for (i, k, j) in want)
    assert st["useful_flops"] == pytest.approx(flops, rel=1e-12)
    # the library's own proof: blocks tile every group and sit where its views point
    assert P.check_groups() == (0, -1)


@pytest.mark.parametrize("cfg", [1, 2, 4])
def test_plan_c_layout_matches_oracle(cfg):
    w = bsgen.get(cfg)
    P, _, _ = host_plan(w)
    pr = oracle.problem(w)
    assert P.c_layout.nelems == pr.lc.nelems
    assert np.array_equal(lib_blocks_by_rc(P.c_layout), pr.lc.blocks())


def test_localspace_keys_merge_into_taller_groups():
    """Config 4: the four LocalSpace key rows of a charge share every inner block and
    sit in consecutive row panels with one stride, so they stack into one group."""
    w = bsgen.config4()
    P, _, _ = host_plan(w)
    g = P.groups()
    st = P.stats()
    assert st["triples"] == 1404
    assert st["c_blocks"] == 652
    assert len(g) == 652 // 4
    assert np.all(g[:, 1] % 4 == 0)
    P2, _, _ = host_plan(w, merge_rows=0)
    assert len(P2.groups()) == 652
    # two-axis groups (four key rows x several inner sectors), each proved hole-free
    ptr, tr = P.triples()
    two_axis = sum(1 for g0, g1 in zip(ptr[:-1], ptr[1:])
                   if len(set(tr[g0:g1, 0])) == 4 and len(set(tr[g0:g1, 1])) > 1)
    assert two_axis > 100
    assert P.check_groups() == (0, -1)
    assert P2.check_groups() == (0, -1)
    P3, _, _ = host_plan(w, pack_policy=bs.PACK_ALWAYS, la="blockrow", lb="blockrow")
    assert P3.check_groups() == (0, -1)


def _two_row_problem():
    """Two row sectors (charges 0 and 1) of equal dimension whose inner blocks
    differ (charges -1..1 and 0..2) but have the same count and panel width."""
    rows = bsgen.Axis(np.array([0, 1]), np.array([2, 2]))
    inner = bsgen.Axis(np.array([-1, 0, 1, 2]), np.array([3, 3, 3, 3]))
    cols = bsgen.Axis(np.array([0]), np.array([2]))
    A = bs.Layout(rows, inner, bsgen.Rule(-1, 1), "rowpanel|charge_sorted", 8)
    B = bs.Layout(inner, cols, bsgen.Rule(-10, 10), "colpanel|charge_sorted", 8)
    return A, B


def test_group_validator_finds_a_planted_hole():
    """With the same-inner-blocks check switched off, row stacking puts both rows
    into one group whose 2 x 4 rectangle holds only 6 of its 8 blocks: the
    validator must report that group.  With the check on, the rows stay apart."""
    A, B = _two_row_problem()
    ok = bs.Plan(A, B, bs.F64, host_only=1, merge_rows=1, axis_policy=bs.AXIS_CONTRACTION, c_layout_flags="rowpanel")
    assert len(ok.groups()) == 2
    assert ok.check_groups() == (0, -1)
    bad = bs.Plan(A, B, bs.F64, host_only=1, merge_rows=1, axis_policy=bs.AXIS_CONTRACTION, c_layout_flags="rowpanel",
                  debug_flags=bs.DEBUG_MERGE_UNCHECKED)
    assert len(bad.groups()) == 1
    assert bad.check_groups() == (bs.ERR_HOLE, 0)


def test_unchecked_merge_is_refused_for_a_device_plan():
    A, B = _two_row_problem()
    with pytest.raises(bs.BsError) as e:
        bs.Plan(A, B, bs.F64, merge_rows=1, debug_flags=bs.DEBUG_MERGE_UNCHECKED)
    assert e.value.code == 1


def test_group_validator_on_the_stress_workload():
    w = bsgen.config5()
    P, _, _ = host_plan(w)
    assert P.check_groups() == (0, -1)


def test_band_layouts_give_single_view_groups():
    """Row-panel A and column-panel B sorted by charge turn every contraction-axis
    group of the band and parity rules into one strided view (zero copy)."""
    for cfg in (1, 2, 3):
        P, _, _ = host_plan(bsgen.get(cfg), axis_policy=bs.AXIS_CONTRACTION)
        g = P.groups()
        assert np.all(g[:, 5] == 1)
    w5 = bsgen.config5()
    P5, _, _ = host_plan(w5, axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_NEVER)
    assert np.all(P5.groups()[:, 5] == 1)
    assert P5.stats()["triples"] > 4_000_000


def test_blockrow_layout_fragments_groups_and_pack_merges_them():
    w = bsgen.config2()
    P, _, _ = host_plan(w, "blockrow", "blockrow", axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_NEVER)
    assert np.any(P.groups()[:, 5] > 1)
    Pk, _, _ = host_plan(w, "blockrow", "blockrow", axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)
    assert np.all(Pk.groups()[:, 5] == 1)
    st = Pk.stats()
    assert st["packed_a"] == 1 and st["packed_b"] == 1 and st["packed_bytes"] > 0


def _gather_map(src_layout, dst_layout):
    """(source element, destination element) of every populated element: block (r, c)
    of the source layout goes to block (r, c) of the panel layout, row by row."""
    from harness import element_index
    sb, db = src_layout.blocks(), dst_layout.blocks()
    key = {(int(b[0]), int(b[1])): i for i, b in enumerate(db)}
    db = db[[key[(int(b[0]), int(b[1]))] for b in sb]]
    return element_index(sb), element_index(db)


@pytest.mark.parametrize("case", ["tail", "tiny0", "tiny2", "tiny3", "mixed"])
def test_gather_segments_move_every_element_once(case):
    """The segments of an FP64 gather: each spans at most 2048 source elements and
    holds at most 128 pieces, each piece lies inside its segment, each operand's
    segments come in source order, and the pieces together send every populated
    source element to its place in the panel exactly once."""
    if case == "tail":
        w, la, lb = bsgen.config2(), "blockrow", "blockrow"
    elif case == "mixed":
        w, la, lb = bsgen.config2(), "colpanel", "blockrow|charge_sorted"
    else:
        w = bsgen.tiny_random(700 + int(case[-1]), max_sectors=12, max_dim=300)
        la, lb = "blockrow", "blockrow|align16"
    P, A, B = host_plan(w, la, lb, axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)
    segs, pcs = P.gather_segments()
    assert len(segs) > 0 and len(segs) <= 2 * 152
    assert np.all(segs[:, 1] <= 2048) and np.all((segs[:, 3] >= 1) & (segs[:, 3] <= 128))
    assert segs[:, 3].sum() == len(pcs) and np.array_equal(segs[:, 2], np.concatenate([[0], np.cumsum(segs[:-1, 3])]))
    for op, (L, flags) in enumerate([(A, "rowpanel|charge_sorted"), (B, "colpanel|charge_sorted")]):
        so = segs[segs[:, 4] == op]
        assert np.all(np.diff(so[:, 0]) > 0)
        seg_src, seg_dst = [], []
        for first, n, p0, npc, _ in so:
            for dst, off, rows, cols, sld, dld in pcs[p0:p0 + npc]:
                assert 0 <= off and off + (rows - 1) * sld + cols <= n
                r, c = np.divmod(np.arange(rows * cols), cols)
                seg_src.append(first + off + r * sld + c)
                seg_dst.append(dst + r * dld + c)
        got_src, got_dst = np.concatenate(seg_src), np.concatenate(seg_dst)
        assert len(np.unique(got_src)) == len(got_src), "a source element is moved twice"
        if op == 0:
            pk = bs.Layout(w.rows, w.inner, w.rule_a, flags, 8)
        else:
            pk = bs.Layout(w.inner, w.cols, w.rule_b, flags, 8)
        want_src, want_dst = _gather_map(L, pk)
        o1, o2 = np.argsort(got_src), np.argsort(want_src)
        assert np.array_equal(got_src[o1], want_src[o2])
        assert np.array_equal(got_dst[o1], want_dst[o2])


def test_large_gathers_keep_no_segments():
    """The stress workload's block-row gather (about 98 segments per SM) goes block
    copy by block copy: the plan keeps no segment tables."""
    w = bsgen.config5()
    P, _, _ = host_plan(w, w.pack_layout_a, w.pack_layout_b, axis_policy=bs.AXIS_CONTRACTION,
                        pack_policy=bs.PACK_ALWAYS)
    segs, pcs = P.gather_segments()
    assert len(segs) == 0 and len(pcs) == 0 and P.stats()["packed_a"] == 1


def test_bf16_misaligned_views_are_packed_or_refused():
    w = bsgen.config4()
    P, _, _ = host_plan(w, "blockrow", "blockrow")
    assert P.stats()["packed_a"] == 1
    with pytest.raises(bs.BsError) as e:
        host_plan(w, "blockrow", "blockrow", pack_policy=bs.PACK_NEVER)
    assert e.value.code == 7
    P2, _, _ = host_plan(w)
    assert P2.stats()["packed_a"] == 0


def test_errors_are_status_codes():
    w = bsgen.config1()
    A = bs.Layout(w.rows, w.inner, w.rule_a, "blockrow", 8)
    other = bsgen.Axis(np.arange(-4, 5), np.ones(9))
    Bbad = bs.Layout(other, w.cols, w.rule_b, "blockrow", 8)
    with pytest.raises(bs.BsError) as e:
        bs.Plan(A, Bbad, bs.F64, host_only=1)
    assert e.value.code == 2
    with pytest.raises(bs.BsError) as e:
        bs.Plan(A, A, bs.BF16_F32, host_only=1)
    assert e.value.code == 1
    with pytest.raises(bs.BsError) as e:
        bs.Layout(w.rows, w.inner, bsgen.Rule(0, 0, True), "blockrow", 8)   # parity rule without parities
    assert e.value.code == 1
    with pytest.raises(bs.BsError) as e:
        bs.Layout(w.rows, w.inner, w.rule_a, 3, 8)
    assert e.value.code == 1
    with pytest.raises(bs.BsError) as e:
        bs.Layout(bsgen.Axis([0], [0]), w.inner, w.rule_a, 0, 8)
    assert e.value.code == 1
    w4 = bsgen.config4()
    A4 = bs.Layout(w4.rows, w4.inner, w4.rule_a, w4.layout_a, 2)
    B4 = bs.Layout(w4.inner, w4.cols, w4.rule_b, w4.layout_b, 2)
    with pytest.raises(bs.BsError) as e:
        bs.Plan(A4, B4, bs.BF16_F32, host_only=1, axis_policy=bs.AXIS_FREE)
    assert e.value.code == 3
    assert bs.lib.bs_status_string(2) == b"shape mismatch"
    P = bs.Plan(A, bs.Layout(w.inner, w.cols, w.rule_b, "blockrow", 8), bs.F64, host_only=1)
    with pytest.raises(bs.BsError):
        bs.contract(P, 0, 0, 0)


def test_axis_dimensions_beyond_32_bits_are_overflow():
    """A group's M, N and K are sums of one axis's dimensions, held in 32 bits:
    an axis adding up to more than INT32_MAX is refused at layout creation."""
    small = bsgen.Axis([100], [1])
    big = bsgen.Axis([0, 1], [2 ** 30, 2 ** 30])
    with pytest.raises(bs.BsError) as e:
        bs.Layout(big, small, bsgen.Rule(0, 0), "blockrow", 8)
    assert e.value.code == 9 and bs.lib.bs_status_string(9) == b"size overflow"
    with pytest.raises(bs.BsError) as e:
        bs.Layout(small, big, bsgen.Rule(0, 0), "colpanel", 8)
    assert e.value.code == 9
    # one less fits (the rule populates no block, so nothing is allocated)
    L = bs.Layout(bsgen.Axis([0, 1], [2 ** 30, 2 ** 30 - 1]), small, bsgen.Rule(0, 0), "blockrow", 8)
    assert L.nelems == 0


def test_empty_structure():
    """A rule that admits no block gives an empty plan and an empty C."""
    w = bsgen.config1()
    A = bs.Layout(w.rows, w.inner, bsgen.Rule(50, 60), "blockrow", 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, "blockrow", 8)
    P = bs.Plan(A, B, bs.F64, host_only=1)
    st = P.stats()
    assert st["triples"] == 0 and st["c_blocks"] == 0 and P.c_layout.nelems == 0


def test_chain_stage2_plans_on_stage1_c_layout():
    """A plan's C layout serves as the next plan's A layout (per-stage axis choice)."""
    w1, w2 = bsgen.chain2()
    A = bs.Layout(w1.rows, w1.inner, w1.rule_a, w1.layout_a, 8)
    B = bs.Layout(w1.inner, w1.cols, w1.rule_b, w1.layout_b, 8)
    P1 = bs.Plan(A, B, bs.F64, host_only=1, axis_policy=bs.AXIS_FREE, c_layout_flags=w1.layout_c)
    D = bs.Layout(w2.inner, w2.cols, w2.rule_b, w2.layout_b, 8)
    P2 = bs.Plan(P1.c_layout, D, bs.F64, host_only=1, axis_policy=bs.AXIS_CONTRACTION, c_layout_flags=w2.layout_c)
    s1, s2 = P1.stats(), P2.stats()
    assert s1["axis"] == bs.AXIS_FREE and s2["axis"] == bs.AXIS_CONTRACTION
    pr1 = oracle.problem(w1)
    assert s2["c_blocks"] == int(oracle.product_mask(pr1.mc, oracle.rule_mask(w2.inner, w2.cols, w2.rule_b)).sum())
    # T in charge-sorted row panels makes every stage-2 group one view
    assert np.all(P2.groups()[:, 5] == 1)


def test_bucket_padding_accounts_its_waste():
    """Power-of-two buckets: the same triples and groups, more executed flops (the
    padding), and nothing changes when bucket_pad is off."""
    w = bsgen.config2()
    for axis in (bs.AXIS_CONTRACTION, bs.AXIS_NONE):
        ex, _, _ = host_plan(w, axis_policy=axis)
        bk, _, _ = host_plan(w, axis_policy=axis, bucket_pad=1)
        se, sb = ex.stats(), bk.stats()
        assert sb["triples"] == se["triples"] and sb["groups"] == se["groups"]
        assert sb["useful_flops"] == se["useful_flops"]
        assert se["executed_flops"] < 1.001 * se["useful_flops"]
        # splitting long-K outputs over two lanes pads only the last 16-output chunk of a group
        split, _, _ = host_plan(w, axis_policy=axis, tail_split_k=64)
        assert se["executed_flops"] < split.stats()["executed_flops"] < 1.01 * se["useful_flops"]
        assert sb["executed_flops"] > 1.5 * sb["useful_flops"]
        assert sb["tail_tasks"] > se["tail_tasks"]
        assert bk.check_groups() == (0, -1)
    with pytest.raises(bs.BsError):
        host_plan(w, bucket_pad=2)


def test_plan_onto_a_given_c_layout():
    """bs_plan_create_into: a C layout equal to the structural product is taken as
    given; a subset or superset of it, or the wrong element size, is refused."""
    w = bsgen.config2()
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, 8)
    C = bs.Layout(w.rows, w.cols, bsgen.Rule(-2, 2), "colpanel|charge_sorted", 8)   # |dq| <= 1 twice
    P = bs.Plan(A, B, bs.F64, C=C, host_only=1)
    assert P.c_layout.nelems == C.nelems and np.array_equal(P.c_layout.blocks(), C.blocks())
    assert P.check_groups() == (0, -1)
    want, _, _ = oracle_triples(w)
    assert P.stats()["triples"] == len(want)
    for rule in (bsgen.Rule(-1, 1), bsgen.Rule(-3, 3)):
        with pytest.raises(bs.BsError) as e:
            bs.Plan(A, B, bs.F64, C=bs.Layout(w.rows, w.cols, rule, "blockrow", 8), host_only=1)
        assert e.value.code == 2
    with pytest.raises(bs.BsError) as e:
        bs.Plan(A, B, bs.F64, C=bs.Layout(w.rows, w.cols, bsgen.Rule(-2, 2), "blockrow", 4), host_only=1)
    assert e.value.code == 1
    other = bsgen.Axis(w.rows.q[:-1], w.rows.d[:-1])   # a row axis that is not A's
    with pytest.raises(bs.BsError) as e:
        bs.Plan(A, B, bs.F64, C=bs.Layout(other, w.cols, bsgen.Rule(-2, 2), "blockrow", 8), host_only=1)
    assert e.value.code == 2


@pytest.mark.parametrize("seed", range(40))
def test_random_structures_plan_exactly_and_hole_free(seed):
    """Random small structures (repeated charges, optional parity, random band
    rules): every policy covers the oracle's triples once, builds the oracle's C
    layout and passes the group validator."""
    w = bsgen.tiny_random(1000 + seed, max_sectors=10, max_dim=7)
    want, _, _ = oracle_triples(w)
    pr = oracle.problem(w)
    for pol in POLICIES + [dict(axis_policy=bs.AXIS_CONTRACTION, merge_rows=1)]:
        P, _, _ = host_plan(w, **pol)
        ptr, tr = P.triples()
        got = [tuple(int(x) for x in t) for t in tr]
        assert len(got) == len(set(got)) and set(got) == want
        assert P.check_groups() == (0, -1)
        assert P.c_layout.nelems == pr.lc.nelems
        assert np.array_equal(lib_blocks_by_rc(P.c_layout), pr.lc.blocks())


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("bucket", [0, 1])
def test_auto_plan_costs_candidates_like_forced_plans(cfg, bucket):
    """The AUTO planner costs every (axis, pack) candidate without listing its tail
    outputs; a plan forced onto one candidate lists it in full.  Both must give the
    same modelled time, and the AUTO plan's groups and triples must be the chosen
    candidate's."""
    w = bsgen.get(cfg)
    if w.dtype == "bf16":
        pytest.skip("the BF16 path has no axis or pack candidates to cost")
    if cfg == 5 and bucket:
        pytest.skip("one bucket setting is enough on the largest workload")
    auto, _, _ = host_plan(w, bucket_pad=bucket)
    sa = auto.stats()
    forced = {}
    for axis in (bs.AXIS_CONTRACTION, bs.AXIS_FREE):
        for pack in (bs.PACK_NEVER, bs.PACK_ALWAYS):
            P, _, _ = host_plan(w, axis_policy=axis, pack_policy=pack, bucket_pad=bucket)
            forced[(axis, pack)] = P
    chosen = (sa["axis"], bs.PACK_ALWAYS if (sa["packed_a"] or sa["packed_b"]) else bs.PACK_NEVER)
    fc = forced[chosen]
    sf = fc.stats()
    assert sf["model_us"] == pytest.approx(sa["model_us"], rel=1e-12)
    assert sf["executed_flops"] == pytest.approx(sa["executed_flops"], rel=1e-12)
    assert sf["tasks"] == sa["tasks"] and sf["groups"] == sa["groups"]
    others = [P.stats()["model_us"] for key, P in forced.items() if key != chosen]
    assert min(others) == pytest.approx(sa["model_us_alt"], rel=1e-12)
    assert all(sa["model_us"] <= o for o in others)
    pa, ta = auto.triples()
    pf, tf = fc.triples()
    assert np.array_equal(pa, pf) and np.array_equal(ta, tf)
    assert np.array_equal(auto.groups(), fc.groups())


def test_host_allocation_fault_injection_returns_oom(monkeypatch):
    """BS_FAULT_INJECT=alloc makes the host allocations of layout and plan
    construction fail: the calls return BS_ERR_OOM and leave nothing behind, and
    the same calls succeed again once the variable is gone."""
    w = bsgen.config1()
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, 8)
    monkeypatch.setenv("BS_FAULT_INJECT", "alloc")
    with pytest.raises(bs.BsError) as e:
        bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 8)
    assert e.value.code == 4
    for _ in range(3):
        with pytest.raises(bs.BsError) as e:
            bs.Plan(A, B, bs.F64, host_only=1)
        assert e.value.code == 4
    monkeypatch.delenv("BS_FAULT_INJECT")
    P = bs.Plan(A, B, bs.F64, host_only=1)
    assert P.stats()["triples"] == 71
