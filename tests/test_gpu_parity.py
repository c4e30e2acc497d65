"""Parity of the CUDA path (through the C ABI) with the CPU oracle, on a GB300.

Small workloads are compared on every output block; the full-size workloads
in the launch configuration the bench times are compared on sampled blocks
the oracle computes one by one.  FP64: max per-block relative Frobenius error
1e-12; BF16 inputs with FP32 accumulation: 5e-3 against the FP64 oracle on the
same BF16 inputs.  Integer-valued inputs make every partial sum exact, so
there the GPU must match bit for bit in any summation order, atomic scatter
included.  Block tables and offsets are compared exactly.
"""
import numpy as np
import pytest

import bsgen
import oracle
from harness import TOL, check_blocks, operand_host, sort_rc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402


class Run:
    """Library layouts, plan and device buffers for one workload."""

    def __init__(self, w, la=None, lb=None, lc=None, **opts):
        self.w = w
        eb = 2 if w.dtype == "bf16" else 8
        self.la, self.lb, self.lc = la or w.layout_a, lb or w.layout_b, lc or w.layout_c
        self.A = bs.Layout(w.rows, w.inner, w.rule_a, self.la, eb)
        self.B = bs.Layout(w.inner, w.cols, w.rule_b, self.lb, eb)
        dt = bs.BF16_F32 if w.dtype == "bf16" else bs.F64
        self.P = bs.Plan(self.A, self.B, dt, c_layout_flags=self.lc, **opts)
        self.a_host = operand_host(w, 0, self.A.blocks(), self.A.nelems)
        self.b_host = operand_host(w, 1, self.B.blocks(), self.B.nelems)
        tdt = torch.int16 if w.dtype == "bf16" else torch.float64
        self.a = torch.from_numpy(self.a_host.view(np.int16) if w.dtype == "bf16" else self.a_host).to("cuda")
        self.b = torch.from_numpy(self.b_host.view(np.int16) if w.dtype == "bf16" else self.b_host).to("cuda")
        self.cdt = torch.float32 if w.dtype == "bf16" else torch.float64
        self.c = torch.full((max(self.P.c_layout.nelems, 1),), float("nan"), dtype=self.cdt, device="cuda")
        del tdt

    def run(self, fn=None):
        (fn or bs.contract)(self.P, self.a, self.b, self.c)
        torch.cuda.synchronize()
        assert bs.last_device_error(self.P) == 0
        return self.c.cpu().numpy().astype(np.float64)


def oracle_for(run: Run):
    return oracle.problem(run.w, run.la, run.lb, run.lc)


def compare(run: Run, c_got: np.ndarray, sel=None, exact=False):
    pr = oracle_for(run)
    lib_c = sort_rc(run.P.c_layout.blocks())
    assert np.array_equal(lib_c, pr.lc.blocks()), "C block table differs from the oracle's"
    C, S = oracle.contract(pr, sel)
    blocks = lib_c
    if sel is not None:
        keep = {(int(i), int(j)) for i, j in np.asarray(sel).reshape(-1, 2)}
        blocks = np.array([b for b in lib_c if (int(b[0]), int(b[1])) in keep])
    tol = 0.0 if exact else TOL[run.w.dtype]
    ok, worst, ncancel = check_blocks(c_got, C, S, blocks, tol)
    print(f"[parity] {run.w.name}: {len(blocks)} blocks, worst {worst:.3e}, {ncancel} judged against ||S||")
    assert ok, f"worst per-block relative error {worst:.3e} > {tol} ({ncancel} cancelling blocks)"
    return worst


def sample_blocks(run: Run, budget_flops: float, seed: int = 0, n_random: int = 400):
    """Output blocks for the oracle: the costliest one, plus random ones within a flop budget."""
    ptr, tr = run.P.triples()
    w = run.w
    fl = {}
    for i, k, j in tr:
        fl[(int(i), int(j))] = fl.get((int(i), int(j)), 0) + 2 * int(w.rows.d[i]) * int(w.inner.d[k]) * int(w.cols.d[j])
    keys = list(fl)
    rng = np.random.default_rng(seed)
    pick = [max(keys, key=lambda x: fl[x])]
    used = fl[pick[0]]
    for t in rng.permutation(len(keys))[: n_random * 4]:
        kk = keys[t]
        if kk in pick or used + fl[kk] > budget_flops:
            continue
        pick.append(kk)
        used += fl[kk]
        if len(pick) > n_random:
            break
    return np.array(pick, np.int32)


# ---------------------------------------------------------------- small workloads, every block
POLICIES = {
    "auto": {},
    "contraction": dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_NEVER),
    "free": dict(axis_policy=bs.AXIS_FREE, pack_policy=bs.PACK_NEVER),
    "none": dict(axis_policy=bs.AXIS_NONE),
    "contraction_pack": dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS),
    "free_pack": dict(axis_policy=bs.AXIS_FREE, pack_policy=bs.PACK_ALWAYS),
}
LAYOUTS = {"panels": (None, None, None), "blockrow": ("blockrow", "blockrow", "blockrow"),
           "mixed": ("colpanel", "rowpanel|charge_sorted", "rowpanel")}


@pytest.mark.parametrize("cfg", [1, 2])
@pytest.mark.parametrize("pol", sorted(POLICIES))
@pytest.mark.parametrize("lay", sorted(LAYOUTS))
def test_fp64_small_configs_every_block(cfg, pol, lay):
    r = Run(bsgen.get(cfg), *LAYOUTS[lay], **POLICIES[pol])
    compare(r, r.run())


@pytest.mark.parametrize("seed", range(16))
@pytest.mark.parametrize("pol", ["contraction", "free", "none", "contraction_pack", "auto"])
def test_integer_inputs_bit_exact(seed, pol):
    w = bsgen.tiny_random(seed, values="int3", max_sectors=14, max_dim=40 if seed % 4 == 0 else 9)
    r = Run(w, *LAYOUTS[["panels", "blockrow", "mixed"][seed % 3]], **POLICIES[pol])
    compare(r, r.run(), exact=True)


@pytest.mark.parametrize("cfg", [1, 2])
@pytest.mark.parametrize("pol", ["contraction", "none", "free"])
def test_bucket_padding_matches_oracle(cfg, pol):
    """Tail groups padded to power-of-two shapes (batched buckets): the padded lanes
    and steps add only zeros, so every block still matches the oracle."""
    r = Run(bsgen.get(cfg), bucket_pad=1, **POLICIES[pol])
    assert r.P.stats()["executed_flops"] >= r.P.stats()["useful_flops"]
    compare(r, r.run())


@pytest.mark.parametrize("seed", range(8))
def test_bucket_padding_integer_inputs_bit_exact(seed):
    w = bsgen.tiny_random(100 + seed, values="int3", max_sectors=14, max_dim=9 if seed % 2 else 30)
    r = Run(w, *LAYOUTS[["panels", "blockrow", "mixed"][seed % 3]], bucket_pad=1,
            **POLICIES[["contraction", "none", "free", "auto"][seed % 4]])
    compare(r, r.run(), exact=True)


@pytest.mark.parametrize("seed", range(8))
def test_bf16_integer_inputs_bit_exact(seed):
    """|x| <= 3 integers are exact in bfloat16 and every FP32 partial sum stays exact."""
    w = bsgen.tiny_random(50 + seed, values="int3", dtype="bf16", max_sectors=10, max_dim=70 if seed % 2 else 20)
    r = Run(w, "rowpanel|align16", "colpanel|align16", "rowpanel|align16")
    compare(r, r.run(), exact=True)
    r2 = Run(w, "blockrow", "blockrow", "blockrow", pack_policy=bs.PACK_ALWAYS)   # gathered into aligned panels
    assert r2.P.stats()["packed_a"] == 1
    compare(r2, r2.run(), exact=True)


@pytest.mark.parametrize("mkn", [(1, 1, 1), (7, 5, 3), (128, 64, 16), (129, 257, 65), (300, 700, 40), (1024, 96, 1024)])
@pytest.mark.parametrize("dtype", ["f64", "bf16"])
def test_single_sector_is_a_dense_gemm(mkn, dtype):
    m, k, n = mkn
    w = bsgen.Workload("dense", dtype, bsgen.Axis([0], [m]), bsgen.Axis([0], [k]), bsgen.Axis([0], [n]),
                       bsgen.Rule(0, 0), bsgen.Rule(0, 0), "uniform", 1234 + m + k + n)
    lay = ("blockrow|align16",) * 3 if dtype == "bf16" else ("blockrow",) * 3
    r = Run(w, *lay)
    compare(r, r.run())


def _poison_check(r, c, granule_elems):
    """Populated elements are all written; padding keeps its NaN.  (granule_elems > 1
    would also admit zeros in the padding that completes a row's last granule of
    that many elements, for a store path that writes whole granules.)"""
    from harness import element_index
    blocks = r.P.c_layout.blocks()
    idx = np.zeros(r.P.c_layout.nelems, bool)
    idx[element_index(blocks)] = True
    assert not np.any(np.isnan(c[idx]))
    pad = ~idx
    assert pad.sum() > 0
    allowed = np.zeros_like(pad)
    if granule_elems > 1:
        for (_, _, off, nr, nc, ld) in blocks:
            ends = off + np.arange(nr) * ld + nc                   # first element after each row
            granule_end = ((ends - 1) // granule_elems + 1) * granule_elems
            for e in range(granule_elems - 1):
                pos = ends + e
                allowed[pos[pos < granule_end]] = True
    assert np.all(np.isnan(c[pad & ~allowed])), "padding outside the last granule of a row was written"
    assert np.all(np.isnan(c[pad & allowed]) | (c[pad & allowed] == 0.0))


def test_poisoned_c_bf16_padding_untouched():
    w = bsgen.config4()
    w.rows, w.inner, w.cols = (bsgen.Axis(a.q[:40], a.d[:40]) if a.n == 100 else bsgen.Axis(a.q[:10], a.d[:10])
                               for a in (w.rows, w.inner, w.cols))
    r = Run(w)
    c = r.run()
    _poison_check(r, c, granule_elems=1)
    compare(r, c)


def test_poisoned_c_fp64_padding_untouched():
    w = bsgen.config2()
    for pol in ("contraction", "free", "none"):
        r = Run(w, "rowpanel|charge_sorted", "colpanel|charge_sorted", "rowpanel|align16", **POLICIES[pol])
        c = r.run()
        _poison_check(r, c, granule_elems=1)
        compare(r, c)


def test_repeated_calls_are_identical():
    r = Run(bsgen.config2(), axis_policy=bs.AXIS_CONTRACTION)
    c1 = r.run()
    c2 = r.run()
    assert np.array_equal(c1, c2)          # one writer per C element: deterministic


def _populated(run):
    L = run.P.c_layout
    mask = np.zeros(L.nelems, bool)
    mask[L.element_index(L.blocks())] = True
    return mask


@pytest.mark.parametrize("pol", ["contraction", "free"])
def test_host_buffer_entry_point_matches_device_entry_point(pol):
    """Unpinned C: copied back whole (padding arrives as zeros).  Pinned C under a
    write-once plan: the kernel stores into it and leaves padding untouched.  A
    free-axis plan (zero fill, accumulation) always copies."""
    r = Run(bsgen.config2(), None, None, "blockrow|align16", **POLICIES[pol])   # C rows padded to 16 bytes
    c_dev = r.run()
    pop = _populated(r)
    assert (~pop).sum() > 0
    # free-axis groups accumulate with atomics, so two runs may round differently
    same = (np.array_equal if pol == "contraction" else
            lambda x, y: np.allclose(x, y, rtol=1e-12, atol=1e-12 * np.abs(y).max()))
    c_host = np.full(r.P.c_layout.nelems, np.nan)
    bs.contract_host(r.P, r.a_host, r.b_host, c_host)
    assert same(c_host[pop], c_dev[pop]) and np.all(c_host[~pop] == 0)
    a_pin = torch.from_numpy(r.a_host).pin_memory()
    b_pin = torch.from_numpy(r.b_host).pin_memory()
    c_pin = torch.full((r.P.c_layout.nelems,), float("nan"), dtype=torch.float64).pin_memory()
    for _ in range(2):
        bs.contract_host(r.P, a_pin, b_pin, c_pin)
        got = c_pin.numpy()
        assert same(got[pop], c_dev[pop])
        if pol == "contraction":
            assert r.P.stats()["launches"] == 1 and np.all(np.isnan(got[~pop]))
        else:
            assert np.all(got[~pop] == 0)


def test_host_entry_point_large_pinned_c_is_copied_back():
    """A pinned C larger than 4 MiB that its kernel writes fast (workload 4: 55 MB
    of FP32 in a few tens of microseconds) is not stored into directly: it
    arrives by one copy of the whole buffer, padding as zeros."""
    r = Run(bsgen.config4())
    c_dev = r.run()
    pop = _populated(r)
    assert (~pop).sum() > 0 and r.P.c_layout.nelems * 4 > (4 << 20)
    a_pin = torch.from_numpy(r.a_host.view(np.int16)).pin_memory()
    b_pin = torch.from_numpy(r.b_host.view(np.int16)).pin_memory()
    c_pin = torch.full((r.P.c_layout.nelems,), float("nan"), dtype=torch.float32).pin_memory()
    bs.contract_host(r.P, a_pin, b_pin, c_pin)
    got = c_pin.numpy()
    assert np.array_equal(got[pop], c_dev[pop]) and np.all(got[~pop] == 0)


def test_host_entry_point_large_pinned_c_under_a_long_fp64_kernel_is_stored_directly():
    """A pinned C far beyond 4 MiB whose FP64 kernel spreads its stores over
    milliseconds (workload 3 on the contraction axis) is stored into directly:
    every populated element matches the device entry point and the padding of
    C_host keeps what it held."""
    r = Run(bsgen.config3(), None, None, "blockrow|align16", **POLICIES["contraction"])
    c_dev = r.run()
    pop = _populated(r)
    st = r.P.stats()
    nc = r.P.c_layout.nelems * 8
    assert (~pop).sum() > 0 and nc > (4 << 20) and nc <= 50e3 * st["model_us"]
    a_pin = torch.from_numpy(r.a_host).pin_memory()
    b_pin = torch.from_numpy(r.b_host).pin_memory()
    c_pin = torch.full((r.P.c_layout.nelems,), float("nan"), dtype=torch.float64).pin_memory()
    for _ in range(2):
        bs.contract_host(r.P, a_pin, b_pin, c_pin)
        got = c_pin.numpy()
        assert np.array_equal(got[pop], c_dev[pop]) and np.all(np.isnan(got[~pop]))


@pytest.mark.parametrize("seed", [71, 75, 78, 81])
def test_host_entry_point_staging_kernel_ragged_and_offset_inputs(seed):
    """Pinned, 16-byte aligned A and B are pulled in by the staging kernel, whose
    ragged last 8 bytes (operands with an odd element count) must arrive too; a
    pinned operand that starts 8 bytes into its allocation takes the copy-engine
    path.  Both give the device entry point's C bit for bit."""
    w = bsgen.tiny_random(seed, values="int3", max_sectors=9, max_dim=23)
    r = Run(w, "blockrow", "blockrow", "blockrow", **POLICIES["contraction"])
    assert (r.A.nelems % 2) or (r.B.nelems % 2)
    c_dev = r.run()
    pop = _populated(r)
    a_pin, b_pin = torch.from_numpy(r.a_host).pin_memory(), torch.from_numpy(r.b_host).pin_memory()
    c_pin = torch.full((r.P.c_layout.nelems,), float("nan"), dtype=torch.float64).pin_memory()
    bs.contract_host(r.P, a_pin, b_pin, c_pin)
    assert np.array_equal(c_pin.numpy()[pop], c_dev[pop])
    a_off = torch.zeros(r.A.nelems + 1, dtype=torch.float64).pin_memory()
    a_off[1:] = torch.from_numpy(r.a_host)
    c_pin.fill_(float("nan"))
    bs.contract_host(r.P, a_off[1:], b_pin, c_pin)
    assert np.array_equal(c_pin.numpy()[pop], c_dev[pop])
    compare(r, c_pin.numpy().astype(np.float64), exact=True)


def test_plan_onto_a_given_c_layout_matches_oracle():
    w = bsgen.config2()
    lc = "colpanel|charge_sorted"
    r = Run(w, None, None, lc)
    c1 = r.run()
    compare(r, c1)
    C = bs.Layout(w.rows, w.cols, bsgen.Rule(-2, 2), lc, 8)
    P2 = bs.Plan(r.A, r.B, bs.F64, C=C)
    assert np.array_equal(P2.c_layout.blocks(), r.P.c_layout.blocks())
    c2 = torch.full_like(r.c, float("nan"))
    bs.contract(P2, r.a, r.b, c2)
    torch.cuda.synchronize()
    assert bs.last_device_error(P2) == 0
    assert np.array_equal(c2.cpu().numpy(), c1, equal_nan=True)


def test_uncoalesced_control_matches_oracle():
    r = Run(bsgen.config2())
    c = r.run(bs.contract_uncoalesced)
    compare(r, c)


def test_bf16_wait_timeout_is_reported_and_context_survives():
    """A producer that withholds one copy makes the consumer's bounded wait run out;
    the kernel reports BS_ERR_TIMEOUT and the context stays usable."""
    w = bsgen.config4()
    r = Run(w, wait_timeout_ms=50, debug_flags=1)
    bs.contract(r.P, r.a, r.b, r.c)
    assert bs.last_device_error(r.P) == 6
    r2 = Run(w)
    compare(r2, r2.run(), sel=sample_blocks(r2, 2e8, n_random=60))


# ---------------------------------------------------------------- integer inputs on the large-block paths
def _int_workload(seed, dtype, rows_d, inner_d, cols_d, name):
    """Three short band axes with large sectors: charges 0, 1, 2, ... (repeats allowed),
    |dq| <= 1 for both operands, integer values in -3..3 (exact in any order)."""
    rng = np.random.default_rng(seed)

    def axis(ds):
        q = np.sort(rng.integers(0, 3, len(ds)))
        return bsgen.Axis(q, np.array(ds))

    return bsgen.Workload(name, dtype, axis(rows_d), axis(inner_d), axis(cols_d), bsgen.Rule(-1, 1),
                          bsgen.Rule(-1, 1), "int3", 0x1A7E0000 + seed)


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("pol", ["contraction", "free", "contraction_pack", "auto"])
@pytest.mark.parametrize("lay", ["panels", "blockrow"])
def test_fp64_tile_path_integer_inputs_bit_exact(seed, pol, lay):
    """C blocks of more than 4096 outputs take the shared-memory tile path; their
    K runs over several inner blocks (several views with block-row layouts) and
    more than 16 chunks of 16.  Integer inputs: bit-exact in any summation order."""
    rng = np.random.default_rng(100 + seed)
    w = _int_workload(seed, "f64", rng.integers(60, 130, 4), rng.integers(60, 130, 5), rng.integers(65, 130, 3),
                      f"int_tiles_{seed}")
    r = Run(w, *LAYOUTS[lay], **POLICIES[pol])
    st = r.P.stats()
    assert st["tile_tasks"] > 0, "the case must reach the tile path"
    assert max(g[3] for g in r.P.groups()) > 16 * 16 or st["axis"] == bs.AXIS_FREE
    compare(r, r.run(), exact=True)


@pytest.mark.parametrize("seed", range(3))
@pytest.mark.parametrize("lay", [("blockrow", "blockrow"), ("blockrow|charge_sorted", "rowpanel"),
                                 ("colpanel", "blockrow|charge_sorted")])
def test_fp64_gather_every_alignment_integer_inputs_bit_exact(seed, lay):
    """The gather into panels on dimensions of both parities, from 1 to 300: blocks
    whose rows are 1 to 300 doubles, source and destination rows starting on or 8
    bytes off a 16-byte boundary, flat runs of both lengths' parities, runs under
    and over 64 elements and of more than 2048 (banded), and copies of at most 64
    elements.  Every path of the gather is taken; integer inputs, so C must match
    the oracle bit for bit."""
    rng = np.random.default_rng(300 + seed)
    dims = lambda n: [int(x) for x in rng.choice([1, 2, 3, 5, 8, 63, 64, 65, 130, 131, 257, 300], n)]
    w = _int_workload(seed, "f64", dims(6), dims(7), dims(5), f"int_gather_{seed}")
    r = Run(w, lay[0], lay[1], "rowpanel", axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)
    st = r.P.stats()
    assert st["packed_a"] == 1 and st["packed_b"] == 1
    compare(r, r.run(), exact=True)


@pytest.mark.parametrize("seed", range(4))
def test_bf16_multi_tile_integer_inputs_bit_exact(seed):
    """Groups of several 128-row M tiles, tile widths of 192 to 256 columns plus a
    ragged second column tile, and K of more than four 64-deep stages over several
    inner blocks.  Integers in -3..3 are exact in bfloat16 and every FP32 partial
    sum stays exact, so the result must match bit for bit."""
    rng = np.random.default_rng(200 + seed)
    cols = [int(rng.integers(192, 257)), int(rng.integers(257, 330)), int(rng.integers(20, 100))]
    w = _int_workload(seed, "bf16", rng.integers(130, 400, 3), rng.integers(70, 200, 4), cols, f"int_bf16_{seed}")
    r = Run(w, "rowpanel|charge_sorted|align16", "colpanel|charge_sorted|align16", "rowpanel|align16")
    st = r.P.stats()
    g = r.P.groups()
    assert st["tasks"] > st["groups"], "some group must span several tiles"
    assert g[:, 1].max() > 128 and g[:, 2].max() > 256 and g[:, 3].max() > 256
    compare(r, r.run(), exact=True)
    r2 = Run(w, "blockrow", "blockrow", "blockrow", pack_policy=bs.PACK_ALWAYS)   # gathered into aligned panels
    compare(r2, r2.run(), exact=True)


# ---------------------------------------------------------------- full-size workloads, every block
def compare_all(run: Run, c_got: np.ndarray):
    """Every C block of a full-size workload against the oracle, run over every host core."""
    from harness import oracle_all_blocks
    C, S, pr = oracle_all_blocks(run.w, run.la, run.lb, run.lc)
    lib_c = sort_rc(run.P.c_layout.blocks())
    assert np.array_equal(lib_c, pr.lc.blocks()), "C block table differs from the oracle's"
    tol = TOL[run.w.dtype]
    ok, worst, ncancel = check_blocks(c_got, C, S, lib_c, tol)
    print(f"[parity] {run.w.name}: all {len(lib_c)} blocks, worst {worst:.3e}, {ncancel} judged against ||S||")
    assert ok, f"worst per-block relative error {worst:.3e} > {tol} ({ncancel} cancelling blocks)"


@pytest.mark.parametrize("cfg", [3, 4, 5])
def test_full_size_every_block(cfg):
    w = bsgen.get(cfg)
    r = Run(w)
    c = r.run()
    from harness import element_index
    assert not np.any(np.isnan(c[element_index(r.P.c_layout.blocks())]))   # every populated element written
    compare_all(r, c)


@pytest.mark.parametrize("n", [16, 64, 100, 128, 200, 256, 320, 384, 515])
@pytest.mark.parametrize("align", ["align16", "align64"])
def test_bf16_column_widths_integer_inputs_bit_exact(n, align):
    """Column sectors of width n: whole 64-column chunks of a tile come in one 3-D box
    (2 to 4 of them), a ragged last chunk in its own 2-D box; tiles past the first
    256 columns take fewer whole chunks."""
    rng = np.random.default_rng(400 + n)
    w = _int_workload(n, "bf16", rng.integers(100, 300, 2), rng.integers(40, 140, 3), [n, n, n // 2 + 8],
                      f"int_bf16_n{n}_{align}")
    r = Run(w, f"rowpanel|charge_sorted|{align}", f"colpanel|charge_sorted|{align}", f"rowpanel|{align}")
    compare(r, r.run(), exact=True)


def test_config4_align64_layouts_every_block():
    """The BF16 workload with every operand and C row on a 64-byte boundary."""
    w = bsgen.config4()
    r = Run(w, "rowpanel|charge_sorted|align64", "colpanel|charge_sorted|align64", "rowpanel|charge_sorted|align64")
    assert r.P.stats()["packed_a"] == 0
    compare_all(r, r.run())


@pytest.mark.parametrize("seed", range(4))
def test_align64_layouts_integer_inputs_bit_exact(seed):
    """64-byte layouts on the FP64 paths (tail, tiles, gather) and the BF16 path."""
    rng = np.random.default_rng(300 + seed)
    w = _int_workload(seed, "bf16", rng.integers(130, 300, 3), rng.integers(20, 150, 4), rng.integers(30, 280, 3),
                      f"int_bf16_a64_{seed}")
    r = Run(w, "rowpanel|charge_sorted|align64", "colpanel|charge_sorted|align64", "rowpanel|align64")
    compare(r, r.run(), exact=True)
    wf = _int_workload(seed, "f64", rng.integers(1, 90, 4), rng.integers(1, 90, 4), rng.integers(1, 90, 4),
                       f"int_f64_a64_{seed}")
    for pol in ["contraction", "free", "contraction_pack"]:
        rf = Run(wf, "blockrow|align64", "rowpanel|align64", "colpanel|align64", **POLICIES[pol])
        compare(rf, rf.run(), exact=True)


def test_config5_pack_path_every_block():
    w = bsgen.config5()
    r = Run(w, "blockrow", "blockrow", "blockrow", axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)
    compare_all(r, r.run())


def test_config4_blockrow_gather_path_every_block():
    w = bsgen.config4()
    r = Run(w, w.pack_layout_a, w.pack_layout_b, w.pack_layout_c)
    assert r.P.stats()["packed_a"] == 1
    compare_all(r, r.run())


# ---------------------------------------------------------------- long-K tail outputs on two lanes
@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("split_k", [2, 9, 0])
def test_split_tail_outputs_integer_inputs_bit_exact(seed, split_k):
    """Tail groups of one view whose K reaches tail_split_k run each output on two
    lanes (each sums half of K, one shuffle adds them); integer inputs make the
    result exact, split or not, padded buckets included."""
    w = bsgen.tiny_random(300 + seed, values="int3", max_sectors=12, max_dim=17)
    r = Run(w, *LAYOUTS[["panels", "mixed"][seed % 2]], axis_policy=bs.AXIS_CONTRACTION,
            tail_split_k=split_k, bucket_pad=seed % 3 == 2)
    compare(r, r.run(), exact=True)


@pytest.mark.parametrize("split_k", [8, 64])
def test_split_tail_outputs_tail_workload_every_block(split_k):
    r = Run(bsgen.config2(), tail_split_k=split_k)
    compare(r, r.run())
