"""Degenerate structures on the GPU: an operand with no block at all, and two
non-empty operands whose structural product is empty.  A contraction over an
empty product writes nothing and reports success; the C layout has no block."""
import numpy as np
import pytest

import bsgen

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # collected on CPU-only machines, skipped there
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402

FLAGS = {"f64": ("rowpanel|charge_sorted", "colpanel|charge_sorted", 8, bs.F64, torch.float64),
         "bf16": ("rowpanel|charge_sorted|align16", "colpanel|charge_sorted|align16", 2, bs.BF16_F32, torch.float32)}


def _axis(qs, d):
    return bsgen.Axis(np.array(qs), np.full(len(qs), d))


def _contract_empty(rows, inner, cols, rule_a, rule_b, dtype):
    la, lb, eb, dt, cdt = FLAGS[dtype]
    A = bs.Layout(rows, inner, rule_a, la, eb)
    B = bs.Layout(inner, cols, rule_b, lb, eb)
    P = bs.Plan(A, B, dt)
    assert P.c_layout.nelems == 0 and len(P.c_layout.blocks()) == 0
    assert P.stats()["triples"] == 0
    ebt = torch.int16 if dtype == "bf16" else torch.float64
    a = torch.zeros(max(A.nelems, 8), dtype=ebt, device="cuda")
    b = torch.zeros(max(B.nelems, 8), dtype=ebt, device="cuda")
    c = torch.full((8,), 7.0, dtype=cdt, device="cuda")
    bs.contract(P, a, b, c)
    torch.cuda.synchronize()
    assert bs.last_device_error(P) == 0
    assert torch.all(c == 7.0)   # nothing written
    return A, B


@pytest.mark.parametrize("dtype", ["f64", "bf16"])
def test_operand_without_blocks(dtype):
    # A's rule asks for q_row - q_inner = 10, which no pair of these charges meets
    A, _ = _contract_empty(_axis([0, 1, 2], 8), _axis([0, 1, 2], 8), _axis([0, 1], 8),
                           bsgen.Rule(10, 10), bsgen.Rule(-1, 1), dtype)
    assert A.nelems == 0


@pytest.mark.parametrize("dtype", ["f64", "bf16"])
def test_non_empty_operands_with_empty_product(dtype):
    # A pairs row 3 only with inner charge 0; B uses only inner charges 2 and 3
    A, B = _contract_empty(_axis([0, 1, 2, 3], 8), _axis([0, 1, 2, 3], 8), _axis([0], 8),
                           bsgen.Rule(3, 3), bsgen.Rule(2, 3), dtype)
    assert A.nelems > 0 and B.nelems > 0


@pytest.mark.parametrize("case", ["gather", "zero_fill", "plain"])
def test_phase_profile_reports_each_phase(case):
    """A plan built with profile=1 reports the gather, zero fill and kernel
    times of its last contraction (0 for a phase it does not have), their sum,
    and the gather's bytes; a plan without profiling refuses."""
    w = bsgen.config2()
    lay = {"gather": ("blockrow", "blockrow", "blockrow"), "zero_fill": (None, None, None),
           "plain": (None, None, None)}[case]
    opts = {"gather": dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS),
            "zero_fill": dict(axis_policy=bs.AXIS_FREE), "plain": dict(axis_policy=bs.AXIS_CONTRACTION)}[case]
    A = bs.Layout(w.rows, w.inner, w.rule_a, lay[0] or w.layout_a, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, lay[1] or w.layout_b, 8)
    P = bs.Plan(A, B, bs.F64, c_layout_flags=lay[2] or w.layout_c, profile=1, **opts)
    a = torch.randn(A.nelems, dtype=torch.float64, device="cuda")
    b = torch.randn(B.nelems, dtype=torch.float64, device="cuda")
    c = torch.zeros(P.c_layout.nelems, dtype=torch.float64, device="cuda")
    with pytest.raises(bs.BsError):
        P.profile()   # not run yet
    bs.contract(P, a, b, c)
    t = P.profile()
    st = P.stats()
    assert t["kernel_ms"] > 0
    assert (t["gather_ms"] > 0) == (case == "gather") and (t["zero_ms"] > 0) == (case == "zero_fill")
    assert t["gather_bytes"] == (2 * st["packed_bytes"] if case == "gather" else 0)
    assert abs(t["total_ms"] - (t["gather_ms"] + t["zero_ms"] + t["kernel_ms"])) < 1e-6
    Q = bs.Plan(A, B, bs.F64, c_layout_flags=lay[2] or w.layout_c, **opts)
    bs.contract(Q, a, b, c)
    with pytest.raises(bs.BsError):
        Q.profile()   # built without profiling
