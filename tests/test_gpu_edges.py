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
