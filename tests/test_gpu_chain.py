"""A two-stage chained contraction on the GPU: T = A B with free-axis groups, then
Y = T D with contraction-axis groups, T kept on the device in a layout chosen for
the second stage.  Compared with the oracle's two-stage product, FP64 1e-12."""
import numpy as np
import pytest

import bsgen
import oracle
from harness import TOL, check_blocks, operand_host, sort_rc

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402


@pytest.mark.parametrize("axes", [(bs.AXIS_FREE, bs.AXIS_CONTRACTION), (bs.AXIS_CONTRACTION, bs.AXIS_CONTRACTION),
                                  (bs.AXIS_AUTO, bs.AXIS_FREE)])
def test_two_stage_chain_matches_oracle(axes):
    w1, w2 = bsgen.chain2()
    A = bs.Layout(w1.rows, w1.inner, w1.rule_a, w1.layout_a, 8)
    B = bs.Layout(w1.inner, w1.cols, w1.rule_b, w1.layout_b, 8)
    P1 = bs.Plan(A, B, bs.F64, axis_policy=axes[0], c_layout_flags=w1.layout_c)
    D = bs.Layout(w2.inner, w2.cols, w2.rule_b, w2.layout_b, 8)
    P2 = bs.Plan(P1.c_layout, D, bs.F64, axis_policy=axes[1], c_layout_flags=w2.layout_c)
    a = torch.from_numpy(operand_host(w1, 0, A.blocks(), A.nelems)).cuda()
    b = torch.from_numpy(operand_host(w1, 1, B.blocks(), B.nelems)).cuda()
    d = torch.from_numpy(operand_host(w2, 1, D.blocks(), D.nelems)).cuda()
    t = torch.full((P1.c_layout.nelems,), float("nan"), dtype=torch.float64, device="cuda")
    y = torch.full((P2.c_layout.nelems,), float("nan"), dtype=torch.float64, device="cuda")
    bs.contract(P1, a, b, t)
    bs.contract(P2, t, d, y)           # T never leaves the device
    torch.cuda.synchronize()
    assert bs.last_device_error(P1) == 0 and bs.last_device_error(P2) == 0
    pr1 = oracle.problem(w1)
    T, _ = oracle.contract(pr1)
    pr2 = oracle.chain_stage2(pr1, T, w2)
    Y, S = oracle.contract(pr2)
    lib_c = sort_rc(P2.c_layout.blocks())
    assert np.array_equal(lib_c, pr2.lc.blocks())
    ok, worst, _ = check_blocks(y.cpu().numpy(), Y, S, lib_c, TOL["f64"])
    assert ok, f"worst per-block relative error {worst:.3e}"
