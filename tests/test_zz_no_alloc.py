"""The allocation-free entry point, checked against bs_contract on the GPU.

bs_contract_noalloc serves callers that cannot allocate device memory (a
memory manager owns all of it, or a steady-state loop may not allocate after
start-up): the plan is built on the host only and every call works out of the
library's fixed device array.  Its results must equal those of bs_contract
within the FP64 parity tolerance, on two calls in a row (the array keeps the
previous call's contents, so the second call checks that the counters and
tables are reset).  This file is collected last on purpose.
"""
import numpy as np
import pytest

import bsgen
from harness import TOL, element_index, operand_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402


def _plans(w, la, lb, lc, **opts):
    A = bs.Layout(w.rows, w.inner, w.rule_a, la, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, lb, 8)
    host = bs.Plan(A, B, bs.F64, c_layout_flags=lc, host_only=1, **opts)
    dev = bs.Plan(A, B, bs.F64, c_layout_flags=lc, **opts)
    a = torch.from_numpy(operand_host(w, 0, A.blocks(), A.nelems)).cuda()
    b = torch.from_numpy(operand_host(w, 1, B.blocks(), B.nelems)).cuda()
    return host, dev, a, b


CASES = [
    ("config2_panels", bsgen.config2, (None, None, None), {}),
    ("config2_gathered", bsgen.config2, ("blockrow", "blockrow", "blockrow"),
     dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)),
    ("config1_free_axis", bsgen.config1, ("colpanel", "blockrow", "blockrow"), dict(axis_policy=bs.AXIS_FREE)),
]


@pytest.mark.parametrize("name,make,lay,opts", CASES, ids=[c[0] for c in CASES])
def test_noalloc_matches_contract_on_two_calls(name, make, lay, opts):
    w = make()
    la, lb, lc = (lay[0] or w.layout_a, lay[1] or w.layout_b, lay[2] or w.layout_c)
    host, dev, a, b = _plans(w, la, lb, lc, **opts)
    n = max(dev.c_layout.nelems, 1)
    c_ref = torch.zeros(n, dtype=torch.float64, device="cuda")
    bs.contract(dev, a, b, c_ref)
    torch.cuda.synchronize()
    ref = c_ref.cpu().numpy()
    blocks = host.c_layout.blocks()
    assert np.array_equal(blocks, dev.c_layout.blocks())
    idx = element_index(blocks)
    sizes = blocks[:, 3] * blocks[:, 4]
    starts = np.concatenate([[0], np.cumsum(sizes)[:-1]]).astype(np.int64)
    for call in range(2):
        c = torch.full((n,), float("nan"), dtype=torch.float64, device="cuda")
        bs.contract_noalloc(host, a, b, c)
        torch.cuda.synchronize()
        got = c.cpu().numpy()
        d2 = np.add.reduceat((got[idx] - ref[idx]) ** 2, starts)
        r2 = np.add.reduceat(ref[idx] ** 2, starts)
        rel = np.sqrt(d2) / np.maximum(np.sqrt(r2), 1e-300)
        assert not np.any(np.isnan(got[idx])), f"call {call}: unwritten outputs"
        assert rel.max() <= TOL["f64"], f"call {call}: worst per-block relative error {rel.max():.3e}"


def _small_device_buffers(dtype):
    """Real device buffers for the refusal tests: the call must refuse before it
    touches them, but if a check ever regressed it would only read and write
    these few valid bytes."""
    return tuple(torch.zeros(64, dtype=dtype, device="cuda") for _ in range(3))


def test_noalloc_rejects_a_plan_larger_than_its_array():
    w = bsgen.config5()
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, 8)
    host = bs.Plan(A, B, bs.F64, c_layout_flags=w.layout_c, host_only=1)
    a, b, c = _small_device_buffers(torch.float64)
    with pytest.raises(bs.BsError) as e:
        bs.contract_noalloc(host, a, b, c)     # refused before anything is enqueued
    assert e.value.code == 9
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0


def test_noalloc_refuses_bf16_plans():
    w = bsgen.config4()
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 2)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, 2)
    host = bs.Plan(A, B, bs.BF16_F32, c_layout_flags=w.layout_c, host_only=1)
    a, b, c = _small_device_buffers(torch.float32)
    with pytest.raises(bs.BsError) as e:
        bs.contract_noalloc(host, a, b, c)
    assert e.value.code == 3
    torch.cuda.synchronize()
    assert torch.count_nonzero(c).item() == 0
