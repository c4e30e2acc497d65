"""The bounds-checked contraction (bs_contract_checked) on the GPU.

With the buffers' true sizes it must give bs_contract's result bit for bit and
report nothing.  With a declared size smaller than the buffer, the accesses past
it are still inside the real allocation, so nothing can fault; the checked FP64
kernel must skip them and report a bounds violation (BS_ERR_DEVICE), and the
host must refuse gathers, zero fills and BF16 views that do not fit before
anything runs."""
import numpy as np
import pytest

import bsgen
from harness import operand_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402

DEVICE = 8   # BS_ERR_DEVICE


def _setup(w, la=None, lb=None, lc=None, **opts):
    eb = 2 if w.dtype == "bf16" else 8
    A = bs.Layout(w.rows, w.inner, w.rule_a, la or w.layout_a, eb)
    B = bs.Layout(w.inner, w.cols, w.rule_b, lb or w.layout_b, eb)
    dt = bs.BF16_F32 if w.dtype == "bf16" else bs.F64
    P = bs.Plan(A, B, dt, c_layout_flags=lc or w.layout_c, **opts)
    ah, bh = operand_host(w, 0, A.blocks(), A.nelems), operand_host(w, 1, B.blocks(), B.nelems)
    a = torch.from_numpy(ah.view(np.int16) if eb == 2 else ah).cuda()
    b = torch.from_numpy(bh.view(np.int16) if eb == 2 else bh).cuda()
    c = torch.zeros(max(P.c_layout.nelems, 1), dtype=torch.float32 if eb == 2 else torch.float64, device="cuda")
    return P, a, b, c


CASES = [
    ("tail_panels", bsgen.config2, (None, None, None), {}),
    ("toy_free", bsgen.config1, ("colpanel", "blockrow", "blockrow"), dict(axis_policy=bs.AXIS_FREE)),
    ("tail_blockrow_views", bsgen.config2, ("blockrow", "blockrow", "blockrow"),
     dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_NEVER)),
    ("tail_blockrow_gathered", bsgen.config2, ("blockrow", "blockrow", "blockrow"),
     dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)),
    ("large_tiles", bsgen.config3, (None, None, None), {}),
]


@pytest.mark.parametrize("name,make,lay,opts", CASES, ids=[c[0] for c in CASES])
def test_checked_contraction_with_true_sizes_matches_and_reports_nothing(name, make, lay, opts):
    P, a, b, c = _setup(make(), *lay, **opts)
    bs.contract(P, a, b, c)
    torch.cuda.synchronize()
    ref = c.clone()
    c.zero_()
    bs.contract_checked(P, a, b, c)
    assert bs.last_device_error(P) == 0
    if P.stats()["axis"] == bs.AXIS_CONTRACTION:
        assert torch.equal(c, ref)    # one writer per C element: the same sums in the same order
    else:                             # atomic scatter: the order of the adds may differ
        assert torch.allclose(c, ref, rtol=1e-12, atol=1e-12 * float(ref.abs().max()))


@pytest.mark.parametrize("which", ["A", "B", "C"])
def test_checked_contraction_reports_a_short_buffer(which):
    P, a, b, c = _setup(bsgen.config2())
    sizes = dict(nA=a.numel(), nB=b.numel(), nC=c.numel())
    sizes["n" + which] //= 2          # declared shorter than it is: the skipped accesses were in bounds
    bs.contract_checked(P, a, b, c, **sizes)
    assert bs.last_device_error(P) == DEVICE
    bs.contract(P, a, b, c)           # the plan is reusable afterwards
    assert bs.last_device_error(P) == 0


def test_checked_contraction_refuses_on_the_host():
    # a gathered plan: the gather's reads are checked before anything runs
    P, a, b, c = _setup(bsgen.config2(), "blockrow", "blockrow", "blockrow", axis_policy=bs.AXIS_CONTRACTION,
                        pack_policy=bs.PACK_ALWAYS)
    with pytest.raises(bs.BsError) as e:
        bs.contract_checked(P, a, b, c, nA=a.numel() // 2)
    assert e.value.code == DEVICE
    # a free-axis plan: the zero fill's C blocks
    P, a, b, c = _setup(bsgen.config2(), axis_policy=bs.AXIS_FREE)
    with pytest.raises(bs.BsError) as e:
        bs.contract_checked(P, a, b, c, nC=c.numel() // 2)
    assert e.value.code == DEVICE
    # a BF16 plan: its tensor-map views and output tiles
    w = bsgen.config4()
    P, a, b, c = _setup(w)
    for key in ("nA", "nB", "nC"):
        sizes = dict(nA=a.numel(), nB=b.numel(), nC=c.numel())
        sizes[key] //= 2
        with pytest.raises(bs.BsError) as e:
            bs.contract_checked(P, a, b, c, **sizes)
        assert e.value.code == DEVICE
    bs.contract_checked(P, a, b, c)
    assert bs.last_device_error(P) == 0
