"""Repeated contractions with one plan, eager and replayed from a CUDA graph.

An FP64 plan's launches alternate between two device counter sets, each launch
preparing the other set for the next; a launch captured into a graph resets its
own set at exit instead, so every replay finds it as the capture did.  Both
must give the first eager result on every call: a counter set left in the
wrong state would skip or repeat work and change C."""
import numpy as np
import pytest

import bsgen
from harness import operand_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402


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
    # tail only: CTAs take their first task without a claim
    ("tail_panels", bsgen.config2, (None, None, None), dict(axis_policy=bs.AXIS_CONTRACTION)),
    ("tail_gathered", bsgen.config2, ("blockrow", "blockrow", "blockrow"),
     dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)),
    # tile tasks then tail, free axis (atomic accumulation into C)
    ("toy_free", bsgen.config1, ("colpanel", "blockrow", "blockrow"), dict(axis_policy=bs.AXIS_FREE)),
    ("large_tiles", bsgen.config3, (None, None, None), {}),
    ("bf16_localspace", bsgen.config4, (None, None, None), {}),
]


def _same(x, ref):
    if torch.equal(x, ref):
        return True
    scale = float(ref.abs().max()) if ref.numel() else 0.0
    return torch.allclose(x, ref, rtol=1e-12 if x.dtype == torch.float64 else 1e-6,
                          atol=(1e-12 if x.dtype == torch.float64 else 1e-6) * scale)


@pytest.mark.parametrize("name,make,lay,opts", CASES, ids=[c[0] for c in CASES])
def test_eager_calls_then_graph_replays_repeat_the_first_result(name, make, lay, opts):
    P, a, b, c = _setup(make(), *lay, **opts)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        bs.contract(P, a, b, c, stream=side)
    side.synchronize()
    assert bs.last_device_error(P) == 0
    ref = c.clone()
    # an odd and an even number of eager calls: both counter sets in use
    for _ in range(5):
        c.zero_()
        bs.contract(P, a, b, c, stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert bs.last_device_error(P) == 0
        assert _same(c, ref)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bs.contract(P, a, b, c, stream=torch.cuda.current_stream())
    for _ in range(4):
        c.zero_()
        g.replay()
        torch.cuda.synchronize()
        assert bs.last_device_error(P) == 0
        assert _same(c, ref)
    # eager again after the replays
    for _ in range(2):
        c.zero_()
        bs.contract(P, a, b, c, stream=torch.cuda.current_stream())
        torch.cuda.synchronize()
        assert bs.last_device_error(P) == 0
        assert _same(c, ref)


def test_bf16_capture_with_new_operand_pointers_is_refused_and_capture_survives():
    """A BF16 call with operand pointers its tensor maps were not encoded for must
    upload new maps and wait for them, which a capture cannot hold: the call
    returns UNSUPPORTED (3) before it enqueues anything, the capture ends
    cleanly, and the same call made eagerly afterwards gives the first result."""
    P, a, b, c = _setup(bsgen.config4())
    bs.contract(P, a, b, c, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert bs.last_device_error(P) == 0
    ref = c.clone()
    a2, b2 = a.clone(), b.clone()
    g = torch.cuda.CUDAGraph()
    with pytest.raises(bs.BsError) as err:
        with torch.cuda.graph(g):
            bs.contract(P, a2, b2, c, stream=torch.cuda.current_stream())
    assert err.value.code == 3
    c.zero_()
    bs.contract(P, a2, b2, c, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    assert bs.last_device_error(P) == 0
    assert torch.equal(c, ref)


def test_host_buffer_call_inside_a_capture_is_refused():
    """bs_contract_host synchronizes its stream, which a capture cannot hold: inside
    one it returns UNSUPPORTED (3) before it enqueues anything and the capture ends
    cleanly; outside, the same call gives the device call's result."""
    w = bsgen.config1()
    P, a, b, c = _setup(w)
    bs.contract(P, a, b, c, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    ref = c.cpu().numpy()
    ah, bh = a.cpu().numpy(), b.cpu().numpy()
    ch = np.zeros(c.numel(), ref.dtype)
    g = torch.cuda.CUDAGraph()
    with pytest.raises(bs.BsError) as err:
        with torch.cuda.graph(g):
            bs.contract_host(P, ah, bh, ch, stream=torch.cuda.current_stream())
    assert err.value.code == 3
    bs.contract_host(P, ah, bh, ch)
    assert _same(torch.from_numpy(ch), torch.from_numpy(ref))
