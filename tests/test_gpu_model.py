"""The planner's cost model against the device it runs on.

bs_calibrate measures the model's constants with the library's own kernels;
with them the AUTO plan must pick, among its (axis, gather) candidates, one
whose measured time is within 10% of the fastest candidate's, on the toy
workload, the tail workload and a fragmented (block-row) layout of it."""
import statistics

import numpy as np
import pytest

import bsgen
from harness import operand_host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import block_sparse_tensor_gb300 as bs  # noqa: E402


@pytest.fixture(scope="module")
def calibrated():
    cal = bs.calibrate()
    print("[model] calibration", {k: round(v, 3) if isinstance(v, float) else v for k, v in cal.items()})
    for key in ("t_fixed_us", "tile_gflops", "tail_gflops", "general_gflops", "pack_gbs", "zero_gbs",
                "bf16_stage_us", "bf16_tile_us"):
        assert cal[key] > 0, key
    return bs.calibrated_options(cal)


def _time(P, a, b, c, flush, reps=30):
    ts = []
    for r in range(reps + 3):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        bs.contract(P, a, b, c)
        e1.record()
        torch.cuda.synchronize()
        if r >= 3:
            ts.append(e0.elapsed_time(e1) * 1e3)
    assert bs.last_device_error(P) == 0
    return statistics.median(ts)


CASES = [("toy", 1, None), ("tail", 2, None), ("tail_blockrow", 2, "blockrow")]


@pytest.mark.parametrize("name,cfg,lay", CASES, ids=[c[0] for c in CASES])
def test_model_pick_is_within_ten_percent_of_the_fastest_candidate(calibrated, name, cfg, lay):
    w = bsgen.get(cfg)
    la, lb, lc = (lay or w.layout_a, lay or w.layout_b, lay or w.layout_c)
    A = bs.Layout(w.rows, w.inner, w.rule_a, la, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, lb, 8)
    a = torch.from_numpy(operand_host(w, 0, A.blocks(), A.nelems)).cuda()
    b = torch.from_numpy(operand_host(w, 1, B.blocks(), B.nelems)).cuda()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    auto = bs.Plan(A, B, bs.F64, c_layout_flags=lc, **calibrated)
    sa = auto.stats()
    chosen = (sa["axis"], bs.PACK_ALWAYS if (sa["packed_a"] or sa["packed_b"]) else bs.PACK_NEVER)
    c = torch.zeros(max(auto.c_layout.nelems, 1), dtype=torch.float64, device="cuda")
    times, models = {}, {}
    for axis in (bs.AXIS_CONTRACTION, bs.AXIS_FREE):
        for pack in (bs.PACK_NEVER, bs.PACK_ALWAYS):
            P = bs.Plan(A, B, bs.F64, c_layout_flags=lc, axis_policy=axis, pack_policy=pack, **calibrated)
            times[(axis, pack)] = _time(P, a, b, c, flush)
            models[(axis, pack)] = P.stats()["model_us"]
    best = min(times.values())
    print(f"[model] {name}: measured {({k: round(v, 1) for k, v in times.items()})}, "
          f"model {({k: round(v, 1) for k, v in models.items()})}, chosen {chosen}")
    assert times[chosen] <= 1.10 * best, f"chosen {chosen} at {times[chosen]:.1f} us, fastest {best:.1f} us"
    assert sa["model_us"] == pytest.approx(models[chosen], rel=1e-9)
