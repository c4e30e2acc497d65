#!/usr/bin/env python
"""Benchmark of the coalesced block-sparse contraction C[i,j] = sum_k A[i,k] B[k,j].

One step = one bs_contract over the headline workload (default: the FP64
launch-bound stress workload, 2000 random Z2 x U(1) sectors per axis with dims
1..8 and sixteen sectors of 1024, 4.7 M populated block triples, 455 MB of
operands and output), inputs resident in HBM, L2 flushed between steps by a
256 MiB write (the inputs are larger than L2 as well).  Prints one JSON line:
useful GFLOP/s (sum over populated triples of 2 d_i d_k d_j per second),
blocks/s (populated triples per second), the roofline of the grouped kernel,
an end-to-end number through the host-buffer entry point, the CPU oracle on
the host cores, the one-launch-per-triple control, sampled clocks, and a
per-workload summary of the other synthetic workloads, the chained
contraction, bucketing and the gather kernel.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--config n]

For N > 1 (torchrun) every rank runs its own replica of the workload (weak
scaling); the only collectives are the timing barrier and the max over ranks.
`--impl reference` times the CPU oracle instead, on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import bsgen  # noqa: E402

METRIC = "useful GFLOP/s + blocks/s per contraction; fraction of FP64/BF16 roofline"
FP64_FLOP_PER_CLK_PER_SM = 4          # 1.25 TFLOP/s nominal over 152 SMs at 2070 MHz
NOMINAL_SMS, NOMINAL_MAX_MHZ = 152, 2070.0


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    return int(os.environ.get("RANK", 0)), int(os.environ.get("LOCAL_RANK", 0)), int(os.environ.get("WORLD_SIZE", 1))


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank number over the process group (identity without one)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def weak_scaling_value(per_rank_units: float, world: int, ms_max: float) -> float:
    """Whole-job throughput: every rank processes the same units; time is the slowest rank's."""
    return world * per_rank_units / (ms_max * 1e-3)


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except (OSError, ValueError):
        return {}


def workload_desc(w: bsgen.Workload) -> str:
    return (f"{w.name}: {w.rows.n}x{w.inner.n}x{w.cols.n} sectors, rules A {w.rule_a.dq_min}..{w.rule_a.dq_max}"
            f"{' +parity' if w.rule_a.z2 else ''}, B {w.rule_b.dq_min}..{w.rule_b.dq_max}, values {w.values}, "
            f"layouts A={w.layout_a} B={w.layout_b} C={w.layout_c}")


# ------------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons while it runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.f = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        self.dev = device_index
        self.p = None

    def start(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "50"], stdout=self.f,
                                      stderr=subprocess.DEVNULL)
        except OSError:
            self.p = None
        self.t0 = time.time()

    def stop(self):
        if self.p is not None:
            self.p.terminate()
            try:
                self.p.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.p.kill()
        self.f.flush()
        self.f.seek(0)
        rows = [r.split(",") for r in self.f.read().strip().splitlines() if r.strip()]
        os.unlink(self.f.name)
        mhz, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                mhz.append(float(r[1]))
                mx.append(float(r[2]))
                for n, v in zip(names, r[5:9]):
                    if v.strip().lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                pass
        return {"sm_mhz": statistics.median(mhz) if mhz else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(mhz)}


# ------------------------------------------------------------------------- GPU arm
PLAN_OPTS = {}   # cost-model constants measured on the device (bs_calibrate), given to every plan


class Problem:
    """Layouts, plan and resident device buffers of one workload."""

    def __init__(self, bs, torch, w: bsgen.Workload, **opts):
        opts = {**PLAN_OPTS, **opts}
        self.w = w
        eb = 2 if w.dtype == "bf16" else 8
        self.A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, eb)
        self.B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, eb)
        self.P = bs.Plan(self.A, self.B, bs.BF16_F32 if w.dtype == "bf16" else bs.F64, c_layout_flags=w.layout_c, **opts)
        self.stats = self.P.stats()
        self.a_host = self._operand(0, self.A)
        self.b_host = self._operand(1, self.B)
        self.a = torch.from_numpy(self.a_host).cuda()
        self.b = torch.from_numpy(self.b_host).cuda()
        cdt = torch.float32 if w.dtype == "bf16" else torch.float64
        self.c = torch.zeros(max(self.P.c_layout.nelems, 1), dtype=cdt, device="cuda")

    def _operand(self, op, L):
        b = L.blocks()
        vals = self.w.draw(op, b[:, 0], b[:, 1], b[:, 3], b[:, 4])
        buf = np.zeros(L.nelems)
        buf[L.element_index(b)] = vals
        if self.w.dtype == "bf16":
            return bsgen.rng.bf16_bits(buf).view(np.int16)
        return buf


def time_steps(torch, fn, steps, warmup, flush, stream):
    """Per-step CUDA-event times (ms) on `stream`, L2 flushed before every step."""
    for _ in range(warmup):
        flush.zero_()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in ev:
        flush.zero_()
        s.record(stream)
        fn()
        e.record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in ev]


def kernel_source_tag(dtype: str) -> str:
    src = "bs_bf16.cu" if dtype == "bf16" else "bs_fp64.cu"
    with open(os.path.join(ROOT, "block_sparse_tensor_gb300", "csrc", src), "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:12]


def recorded_traffic(workload: str, tag: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on this kernel source."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    try:
        for line in open(path):
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload and parts[1] == tag:
                return float(parts[2])
    except OSError:
        pass
    return None


def fp64_nominal_tflops():
    return NOMINAL_SMS * FP64_FLOP_PER_CLK_PER_SM * NOMINAL_MAX_MHZ * 1e6 / 1e12


def roofline(w, stats, kernel_ms, calib, peaks, clock_mhz):
    if w.dtype == "bf16":
        # BF16 workload: intensity below the tensor ridge, so HBM bounds it
        hbm = peaks.get("hbm_gbs") or 6800.0
        achieved = stats["useful_bytes"] / (kernel_ms * 1e-3) / 1e9
        out = {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
               "peak_source": "of measured: MEASURED_PEAKS.json hbm_gbs" if peaks.get("hbm_gbs") else "of fallback 6.8 TB/s"}
    else:
        # The FP64 pipe: 4 flop per SM clock at the maximum SM clock.  The probes
        # (bs_calibrate: FMA chains and the FP64 matrix instruction) measure the
        # rate at the clock the part holds under that load, which is lower; the
        # nominal figure is kept as the denominator because it is the higher one.
        peak = fp64_nominal_tflops()
        achieved = stats["useful_flops"] / (kernel_ms * 1e-3) / 1e12
        out = {"bound": "alu", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
               "peak_source": "FP64 pipe: 152 SMs x 4 flop/clk x 2070 MHz (nominal 1.25 TFLOP/s), above every "
                              "measured probe rate"}
        if calib:
            out["fp64_probe_tflops"] = calib["fp64_gflops"] / 1e3
            out["fp64_dmma_probe_tflops"] = calib.get("fp64_dmma_gflops", 0.0) / 1e3
            out["fp64_probe_flop_per_clk_sm"] = calib.get("fp64_flop_per_clk_sm")
            out["fp64_probe_sm_mhz"] = calib.get("fp64_sm_mhz")
        if clock_mhz:
            out["frac_at_sampled_clock"] = achieved / (peak * clock_mhz / NOMINAL_MAX_MHZ)
    return out


def control_record(bs, torch, pb, ms, flush, stream, reps):
    """The one-launch-per-triple control on the same plan and buffers."""
    ctrl = lambda: bs.contract_uncoalesced(pb.P, pb.a, pb.b, pb.c, stream)  # noqa: E731
    cms = statistics.median(time_steps(torch, ctrl, reps, 1 if reps > 1 else 0, flush, stream))
    st = pb.stats
    return {"ms": cms, "speedup": cms / ms, "launches_per_s": st["triples"] / (cms * 1e-3),
            "gflops": st["useful_flops"] / (cms * 1e-3) / 1e9, "repeats": reps}


def run_gpu(args):
    import torch

    import block_sparse_tensor_gb300 as bs

    rank, local, world = dist_env()
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    stream = torch.cuda.current_stream()
    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    peaks = measured_peaks()
    calib = None if args.skip_calib else bs.calibrate(stream)
    log(f"[bench] calibration: {calib}")
    if calib:
        PLAN_OPTS.update(bs.calibrated_options(calib))

    w = workload(args)
    pb = Problem(bs, torch, w)
    st = pb.stats
    fn = lambda: bs.contract(pb.P, pb.a, pb.b, pb.c, stream)  # noqa: E731
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.2)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times = time_steps(torch, fn, args.steps, args.warmup, flush, stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks = sampler.stop()
    assert bs.last_device_error(pb.P, stream) == 0
    ms = max_over_ranks(statistics.mean(times), device="cuda")
    value = weak_scaling_value(st["useful_flops"], world, ms) / 1e9
    blocks_s = weak_scaling_value(st["triples"], world, ms)

    # end to end through the host-buffer entry point, pinned buffers: every call
    # copies A and B in and C back and synchronizes
    a_pin = torch.from_numpy(pb.a_host).pin_memory()
    b_pin = torch.from_numpy(pb.b_host).pin_memory()
    c_pin = torch.zeros(pb.c.numel(), dtype=pb.c.dtype).pin_memory()
    bs.contract_host(pb.P, a_pin, b_pin, c_pin, stream)
    e2e_t = []
    for _ in range(max(args.steps, 5)):
        t0 = time.perf_counter()
        bs.contract_host(pb.P, a_pin, b_pin, c_pin, stream)
        e2e_t.append(time.perf_counter() - t0)
    e2e_s = max_over_ranks(statistics.mean(e2e_t), device="cuda")
    del a_pin, b_pin, c_pin

    line = {
        "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if w.dtype == "bf16" else "f64", "data": "synthetic",
        "blocks_per_s": blocks_s,   # populated (i, k, j) triples per second
        "c_blocks_per_s": weak_scaling_value(st["c_blocks"], world, ms),
        "config": {"workload": workload_desc(w), "triples": st["triples"], "c_blocks": st["c_blocks"],
                   "useful_gflop": st["useful_flops"] / 1e9, "useful_mb": st["useful_bytes"] / 1e6,
                   "groups": st["groups"], "axis": ["auto", "contraction", "free", "none"][st["axis"]],
                   "packed": bool(st["packed_a"] or st["packed_b"]),
                   "l2": "flushed before every step (256 MiB write, untimed)"
                         + ("; inputs larger than L2" if st["useful_bytes"] > 129e6 else ""),
                   "parallelism": f"replicas x{world}" if world > 1 else "1 GPU"},
        "gpu_launches": args.steps * st["launches"],
    }
    # one bs_contract is one kernel when the plan neither gathers nor zero-fills,
    # so the step time is that kernel's launch duration
    kernel_ms = ms
    rl = roofline(w, st, kernel_ms, calib, peaks, clocks.get("sm_mhz"))
    tag = kernel_source_tag(w.dtype)
    rl["traffic"] = recorded_traffic(w.name, tag)
    rl["kernel"] = "bf16_grouped_kernel" if w.dtype == "bf16" else "fp64_grouped_kernel"
    rl["kernel_source"] = tag
    rl["launches_per_step"] = st["launches"]
    line["roofline"] = rl
    line["e2e"] = {"value": world * st["useful_flops"] / e2e_s / 1e9, "unit": "GFLOP/s",
                   "h2d_bytes_per_step": int(pb.a_host.nbytes + pb.b_host.nbytes),
                   "d2h_bytes_per_step": int(pb.c.numel() * pb.c.element_size()),
                   "ms_per_step": e2e_s * 1e3, "entry_point": "bs_contract_host (pinned host buffers)"}
    line["clocks"] = clocks
    line["calibration"] = calib
    line["model_us"] = st["model_us"]
    line["model_over_measured"] = st["model_us"] / (ms * 1e3) if st["model_us"] else None
    line["plan_ms"] = st["plan_ms"]
    if not args.skip_control:
        line["control"] = control_record(bs, torch, pb, ms, flush, stream, 1 if st["triples"] > 1e6 else 3)
        log(f"[bench] control: {json.dumps(line['control'])}")

    if rank == 0 and world == 1 and not args.skip_cpu:
        line["cpu_baseline"] = cpu_baseline(args.config, budget_s=args.cpu_seconds, workers=args.cpu_workers)
    if not args.skip_configs:
        del pb
        torch.cuda.empty_cache()
        line["per_config"] = per_config(bs, torch, flush, stream, calib, peaks, args, clocks.get("sm_mhz"))
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


def per_config(bs, torch, flush, stream, calib, peaks, args, clock_mhz):
    out = {}
    for n in sorted(bsgen.CONFIGS):
        if n == args.config:
            continue
        w = bsgen.get(n)
        t0 = time.time()
        pb = Problem(bs, torch, w)
        st = pb.stats
        setup_s = time.time() - t0
        steps = 10 if n != 1 else 50
        ms = statistics.median(time_steps(torch, lambda: bs.contract(pb.P, pb.a, pb.b, pb.c, stream), steps, 3,
                                          flush, stream))
        assert bs.last_device_error(pb.P, stream) == 0
        rl = roofline(w, st, ms, calib, peaks, clock_mhz)
        rec = {"workload": w.name, "dtype": w.dtype, "ms": ms, "gflops": st["useful_flops"] / (ms * 1e-3) / 1e9,
               "blocks_per_s": st["triples"] / (ms * 1e-3), "c_blocks_per_s": st["c_blocks"] / (ms * 1e-3),
               "triples": st["triples"], "c_blocks": st["c_blocks"],
               "groups": st["groups"], "tasks": st["tasks"], "useful_gflop": st["useful_flops"] / 1e9,
               "useful_mb": st["useful_bytes"] / 1e6, "roofline_frac": rl["frac"], "roofline_bound": rl["bound"],
               "roofline_achieved": rl["achieved"], "roofline_unit": rl["unit"], "roofline_peak": rl["peak"],
               "traffic": recorded_traffic(w.name, kernel_source_tag(w.dtype)),
               "executed_over_useful": st["executed_flops"] / max(st["useful_flops"], 1),
               "plan_ms": st["plan_ms"], "model_us": st["model_us"],
               "model_over_measured": st["model_us"] / (ms * 1e3) if st["model_us"] else None, "setup_s": setup_s}
        if not args.skip_control:
            rec["control"] = control_record(bs, torch, pb, ms, flush, stream, 3)
        out[str(n)] = rec
        log(f"[bench] config {n}: {json.dumps(rec)}")
        del pb
        torch.cuda.empty_cache()
    out["4_align64"] = align64_record(bs, torch, flush, stream, calib, peaks, clock_mhz)
    log(f"[bench] 4_align64: {json.dumps(out['4_align64'])}")
    out["chain"] = chain_record(bs, torch, flush, stream)
    log(f"[bench] chain: {json.dumps(out['chain'])}")
    out["bucket"] = bucket_record(bs, torch, flush, stream)
    log(f"[bench] bucket: {json.dumps(out['bucket'])}")
    out["gather"] = gather_record(bs, torch, flush, stream, peaks)
    log(f"[bench] gather: {json.dumps(out['gather'])}")
    return out


def gather_record(bs, torch, flush, stream, peaks):
    """The gather ("pack") kernel on the pack-exercise layouts (every operand in
    block-row order, gathered into charge-sorted panels), timed by the plan's own
    phase events: bytes moved = 2 x packed bytes (each element read and written once)."""
    hbm = peaks.get("hbm_gbs") or 6800.0
    out = {}
    for n, opts in ((5, dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)),
                    (2, dict(axis_policy=bs.AXIS_CONTRACTION, pack_policy=bs.PACK_ALWAYS)), (4, {})):
        w = bsgen.get(n)
        w.layout_a, w.layout_b, w.layout_c = w.pack_layout_a, w.pack_layout_b, w.pack_layout_c
        pb = Problem(bs, torch, w, profile=1, **opts)
        g, k, tot = [], [], []
        for _ in range(3 + 10):
            flush.zero_()
            bs.contract(pb.P, pb.a, pb.b, pb.c, stream)
            pr = pb.P.profile()
            g.append(pr["gather_ms"])
            k.append(pr["kernel_ms"])
            tot.append(pr["total_ms"])
        assert bs.last_device_error(pb.P, stream) == 0
        gm = statistics.median(g[3:])
        gbs = pr["gather_bytes"] / (gm * 1e-3) / 1e9
        out[str(n)] = {"workload": w.name + " (block-row operands)", "gather_ms": gm, "gather_bytes": pr["gather_bytes"],
                       "gather_gbs": gbs, "gather_frac_of_hbm": gbs / hbm, "kernel_ms": statistics.median(k[3:]),
                       "contract_ms": statistics.median(tot[3:]),
                       "gflops": pb.stats["useful_flops"] / (statistics.median(tot[3:]) * 1e-3) / 1e9}
        del pb
        torch.cuda.empty_cache()
    return out


def bucket_record(bs, torch, flush, stream):
    """Exact grouping against tail groups padded to power-of-two buckets, workload 2."""
    w = bsgen.config2()
    rec = {"workload": w.name}
    for name, axis in (("contraction", bs.AXIS_CONTRACTION), ("none", bs.AXIS_NONE)):
        for pad in (0, 1):
            pb = Problem(bs, torch, w, axis_policy=axis, bucket_pad=pad)
            ms = statistics.median(time_steps(torch, lambda: bs.contract(pb.P, pb.a, pb.b, pb.c, stream), 50, 3, flush,
                                              stream))
            st = pb.stats
            rec[f"{name}_{'padded' if pad else 'exact'}"] = {
                "ms": ms, "gflops": st["useful_flops"] / (ms * 1e-3) / 1e9,
                "executed_over_useful": st["executed_flops"] / st["useful_flops"], "tail_pieces": st["tail_tasks"]}
            del pb
    return rec


def align64_record(bs, torch, flush, stream, calib, peaks, clock_mhz):
    """The BF16 workload with its three layouts padded to 64 bytes instead of 16 (every row the
    kernel's tensor-map copies read starts on a 64-byte boundary); same values, same useful bytes."""
    w = bsgen.get(4)
    w.layout_a, w.layout_b, w.layout_c = (x.replace("align16", "align64") for x in (w.layout_a, w.layout_b, w.layout_c))
    pb = Problem(bs, torch, w)
    st = pb.stats
    ms = statistics.median(time_steps(torch, lambda: bs.contract(pb.P, pb.a, pb.b, pb.c, stream), 10, 3, flush, stream))
    assert bs.last_device_error(pb.P, stream) == 0
    rl = roofline(w, st, ms, calib, peaks, clock_mhz)
    padded = 2 * (pb.a.numel() + pb.b.numel()) + 4 * pb.c.numel()
    rec = {"workload": w.name + " (layouts " + w.layout_a + ", " + w.layout_b + ", " + w.layout_c + ")", "ms": ms,
           "gflops": st["useful_flops"] / (ms * 1e-3) / 1e9, "useful_mb": st["useful_bytes"] / 1e6,
           "layout_mb": padded / 1e6, "roofline_frac": rl["frac"], "roofline_bound": rl["bound"],
           "roofline_achieved": rl["achieved"], "roofline_unit": rl["unit"], "roofline_peak": rl["peak"]}
    del pb
    torch.cuda.empty_cache()
    return rec


def workload(args):
    """The timed workload; --align64 pads its layouts to 64 bytes instead of 16."""
    w = bsgen.get(args.config)
    if args.align64:
        w.layout_a, w.layout_b, w.layout_c = (x.replace("align16", "align64") if "align16" in x else x + "|align64"
                                              for x in (w.layout_a, w.layout_b, w.layout_c))
    return w


def chain_record(bs, torch, flush, stream):
    """Two chained contractions T = A B (free axis), Y = T D (contraction axis), T on the device;
    then the same chain with each stage's axis chosen by the cost model."""
    w1, w2 = bsgen.chain2()
    A = bs.Layout(w1.rows, w1.inner, w1.rule_a, w1.layout_a, 8)
    B = bs.Layout(w1.inner, w1.cols, w1.rule_b, w1.layout_b, 8)
    D = bs.Layout(w2.inner, w2.cols, w2.rule_b, w2.layout_b, 8)
    rec = _chain_run(bs, torch, flush, stream, w1, w2, A, B, D, bs.AXIS_FREE, bs.AXIS_CONTRACTION)
    rec["auto"] = _chain_run(bs, torch, flush, stream, w1, w2, A, B, D, bs.AXIS_AUTO, bs.AXIS_AUTO)
    return rec


def _chain_run(bs, torch, flush, stream, w1, w2, A, B, D, axis1, axis2):
    P1 = bs.Plan(A, B, bs.F64, axis_policy=axis1, c_layout_flags=w1.layout_c, **PLAN_OPTS)
    P2 = bs.Plan(P1.c_layout, D, bs.F64, axis_policy=axis2, c_layout_flags=w2.layout_c, **PLAN_OPTS)

    def dev(w, op, L):
        b = L.blocks()
        buf = np.zeros(L.nelems)
        buf[L.element_index(b)] = w.draw(op, b[:, 0], b[:, 1], b[:, 3], b[:, 4])
        return torch.from_numpy(buf).cuda()

    a, b, d = dev(w1, 0, A), dev(w1, 1, B), dev(w2, 1, D)
    t = torch.zeros(P1.c_layout.nelems, dtype=torch.float64, device="cuda")
    y = torch.zeros(P2.c_layout.nelems, dtype=torch.float64, device="cuda")

    def step():
        bs.contract(P1, a, b, t, stream)
        bs.contract(P2, t, d, y, stream)

    ms = statistics.median(time_steps(torch, step, 20, 3, flush, stream))
    s1, s2 = P1.stats(), P2.stats()
    fl = s1["useful_flops"] + s2["useful_flops"]
    names = ["auto", "contraction", "free", "none"]
    return {"workload": "chain " + w1.name + " -> " + w2.name, "ms": ms, "gflops": fl / (ms * 1e-3) / 1e9,
            "stage_axes": [names[s1["axis"]], names[s2["axis"]]], "launches": s1["launches"] + s2["launches"],
            "useful_gflop": fl / 1e9, "triples": s1["triples"] + s2["triples"],
            "roofline_frac": fl / (ms * 1e-3) / 1e12 / (NOMINAL_SMS * FP64_FLOP_PER_CLK_PER_SM * NOMINAL_MAX_MHZ * 1e6 / 1e12)}


# ------------------------------------------------------------------------- CPU oracle
def _workload_flops(w, pr):
    ma, mb = pr.ma.astype(np.int64), pr.mb.astype(np.int64)
    flops, triples = 0.0, 0
    for i, k in zip(*np.nonzero(ma)):
        js = np.nonzero(mb[k])[0]
        triples += len(js)
        flops += 2.0 * int(w.rows.d[i]) * int(w.inner.d[k]) * float(w.cols.d[js].astype(np.int64).sum())
    return flops, triples


_POOL_PR = None


def _pool_init(n):
    global _POOL_PR
    import oracle
    _POOL_PR = oracle.problem(bsgen.get(n))


def _pool_contract(sel):
    import oracle
    oracle.contract(_POOL_PR, sel=sel)
    return len(sel)


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name"):
                return line.split(":", 1)[1].strip()
    except Exception:
        pass
    return platform.processor() or platform.machine()


class OraclePool:
    """The oracle as it stands, run over every host core: worker processes (spawned,
    so they never inherit a CUDA context) each hold the problem and compute a slice
    of the C blocks, the slices dealt longest-first by flops so they take equal time."""

    def __init__(self, n: int, workers: int = 0):
        import multiprocessing as mp
        import oracle
        w = bsgen.get(n)
        pr = oracle.problem(w)
        self.flops, self.triples = _workload_flops(w, pr)
        cores = len(os.sched_getaffinity(0))
        ij = np.argwhere(pr.mc)
        cost = [float(w.rows.d[i]) * float(w.cols.d[j]) * float(w.inner.d[np.nonzero(pr.ma[i] * pr.mb[:, j])[0]].sum())
                for i, j in ij]
        self.workers = max(1, min(workers or cores, len(ij)))
        load = [0.0] * self.workers
        parts = [[] for _ in range(self.workers)]
        for t in np.argsort(cost)[::-1]:
            b = int(np.argmin(load))
            load[b] += cost[t]
            parts[b].append(ij[t])
        self.parts = [np.asarray(p, np.int32).reshape(-1, 2) for p in parts if p]
        self.pool = mp.get_context("spawn").Pool(len(self.parts), initializer=_pool_init, initargs=(n,))

    def step(self):
        done = sum(self.pool.map(_pool_contract, self.parts, chunksize=1))
        assert done == sum(len(p) for p in self.parts)

    def close(self):
        self.pool.close()
        self.pool.join()


def cpu_baseline(n: int, budget_s: float = 12.0, workers: int = 0):
    """The oracle as it stands on the host cores, on the same workload: over every
    core (C blocks dealt longest-first over worker processes), the full contraction
    per step; and single-threaded, on one worker's share of the C blocks."""
    pool = OraclePool(n, workers)
    try:
        pool.step()   # workers warm
        reps, t0 = 0, time.perf_counter()
        while True:
            pool.step()
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s / 2 or (reps >= 1 and el * (reps + 1) / reps > budget_s):
                break
        # one core: the first worker's share, run in this process
        import oracle
        w = bsgen.get(n)
        pr = oracle.problem(w)
        share = pool.parts[0]
        sfl = sum(2.0 * float(w.rows.d[i]) * float(w.cols.d[j]) *
                  float(w.inner.d[np.nonzero(pr.ma[i] * pr.mb[:, j])[0]].sum()) for i, j in share)
        t1 = time.perf_counter()
        oracle.contract(pr, sel=share)
        el1 = time.perf_counter() - t1
    finally:
        pool.close()
    single = {"value": sfl / el1 / 1e9, "unit": "GFLOP/s", "cores": 1, "kind": "oracle",
              "sample": f"{len(share)} of the {w.name} C blocks ({sfl / pool.flops:.1%} of its flops) in {el1:.1f} s "
                        f"(plain C triple loop, FP64)"}
    return {"value": pool.flops * reps / el / 1e9, "unit": "GFLOP/s", "cores": pool.workers, "kind": "oracle",
            "sample": f"the full {w.name} contraction, {reps} times in {el:.1f} s, its C blocks dealt over "
                      f"{pool.workers} worker processes on {cpu_model()}",
            "single_core": single}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return
    w = bsgen.get(args.config)
    pool = OraclePool(args.config, args.cpu_workers)
    try:
        for _ in range(args.warmup):
            pool.step()
        ts = []
        for _ in range(args.steps):
            t0 = time.perf_counter()
            pool.step()
            ts.append(time.perf_counter() - t0)
    finally:
        pool.close()
    s = statistics.mean(ts)
    value = pool.flops / s / 1e9
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": s * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64" if w.dtype == "f64" else "bf16",
            "data": "synthetic", "blocks_per_s": pool.triples / s,
            "config": {"workload": workload_desc(w), "triples": pool.triples,
                       "parallelism": f"{pool.workers} host cores"},
            "cpu_baseline": {"value": value, "unit": "GFLOP/s", "cores": pool.workers, "kind": "oracle",
                             "sample": f"each step is the full {w.name} contraction by the plain C oracle, its C "
                                       f"blocks dealt over {pool.workers} worker processes on {cpu_model()}"},
            "e2e": {"value": value, "unit": "GFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--config", type=int, default=5, choices=sorted(bsgen.CONFIGS))
    ap.add_argument("--skip-configs", action="store_true", help="headline workload only")
    ap.add_argument("--skip-control", action="store_true", help="skip the one-launch-per-triple controls")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--cpu-workers", type=int, default=0, help="oracle worker processes (0: every core)")
    ap.add_argument("--skip-calib", action="store_true", help="skip the probe kernels (profiling runs)")
    ap.add_argument("--align64", action="store_true",
                    help="the workload's layouts padded to 64 bytes (profiling and layout comparisons)")
    ap.add_argument("--gather-only", action="store_true",
                    help="only time the gather kernel on the block-row layouts (profiling runs)")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        run_reference(args)
    elif args.gather_only:
        import torch

        import block_sparse_tensor_gb300 as bs
        torch.cuda.set_device(0)
        flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
        print(json.dumps(gather_record(bs, torch, flush, torch.cuda.current_stream(), measured_peaks())), flush=True)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
