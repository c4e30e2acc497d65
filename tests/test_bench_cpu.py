"""CPU checks of bench.py: the reference (oracle) arm, its torchrun launch with two
ranks, and the max-over-ranks timing reduction under a gloo process group."""
import json
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _json_lines(out: str):
    return [json.loads(l) for l in out.splitlines() if l.startswith("{")]


def test_reference_arm_prints_one_line():
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "2", "--warmup", "3",
                        "--cpu-workers", "2", "--config", "2"], cwd=ROOT, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = _json_lines(r.stdout)
    assert len(lines) == 1
    d = lines[0]
    assert d["impl"] == "reference" and d["unit"] == "GFLOP/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["e2e"]["h2d_bytes_per_step"] == 0
    assert d["warmup"] >= 3 and d["steps"] == 2
    assert d["cpu_baseline"]["cores"] == 2


def test_reference_arm_under_torchrun_two_ranks():
    port = _free_port()
    r = subprocess.run([sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
                        "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3", "--cpu-workers", "2",
                        "--config", "1"],
                       cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = _json_lines(r.stdout)
    assert len(lines) == 1 and lines[0]["n_gpus"] == 2


_WORKER = r'''
import os, sys
sys.path.insert(0, os.environ["ROOT"])
import torch.distributed as dist
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:" + os.environ["PORT"],
                        rank=int(os.environ["RANK"]), world_size=2)
import bench
rank = dist.get_rank()
got = bench.max_over_ranks(1.5 + rank, device="cpu")
assert got == 2.5, got
assert bench.weak_scaling_value(100.0, 2, got) == 2 * 100.0 / 2.5e-3
dist.destroy_process_group()
print("ok", rank)
'''


def test_max_over_ranks_with_gloo_world_size_two():
    port = str(_free_port())
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, PORT=port, RANK=str(rank))
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=300) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-2000:]
        assert o.strip().startswith("ok")


def test_oracle_pool_covers_every_c_block_once():
    """The all-cores baseline deals each populated C block to exactly one worker."""
    import numpy as np
    import bench
    import oracle
    pool = bench.OraclePool(1, workers=3)
    try:
        got = np.concatenate(pool.parts)
        want = np.argwhere(oracle.problem(bench.bsgen.get(1)).mc)
        assert len(got) == len(want) == len({tuple(x) for x in got.tolist()})
        assert {tuple(x) for x in got.tolist()} == {tuple(x) for x in want.tolist()}
        pool.step()
    finally:
        pool.close()
