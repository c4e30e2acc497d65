"""C-block sharding of a contraction over several ranks (bs_plan_create_shard).

On the CPU, two gloo ranks each build their shard's host-only plan and exchange
what it covers: the shards' triples are exactly the full contraction's, their C
blocks are disjoint and cover every populated block, and their flops are
balanced.  On a GPU, the shards of one contraction run one after the other into
one C buffer: each writes only its own blocks, and together they match the
oracle on every block."""
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

import bsgen

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_WORKER = r'''
import os, sys
sys.path.insert(0, os.environ["ROOT"])
import numpy as np
import torch.distributed as dist
dist.init_process_group("gloo", init_method="tcp://127.0.0.1:" + os.environ["PORT"],
                        rank=int(os.environ["RANK"]), world_size=2)
import bsgen
import block_sparse_tensor_gb300 as bs
rank, world = dist.get_rank(), dist.get_world_size()
for cfg in (1, 2, 5):
    w = bsgen.get(cfg)
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, 8)
    for pol in (bs.AXIS_CONTRACTION, bs.AXIS_FREE, bs.AXIS_NONE):
        if cfg == 5 and pol != bs.AXIS_CONTRACTION:
            continue
        P = bs.Plan(A, B, bs.F64, c_layout_flags=w.layout_c, host_only=1, axis_policy=pol, shard=(rank, world))
        _, tr = P.triples()
        mine = {"tr": tr.astype(np.int64), "c": P.operand_blocks(2), "flops": P.stats()["useful_flops"],
                "c_blocks": P.stats()["c_blocks"], "ok": P.check_groups()[0]}
        got = [None] * world
        dist.all_gather_object(got, mine)
        if rank == 0:
            full = bs.Plan(A, B, bs.F64, c_layout_flags=w.layout_c, host_only=1, axis_policy=pol)
            _, ftr = full.triples()
            allt = np.concatenate([g["tr"] for g in got])
            key = lambda t: t[:, 0] * (1 << 42) + t[:, 1] * (1 << 21) + t[:, 2]
            assert len(allt) == len(ftr), (cfg, pol, len(allt), len(ftr))
            assert np.array_equal(np.sort(key(allt)), np.sort(key(ftr.astype(np.int64)))), (cfg, pol)
            cs = np.concatenate([g["c"] for g in got])
            assert len(cs) == len(set(cs.tolist())) == full.stats()["c_blocks"], (cfg, pol)
            assert sum(g["c_blocks"] for g in got) == full.stats()["c_blocks"]
            assert all(g["ok"] == 0 for g in got)
            fl = [g["flops"] for g in got]
            assert abs(sum(fl) - full.stats()["useful_flops"]) <= 1e-9 * sum(fl)
            big = max(fl) / (sum(fl) / world)
            assert big < 1.05 or cfg == 5, (cfg, pol, fl)   # the stress workload's largest C blocks are lumpy
            print("shard", cfg, pol, [round(x / sum(fl), 4) for x in fl], flush=True)
dist.barrier()
dist.destroy_process_group()
print("ok", rank)
'''


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def test_shards_cover_the_contraction_exactly_with_gloo_world_size_two():
    pytest.importorskip("block_sparse_tensor_gb300")
    port = str(_free_port())
    procs = []
    for rank in range(2):
        env = dict(os.environ, ROOT=ROOT, PORT=port, RANK=str(rank))
        procs.append(subprocess.Popen([sys.executable, "-c", _WORKER], env=env, stdout=subprocess.PIPE,
                                      stderr=subprocess.PIPE, text=True))
    outs = [p.communicate(timeout=600) for p in procs]
    for p, (o, e) in zip(procs, outs):
        assert p.returncode == 0, e[-3000:]
        assert o.strip().endswith(f"ok {procs.index(p)}")


def test_shard_arguments_are_checked():
    bs = pytest.importorskip("block_sparse_tensor_gb300")
    w = bsgen.config1()
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, 8)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, 8)
    for rank, world in ((0, 0), (2, 2), (-1, 2)):
        with pytest.raises(bs.BsError) as e:
            bs.Plan(A, B, bs.F64, host_only=1, shard=(rank, world))
        assert e.value.code == 1
    one = bs.Plan(A, B, bs.F64, host_only=1, shard=(0, 1))
    assert one.stats()["c_blocks"] == 39 and one.stats()["triples"] == 71
    # a shard reads only the A and B blocks of its own triples
    s0 = bs.Plan(A, B, bs.F64, host_only=1, shard=(0, 3))
    _, tr = s0.triples()
    ablk = A.blocks()
    want = sorted({int(np.nonzero((ablk[:, 0] == i) & (ablk[:, 1] == k))[0][0]) for i, k, _ in tr})
    assert s0.operand_blocks(0).tolist() == want


@pytest.mark.gpu
@pytest.mark.parametrize("cfg,world", [(2, 2), (2, 3), (5, 2), (4, 2)])
def test_shards_run_one_after_another_match_the_oracle(cfg, world):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import block_sparse_tensor_gb300 as bs
    from harness import TOL, check_blocks, element_index, oracle_all_blocks, operand_host, sort_rc
    w = bsgen.get(cfg)
    eb = 2 if w.dtype == "bf16" else 8
    A = bs.Layout(w.rows, w.inner, w.rule_a, w.layout_a, eb)
    B = bs.Layout(w.inner, w.cols, w.rule_b, w.layout_b, eb)
    dt = bs.BF16_F32 if w.dtype == "bf16" else bs.F64
    plans = [bs.Plan(A, B, dt, c_layout_flags=w.layout_c, shard=(r, world)) for r in range(world)]
    ah, bh = operand_host(w, 0, A.blocks(), A.nelems), operand_host(w, 1, B.blocks(), B.nelems)
    a = torch.from_numpy(ah.view(np.int16) if eb == 2 else ah).cuda()
    b = torch.from_numpy(bh.view(np.int16) if eb == 2 else bh).cuda()
    cdt = torch.float32 if eb == 2 else torch.float64
    c = torch.full((plans[0].c_layout.nelems,), float("nan"), dtype=cdt, device="cuda")
    cblocks = plans[0].c_layout.blocks()
    for r, P in enumerate(plans):
        bs.contract(P, a, b, c)
        torch.cuda.synchronize()
        assert bs.last_device_error(P) == 0
        got = c.cpu().numpy()
        done = np.concatenate([p.operand_blocks(2) for p in plans[:r + 1]])
        rest = np.setdiff1d(np.arange(len(cblocks)), done)
        assert not np.any(np.isnan(got[element_index(cblocks[done])]))
        if len(rest):
            assert np.all(np.isnan(got[element_index(cblocks[rest])])), "a shard wrote another shard's block"
    C, S, pr = oracle_all_blocks(w, w.layout_a, w.layout_b, w.layout_c)
    lib_c = sort_rc(cblocks)
    assert np.array_equal(lib_c, pr.lc.blocks())
    ok, worst, ncancel = check_blocks(c.cpu().numpy().astype(np.float64), C, S, lib_c, TOL[w.dtype])
    print(f"[parity] {w.name} in {world} shards: worst {worst:.3e}, {ncancel} judged against ||S||")
    assert ok, worst
