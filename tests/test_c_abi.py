"""The C ABI from a plain C program: tests/c_abi/abi_check.c is compiled with gcc
against include/bs.h alone and linked with libbs.so.  On the host it builds
layouts and a host-only plan and checks them against the oracle's counts; on a
GPU it also runs bs_contract_host on host buffers and compares every C element
with the oracle's (integer inputs, so the comparison is exact)."""
import os
import shutil
import struct
import subprocess
import tempfile

import numpy as np
import pytest

import bsgen
import oracle

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PKG = os.path.join(ROOT, "block_sparse_tensor_gb300")
SRC = os.path.join(ROOT, "tests", "c_abi", "abi_check.c")
FLAGS = {"blockrow": 0, "rowpanel": 1, "colpanel": 2, "charge_sorted": 4, "align16": 8, "align64": 16}


def _flags(name):
    return sum(FLAGS[p] for p in name.split("|") if p)


@pytest.fixture(scope="module")
def abi_check():
    pytest.importorskip("block_sparse_tensor_gb300")   # libbs.so must be built
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    d = tempfile.mkdtemp()
    exe = os.path.join(d, "abi_check")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-O1", "-I", os.path.join(ROOT, "include"),
                    SRC, "-L", PKG, "-lbs", "-Wl,-rpath," + PKG, "-o", exe], check=True)
    yield exe, d
    shutil.rmtree(d, ignore_errors=True)


def _write_problem(path, w, la, lb, lc):
    pr = oracle.problem(w, la, lb, lc)
    C, _ = oracle.contract(pr)
    triples = int((pr.ma.astype(np.int64) @ pr.mb.astype(np.int64)).sum())
    with open(path, "wb") as f:
        f.write(struct.pack("<3i", w.rows.n, w.inner.n, w.cols.n))
        for ax in (w.rows, w.inner, w.cols):
            f.write(np.asarray(ax.q, "<i4").tobytes())
            f.write(np.asarray(ax.d, "<i4").tobytes())
        for r in (w.rule_a, w.rule_b):
            f.write(struct.pack("<3i", r.dq_min, r.dq_max, 1 if r.z2 else 0))
        f.write(struct.pack("<3I", _flags(la), _flags(lb), _flags(lc)))
        f.write(struct.pack("<q", triples))
        for v in (pr.A, pr.B, C):
            f.write(struct.pack("<q", len(v)))
            f.write(np.asarray(v, "<f8").tobytes())


CASES = [(3, "rowpanel|charge_sorted", "colpanel|charge_sorted", "blockrow"),
         (5, "blockrow", "blockrow", "rowpanel|align16"),
         (9, "colpanel", "rowpanel", "colpanel|charge_sorted")]


@pytest.mark.parametrize("seed,la,lb,lc", CASES)
def test_c_program_builds_layouts_and_plans(abi_check, seed, la, lb, lc):
    exe, d = abi_check
    w = bsgen.tiny_random(seed, values="int3", z2=False, max_dim=12)
    path = os.path.join(d, f"p{seed}.bin")
    _write_problem(path, w, la, lb, lc)
    r = subprocess.run([exe, "host", path], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert "abi_check host ok" in r.stdout


@pytest.mark.gpu
@pytest.mark.parametrize("seed,la,lb,lc", CASES)
def test_c_program_contracts_through_the_abi(abi_check, seed, la, lb, lc):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    exe, d = abi_check
    w = bsgen.tiny_random(seed, values="int3", z2=False, max_dim=12)
    path = os.path.join(d, f"g{seed}.bin")
    _write_problem(path, w, la, lb, lc)
    r = subprocess.run([exe, "device", path], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert "abi_check device ok" in r.stdout
