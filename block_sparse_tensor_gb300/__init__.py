"""Python binding of libbs.so, the coalesced block-sparse contraction library.

Argument marshalling only: every step of a contraction runs in the library's
CUDA kernels.  PyTorch supplies device memory and streams; tensors are passed
by data pointer.  The library must be built first (`build.build()`); importing
the package without it raises ImportError, and there is no CPU fallback.

Names follow the C ABI in include/bs.h: `Layout` wraps bs_layout_create,
`Plan` wraps bs_plan_create, `contract` wraps bs_contract.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libbs.so")

F64, BF16_F32 = 0, 1
AXIS_AUTO, AXIS_CONTRACTION, AXIS_FREE, AXIS_NONE = 0, 1, 2, 3
DEBUG_WITHHOLD_COPY, DEBUG_MERGE_UNCHECKED = 1, 2
ERR_HOLE = 10
PACK_AUTO, PACK_NEVER, PACK_ALWAYS = 0, 1, 2
LAYOUT_FLAGS = {"blockrow": 0, "rowpanel": 1, "colpanel": 2, "charge_sorted": 4, "align16": 8, "align64": 16}
STATUS = {0: "ok", 1: "invalid argument", 2: "shape mismatch", 3: "unsupported", 4: "out of memory",
          5: "CUDA error", 6: "device wait timed out", 7: "misaligned", 8: "device check failed",
          9: "size overflow", 10: "group is not a hole-free view of its blocks"}

EXPORTED = ["bs_layout_create", "bs_layout_query", "bs_layout_blocks", "bs_layout_destroy",
            "bs_plan_options_default", "bs_plan_create", "bs_plan_c_layout", "bs_plan_stats_get",
            "bs_plan_groups", "bs_plan_triples", "bs_contract", "bs_contract_host",
            "bs_contract_uncoalesced", "bs_plan_last_device_error", "bs_plan_destroy",
            "bs_status_string", "bs_version", "bs_calibrate", "bs_contract_noalloc",
            "bs_plan_check_groups", "bs_plan_create_into", "bs_plan_profile", "bs_plan_create_shard",
            "bs_plan_operand_blocks", "bs_calibration_apply", "bs_contract_checked", "bs_plan_gather_segments"]


class BsError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)} ({code})")
        self.code = code


class AxisDesc(ctypes.Structure):
    _fields_ = [("n", ctypes.c_int32), ("q_u1", ctypes.c_void_p), ("q_z2", ctypes.c_void_p),
                ("dim", ctypes.c_void_p)]


class Rule(ctypes.Structure):
    _fields_ = [("dq_min", ctypes.c_int32), ("dq_max", ctypes.c_int32), ("z2", ctypes.c_int32)]


class BlockInfo(ctypes.Structure):
    _fields_ = [("row", ctypes.c_int32), ("col", ctypes.c_int32), ("offset", ctypes.c_int64),
                ("rows", ctypes.c_int32), ("cols", ctypes.c_int32), ("ld", ctypes.c_int64)]


class PlanOptions(ctypes.Structure):
    _fields_ = [("axis_policy", ctypes.c_int32), ("pack_policy", ctypes.c_int32),
                ("c_layout_flags", ctypes.c_uint32), ("merge_rows", ctypes.c_int32),
                ("host_only", ctypes.c_int32), ("ctas_per_sm", ctypes.c_int32),
                ("t_launch_us", ctypes.c_double), ("t_task_us", ctypes.c_double),
                ("t_segment_us", ctypes.c_double), ("pack_gbs", ctypes.c_double),
                ("fp64_gflops", ctypes.c_double), ("atomic_penalty", ctypes.c_double),
                ("wait_timeout_ms", ctypes.c_int32), ("debug_flags", ctypes.c_int32),
                ("bucket_pad", ctypes.c_int32), ("profile", ctypes.c_int32), ("tail_split_k", ctypes.c_int32),
                ("reserved", ctypes.c_int32 * 3),
                ("t_fixed_us", ctypes.c_double), ("fp64_tail_gflops", ctypes.c_double),
                ("fp64_general_gflops", ctypes.c_double), ("pack_fixed_us", ctypes.c_double),
                ("zero_gbs", ctypes.c_double), ("bf16_stage_us", ctypes.c_double), ("bf16_tile_us", ctypes.c_double),
                ("tile_k0", ctypes.c_double), ("reserved2", ctypes.c_double * 3)]


class PlanStats(ctypes.Structure):
    _fields_ = [("triples", ctypes.c_int64), ("c_blocks", ctypes.c_int64), ("groups", ctypes.c_int64),
                ("tasks", ctypes.c_int64), ("tile_tasks", ctypes.c_int64), ("tail_tasks", ctypes.c_int64),
                ("segments", ctypes.c_int64), ("packed_bytes", ctypes.c_int64),
                ("workspace_bytes", ctypes.c_int64), ("axis", ctypes.c_int32), ("packed_a", ctypes.c_int32),
                ("packed_b", ctypes.c_int32), ("launches", ctypes.c_int32), ("useful_flops", ctypes.c_double),
                ("useful_bytes", ctypes.c_double), ("executed_flops", ctypes.c_double),
                ("model_us", ctypes.c_double), ("model_us_alt", ctypes.c_double), ("plan_ms", ctypes.c_double)]


class PhaseTimes(ctypes.Structure):
    _fields_ = [("gather_ms", ctypes.c_double), ("zero_ms", ctypes.c_double), ("kernel_ms", ctypes.c_double),
                ("total_ms", ctypes.c_double), ("gather_bytes", ctypes.c_int64), ("reserved", ctypes.c_int64 * 3)]


class Calibration(ctypes.Structure):
    _fields_ = [("fp64_gflops", ctypes.c_double), ("fp64_gflops_quarter_warp", ctypes.c_double),
                ("launch_us", ctypes.c_double), ("copy_gbs", ctypes.c_double), ("sm_count", ctypes.c_int32),
                ("sm_id_bound", ctypes.c_int32), ("fp64_sm_mhz", ctypes.c_double),
                ("fp64_flop_per_clk_sm", ctypes.c_double), ("fp64_dmma_gflops", ctypes.c_double),
                ("dmma_flop_per_clk_sm", ctypes.c_double), ("t_fixed_us", ctypes.c_double),
                ("tile_gflops", ctypes.c_double), ("tail_gflops", ctypes.c_double), ("general_gflops", ctypes.c_double),
                ("pack_gbs", ctypes.c_double), ("pack_fixed_us", ctypes.c_double), ("zero_gbs", ctypes.c_double),
                ("bf16_stage_us", ctypes.c_double), ("bf16_tile_us", ctypes.c_double), ("tile_k0", ctypes.c_double),
                ("atomic_factor", ctypes.c_double), ("reserved", ctypes.c_double * 5)]


def _load(path: str = LIB_PATH):
    if not os.path.exists(path):
        raise ImportError(f"libbs.so is not built ({path}); run block_sparse_tensor_gb300.build.build()")
    L = ctypes.CDLL(path)
    P, i32, i64, u32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_uint32
    st = ctypes.c_int
    sig = {
        "bs_layout_create": (st, [P, P, P, u32, i32, P]),
        "bs_layout_query": (st, [P, P, P]),
        "bs_layout_blocks": (st, [P, P]),
        "bs_layout_destroy": (None, [P]),
        "bs_plan_options_default": (None, [P]),
        "bs_plan_create": (st, [P, P, i32, P, P]),
        "bs_plan_c_layout": (P, [P]),
        "bs_plan_stats_get": (st, [P, P]),
        "bs_plan_groups": (st, [P, P, P]),
        "bs_plan_triples": (st, [P, P, P, P, P]),
        "bs_contract": (st, [P, P, P, P, P]),
        "bs_contract_host": (st, [P, P, P, P, P]),
        "bs_contract_uncoalesced": (st, [P, P, P, P, P]),
        "bs_plan_last_device_error": (st, [P, P]),
        "bs_plan_destroy": (None, [P]),
        "bs_status_string": (ctypes.c_char_p, [st]),
        "bs_version": (ctypes.c_char_p, []),
        "bs_calibrate": (st, [P, P]),
        "bs_contract_noalloc": (st, [P, P, P, P, P]),
        "bs_plan_check_groups": (st, [P, P]),
        "bs_plan_create_into": (st, [P, P, P, i32, P, P]),
        "bs_plan_profile": (st, [P, P]),
        "bs_plan_create_shard": (st, [P, P, i32, P, i32, i32, P]),
        "bs_plan_operand_blocks": (st, [P, i32, P, P]),
        "bs_calibration_apply": (None, [P, P]),
        "bs_contract_checked": (st, [P, P, i64, P, i64, P, i64, P]),
        "bs_plan_gather_segments": (st, [P, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        f = getattr(L, name)
        f.restype = res
        f.argtypes = args
    return L


lib = _load()


def _check(code: int, where: str):
    if code != 0:
        raise BsError(code, where)


def parse_flags(flags) -> int:
    if isinstance(flags, (int, np.integer)):
        return int(flags)
    out = 0
    for part in str(flags).split("|"):
        part = part.strip()
        if part:
            out |= LAYOUT_FLAGS[part]
    return out


class _AxisArrays:
    """Keeps the numpy arrays of one axis alive while the C call reads them."""

    def __init__(self, ax):
        self.q = np.ascontiguousarray(ax.q, dtype=np.int32)
        self.d = np.ascontiguousarray(ax.d, dtype=np.int32)
        p = getattr(ax, "p", None)
        self.p = None if p is None else np.ascontiguousarray(p, dtype=np.uint8)
        self.desc = AxisDesc(len(self.q), self.q.ctypes.data, None if self.p is None else self.p.ctypes.data,
                             self.d.ctypes.data)


def _ptr(x) -> Optional[int]:
    """Device or host address of a torch tensor, numpy array or plain int."""
    if x is None:
        return None
    if isinstance(x, int):
        return x
    if isinstance(x, np.ndarray):
        return x.ctypes.data
    return x.data_ptr()


def _stream(s) -> Optional[int]:
    if s is None:
        return None
    if isinstance(s, int):
        return s
    return s.cuda_stream


class Layout:
    """A sector layout (bs_layout): populated blocks and their (offset, ld) views."""

    def __init__(self, rows, cols, rule, flags="blockrow", elem_bytes=8, _handle=None, _owner=None):
        self._owner = _owner
        if _handle is not None:
            self.h = _handle
            self._own = False
            return
        r, c = _AxisArrays(rows), _AxisArrays(cols)
        ru = Rule(int(rule.dq_min), int(rule.dq_max), 1 if getattr(rule, "z2", False) else 0)
        h = ctypes.c_void_p()
        _check(lib.bs_layout_create(ctypes.byref(r.desc), ctypes.byref(c.desc), ctypes.byref(ru),
                                    parse_flags(flags), int(elem_bytes), ctypes.byref(h)), "bs_layout_create")
        self.h = h
        self._own = True

    def query(self):
        nb, ne = ctypes.c_int64(), ctypes.c_int64()
        _check(lib.bs_layout_query(self.h, ctypes.byref(nb), ctypes.byref(ne)), "bs_layout_query")
        return nb.value, ne.value

    @property
    def nblocks(self) -> int:
        return self.query()[0]

    @property
    def nelems(self) -> int:
        return self.query()[1]

    def blocks(self) -> np.ndarray:
        """Block table in storage order: int64 array of (row, col, offset, rows, cols, ld)."""
        nb = self.nblocks
        arr = (BlockInfo * max(nb, 1))()
        _check(lib.bs_layout_blocks(self.h, arr), "bs_layout_blocks")
        out = np.empty((nb, 6), np.int64)
        for t in range(nb):
            b = arr[t]
            out[t] = (b.row, b.col, b.offset, b.rows, b.cols, b.ld)
        return out

    def element_index(self, blocks: Optional[np.ndarray] = None) -> np.ndarray:
        """Buffer index of every element of every block, block after block in the
        given (default: storage) order, row-major inside a block.  Filling
        buf[layout.element_index()] = values places block-concatenated values."""
        b = self.blocks() if blocks is None else blocks
        if len(b) == 0:
            return np.zeros(0, np.int64)
        sizes = b[:, 3] * b[:, 4]
        starts = np.concatenate([[0], np.cumsum(sizes)[:-1]])
        rep = np.repeat(np.arange(len(b)), sizes)
        local = np.arange(int(sizes.sum()), dtype=np.int64) - starts[rep]
        c = b[rep, 4]
        return b[rep, 2] + (local // c) * b[rep, 5] + local % c

    def __del__(self):
        if getattr(self, "_own", False) and self.h:
            lib.bs_layout_destroy(self.h)
            self.h = None


def plan_options(**kw) -> PlanOptions:
    o = PlanOptions()
    lib.bs_plan_options_default(ctypes.byref(o))
    for k, v in kw.items():
        if k == "c_layout_flags":
            v = parse_flags(v)
        setattr(o, k, v)
    return o


class Plan:
    """A contraction plan (bs_plan) for C = A B."""

    def __init__(self, A: Layout, B: Layout, dtype: int = F64, C: Layout = None, shard=None, **options):
        """With C, plan onto that existing C layout (bs_plan_create_into); with
        shard = (rank, world), plan shard `rank` of `world` (bs_plan_create_shard)."""
        self.opts = plan_options(**options)
        h = ctypes.c_void_p()
        if shard is not None:
            _check(lib.bs_plan_create_shard(A.h, B.h, int(dtype), ctypes.byref(self.opts), int(shard[0]), int(shard[1]),
                                            ctypes.byref(h)), "bs_plan_create_shard")
        elif C is None:
            _check(lib.bs_plan_create(A.h, B.h, int(dtype), ctypes.byref(self.opts), ctypes.byref(h)), "bs_plan_create")
        else:
            _check(lib.bs_plan_create_into(A.h, B.h, C.h, int(dtype), ctypes.byref(self.opts), ctypes.byref(h)),
                   "bs_plan_create_into")
        self.h = h
        self.dtype = dtype
        self.c_layout = Layout(None, None, None, _handle=lib.bs_plan_c_layout(h), _owner=self)

    def stats(self) -> dict:
        s = PlanStats()
        _check(lib.bs_plan_stats_get(self.h, ctypes.byref(s)), "bs_plan_stats_get")
        return {name: getattr(s, name) for name, _ in PlanStats._fields_}

    def groups(self) -> np.ndarray:
        n = ctypes.c_int64()
        _check(lib.bs_plan_groups(self.h, ctypes.byref(n), None), "bs_plan_groups")
        out = np.zeros((max(n.value, 1), 8), np.int64)
        _check(lib.bs_plan_groups(self.h, ctypes.byref(n), out.ctypes.data), "bs_plan_groups")
        return out[:n.value]

    def gather_segments(self):
        """(segments, pieces) of bs_plan_gather_segments: an (n, 5) and an (m, 6) int64 array."""
        ns, npc = ctypes.c_int64(), ctypes.c_int64()
        _check(lib.bs_plan_gather_segments(self.h, ctypes.byref(ns), ctypes.byref(npc), None, None),
               "bs_plan_gather_segments")
        segs = np.zeros((max(ns.value, 1), 5), np.int64)
        pcs = np.zeros((max(npc.value, 1), 6), np.int64)
        _check(lib.bs_plan_gather_segments(self.h, ctypes.byref(ns), ctypes.byref(npc), segs.ctypes.data,
                                           pcs.ctypes.data), "bs_plan_gather_segments")
        return segs[:ns.value], pcs[:npc.value]

    def check_groups(self):
        """(status, first failing group or -1) of bs_plan_check_groups."""
        bad = ctypes.c_int64()
        status = lib.bs_plan_check_groups(self.h, ctypes.byref(bad))
        return status, bad.value

    def triples(self):
        """(group_ptr, triples) with triples an (n, 3) int32 array of (i, k, j)."""
        nt, ng = ctypes.c_int64(), ctypes.c_int64()
        _check(lib.bs_plan_triples(self.h, ctypes.byref(nt), ctypes.byref(ng), None, None), "bs_plan_triples")
        ptr = np.zeros(ng.value + 1, np.int64)
        tr = np.zeros((max(nt.value, 1), 3), np.int32)
        _check(lib.bs_plan_triples(self.h, ctypes.byref(nt), ctypes.byref(ng), ptr.ctypes.data, tr.ctypes.data),
               "bs_plan_triples")
        return ptr, tr[:nt.value]

    def operand_blocks(self, operand: int) -> np.ndarray:
        """Indices (storage order) of the A (0), B (1) or C (2) blocks this plan uses."""
        n = ctypes.c_int64()
        _check(lib.bs_plan_operand_blocks(self.h, int(operand), ctypes.byref(n), None), "bs_plan_operand_blocks")
        out = np.zeros(max(n.value, 1), np.int32)
        _check(lib.bs_plan_operand_blocks(self.h, int(operand), ctypes.byref(n), out.ctypes.data),
               "bs_plan_operand_blocks")
        return out[:n.value]

    def profile(self) -> dict:
        """Phase times (ms) of the last contraction of a plan built with profile=1."""
        t = PhaseTimes()
        _check(lib.bs_plan_profile(self.h, ctypes.byref(t)), "bs_plan_profile")
        return {name: getattr(t, name) for name, _ in PhaseTimes._fields_ if name != "reserved"}

    def __del__(self):
        if getattr(self, "h", None):
            lib.bs_plan_destroy(self.h)
            self.h = None


def contract(plan: Plan, A, B, C, stream=None):
    """Enqueue C = A B on `stream` (torch.cuda.Stream, raw handle or None)."""
    _check(lib.bs_contract(plan.h, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "bs_contract")


def contract_checked(plan: Plan, A, B, C, nA=None, nB=None, nC=None, stream=None):
    """bs_contract_checked: every access tested against the buffers' element counts
    (default: the tensors' own numel).  A violation reads as BS_ERR_DEVICE from
    last_device_error, or is raised at once when the host finds it."""
    n = lambda x, v: int(v) if v is not None else int(x.numel())  # noqa: E731
    _check(lib.bs_contract_checked(plan.h, _ptr(A), n(A, nA), _ptr(B), n(B, nB), _ptr(C), n(C, nC), _stream(stream)),
           "bs_contract_checked")


def contract_host(plan: Plan, A, B, C, stream=None):
    """C = A B on host buffers (numpy arrays or CPU tensors; pinned is fastest); synchronous."""
    _check(lib.bs_contract_host(plan.h, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "bs_contract_host")


def contract_uncoalesced(plan: Plan, A, B, C, stream=None):
    """The one-launch-per-triple control."""
    _check(lib.bs_contract_uncoalesced(plan.h, _ptr(A), _ptr(B), _ptr(C), _stream(stream)),
           "bs_contract_uncoalesced")


def contract_noalloc(plan: Plan, A, B, C, stream=None):
    """C = A B without any device allocation (FP64 plans; the plan may be host_only).

    For callers that cannot allocate device memory: the plan's tables and
    workspace go into a fixed 16 MiB device array inside the library, shared by
    every call, so calls must not overlap on the GPU."""
    _check(lib.bs_contract_noalloc(plan.h, _ptr(A), _ptr(B), _ptr(C), _stream(stream)), "bs_contract_noalloc")


def last_device_error(plan: Plan, stream=None) -> int:
    """Synchronize and return (and clear) the device status as a bs_status code."""
    return int(lib.bs_plan_last_device_error(plan.h, _stream(stream)))


def calibrate(stream=None) -> dict:
    """Measure the cost-model constants on the current device (bs_calibrate)."""
    c = Calibration()
    _check(lib.bs_calibrate(ctypes.byref(c), _stream(stream)), "bs_calibrate")
    return {name: getattr(c, name) for name, _ in Calibration._fields_ if not name.startswith("reserved")}


def calibrated_options(cal: dict) -> dict:
    """Planner options carrying the cost-model constants of a calibration (bs_calibration_apply)."""
    c = Calibration()
    for name, _ in Calibration._fields_:
        if not name.startswith("reserved") and name in cal:
            setattr(c, name, cal[name])
    o = plan_options()
    lib.bs_calibration_apply(ctypes.byref(c), ctypes.byref(o))
    names = ("t_launch_us", "t_task_us", "t_segment_us", "pack_gbs", "fp64_gflops", "atomic_penalty", "t_fixed_us",
             "fp64_tail_gflops", "fp64_general_gflops", "pack_fixed_us", "zero_gbs", "bf16_stage_us", "bf16_tile_us",
             "tile_k0")
    return {n: getattr(o, n) for n in names if getattr(o, n) > 0}


def version() -> str:
    return lib.bs_version().decode()
