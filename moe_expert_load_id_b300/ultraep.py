"""Python binding of libultraep_b300.so (the sm_103a C ABI declared in include/ultraep.h).

Argument marshalling only: every step runs in the library's CUDA kernels.
Tensors are torch CUDA tensors (torch provides device memory and streams);
each call enqueues on the current torch stream unless ``stream`` is given and
raises ``EpError`` when the library returns a non-zero status.

Importing this module fails with ImportError when the library has not been
built (``python -m moe_expert_load_id_b300.build``); there is no fallback.
"""
import ctypes
import os
from dataclasses import dataclass

import torch

_LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libultraep_b300.so")
if not os.path.exists(_LIB_PATH):
    raise ImportError(f"{_LIB_PATH} is missing: build it with python -m moe_expert_load_id_b300.build")
_lib = ctypes.CDLL(_LIB_PATH)

EP_OK, EP_ERR_INVAL, EP_ERR_ITER_LIMIT, EP_ERR_BAD_ID, EP_ERR_WORKSPACE, EP_ERR_CUDA = range(6)
EP_DEV_BAD_ID, EP_DEV_QUOTA_OVERFLOW, EP_DEV_ROW_RANGE, EP_DEV_COPY_TIMEOUT = 1, 2, 4, 8
EP_DEV_COUNTS_MISMATCH, EP_DEV_COPY_UNDRAINED = 16, 32
EP_PLAN_MAX_ITERS = 1 << 16
EP_PLAN_SKIP, EP_PLAN_RELEASE = 1, 2
EP_COUNT_NOALLOC_SCRATCH_BYTES = 64 << 10

EXPORTS = ("ep_count_workspace_bytes", "ep_count", "ep_count_noalloc", "ep_plan", "ep_plan_ex",
           "ep_reroute",
           "ep_balance", "ep_permute", "ep_unpermute", "ep_combine", "ep_stage", "ep_status_str")


class _Domain(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("E", ctypes.c_int32), ("S", ctypes.c_int32),
                ("k", ctypes.c_int32)]


@dataclass(frozen=True)
class Domain:
    """Simulated EP domain: R ranks, E logical experts, S spare slots per rank, top-k k."""
    R: int
    E: int
    S: int
    k: int

    @property
    def H(self):
        return self.E // self.R

    @property
    def P(self):
        return self.R * (self.H + self.S)

    def c(self):
        return _Domain(self.R, self.E, self.S, self.k)


class EpError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__(f"{fn}: {ep_status_str(status)}")
        self.status = status


_vp = ctypes.c_void_p
_i32, _i64, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
_DP = ctypes.POINTER(_Domain)
_lib.ep_count_workspace_bytes.restype = _sz
_lib.ep_count_workspace_bytes.argtypes = [_DP, _i64, _i32]
_lib.ep_count.restype = ctypes.c_int
_lib.ep_count.argtypes = [_DP, _vp, _i64, _i32, _vp, _vp, _vp, _vp, _sz, _vp]
_lib.ep_count_noalloc.restype = ctypes.c_int
_lib.ep_count_noalloc.argtypes = [_DP, _vp, _i64, _i32, _vp, _vp, _vp, _vp]
_lib.ep_plan.restype = ctypes.c_int
_lib.ep_plan.argtypes = [_DP, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]
_lib.ep_plan_ex.restype = ctypes.c_int
_lib.ep_plan_ex.argtypes = [_DP, _vp, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                            _vp]
_lib.ep_reroute.restype = ctypes.c_int
_lib.ep_reroute.argtypes = [_DP, _vp, _i64, _i32, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]


class _BalanceOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "counts", "counts_src", "quota", "slot_expert", "rank_load", "inst_ptr", "inst_id",
        "inst_cum", "n_iter", "inst_status", "dst_row", "src_slot", "inst_offset")]


_lib.ep_balance.restype = ctypes.c_int
_lib.ep_balance.argtypes = [_DP, _vp, _i64, _i32, _i32, ctypes.POINTER(_BalanceOut), _vp, _vp,
                            _sz, _vp]
_lib.ep_permute.restype = ctypes.c_int
_lib.ep_permute.argtypes = [_vp, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp]
_lib.ep_unpermute.restype = ctypes.c_int
_lib.ep_unpermute.argtypes = [_vp, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp]
_lib.ep_combine.restype = ctypes.c_int
_lib.ep_combine.argtypes = [_vp, _i64, _i32, _i32, _i32, _vp, _vp, _vp, _vp, _vp]
_lib.ep_stage.restype = ctypes.c_int
_lib.ep_stage.argtypes = [_DP, _i32, _vp, _i64, _vp, _vp, _vp, _vp, _vp]
_lib.ep_status_str.restype = ctypes.c_char_p
_lib.ep_status_str.argtypes = [ctypes.c_int]


def ep_status_str(status: int) -> str:
    return _lib.ep_status_str(int(status)).decode()


def _ptr(t):
    return None if t is None else t.data_ptr()


def _stream(stream):
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _check(fn, status):
    if status != EP_OK:
        raise EpError(fn, status)


def _shape_ids(topk_ids, k):
    if topk_ids.dim() == 2:
        return 1, topk_ids.shape[0]
    if topk_ids.dim() != 3 or topk_ids.shape[2] != k:
        raise ValueError("topk_ids must be [T, k] or [n_inst, T, k]")
    return topk_ids.shape[0], topk_ids.shape[1]


def ep_count_workspace_bytes(dom: Domain, T: int, n_inst: int) -> int:
    return int(_lib.ep_count_workspace_bytes(ctypes.byref(dom.c()), T, n_inst))


def ep_count(dom, topk_ids, counts, counts_src, dev_status, workspace, stream=None):
    n_inst, T = _shape_ids(topk_ids, dom.k)
    _check("ep_count", _lib.ep_count(ctypes.byref(dom.c()), _ptr(topk_ids), T, n_inst,
                                     _ptr(counts), _ptr(counts_src), _ptr(dev_status),
                                     _ptr(workspace), workspace.numel() * workspace.element_size(),
                                     _stream(stream)))


def ep_count_noalloc(dom, topk_ids, counts, counts_src, dev_status, stream=None):
    """ep_count with the library's own fixed scratch array instead of a workspace,
    for callers that cannot allocate device memory (see include/ultraep.h)."""
    n_inst, T = _shape_ids(topk_ids, dom.k)
    _check("ep_count_noalloc", _lib.ep_count_noalloc(ctypes.byref(dom.c()), _ptr(topk_ids), T,
                                                     n_inst, _ptr(counts), _ptr(counts_src),
                                                     _ptr(dev_status), _stream(stream)))


def ep_plan(dom, counts, quota, slot_expert, rank_load, inst_ptr, inst_id, inst_cum, n_iter,
            inst_status, max_iters=0, stream=None):
    n_inst = counts.numel() // dom.E
    _check("ep_plan", _lib.ep_plan(ctypes.byref(dom.c()), _ptr(counts), n_inst, max_iters,
                                   _ptr(quota),
                                   _ptr(slot_expert), _ptr(rank_load), _ptr(inst_ptr),
                                   _ptr(inst_id), _ptr(inst_cum), _ptr(n_iter),
                                   _ptr(inst_status), _stream(stream)))


def ep_plan_ex(dom, counts, flags, quota, slot_expert, rank_load, inst_ptr, inst_id, inst_cum,
               n_iter, inst_status, max_iters=0, stream=None):
    """ep_plan with rule variants: flags = EP_PLAN_SKIP | EP_PLAN_RELEASE (0: ep_plan)."""
    n_inst = counts.numel() // dom.E
    _check("ep_plan_ex", _lib.ep_plan_ex(ctypes.byref(dom.c()), _ptr(counts), n_inst, max_iters,
                                         flags, _ptr(quota), _ptr(slot_expert), _ptr(rank_load),
                                         _ptr(inst_ptr), _ptr(inst_id), _ptr(inst_cum),
                                         _ptr(n_iter), _ptr(inst_status), _stream(stream)))


def ep_reroute(dom, topk_ids, counts_src, quota, inst_ptr, inst_id, inst_cum, dst_row, src_slot,
               inst_offset, dev_status, stream=None):
    n_inst, T = _shape_ids(topk_ids, dom.k)
    _check("ep_reroute", _lib.ep_reroute(ctypes.byref(dom.c()), _ptr(topk_ids), T, n_inst,
                                         _ptr(counts_src), _ptr(quota), _ptr(inst_ptr),
                                         _ptr(inst_id), _ptr(inst_cum), _ptr(dst_row),
                                         _ptr(src_slot), _ptr(inst_offset), _ptr(dev_status),
                                         _stream(stream)))


def ep_balance(dom, topk_ids, out, dev_status, workspace, max_iters=0, stream=None):
    """count -> plan -> reroute in one call (three chained launches).  ``out``
    has the attributes named like the fields of ep_balance_out_t (a Buffers
    object does); ``out.src_slot`` may be None."""
    n_inst, T = _shape_ids(topk_ids, dom.k)
    o = _BalanceOut(*[_ptr(getattr(out, n)) for n, _ in _BalanceOut._fields_])
    _check("ep_balance", _lib.ep_balance(ctypes.byref(dom.c()), _ptr(topk_ids), T, n_inst,
                                         max_iters, ctypes.byref(o), _ptr(dev_status),
                                         _ptr(workspace),
                                         workspace.numel() * workspace.element_size(),
                                         _stream(stream)))


def _rows(x, k):
    if x.dim() == 2:
        return 1, x.shape[0], x.shape[1]
    return x.shape[0], x.shape[1], x.shape[2]


def ep_permute(hidden, k, dst_row, out, dev_status=None, stream=None):
    """hidden [T, Hd] or [n_inst, T, Hd] bf16 -> out [.., T*k, Hd] bf16."""
    n_inst, T, Hd = _rows(hidden, k)
    _check("ep_permute", _lib.ep_permute(_ptr(hidden), T, k, Hd, n_inst, _ptr(dst_row),
                                         _ptr(out), _ptr(dev_status), _stream(stream)))


def ep_unpermute(grouped, T, k, dst_row, y, dev_status=None, stream=None):
    """grouped [T*k, Hd] or [n_inst, T*k, Hd] bf16 -> y [.., T, k, Hd] bf16."""
    Hd = grouped.shape[-1]
    n_inst = grouped.shape[0] if grouped.dim() == 3 else 1
    _check("ep_unpermute", _lib.ep_unpermute(_ptr(grouped), T, k, Hd, n_inst, _ptr(dst_row),
                                             _ptr(y), _ptr(dev_status), _stream(stream)))


def ep_combine(grouped, T, k, dst_row, weights, y, dev_status=None, stream=None):
    """grouped [T*k, Hd] or [n_inst, T*k, Hd] bf16, weights [.., T, k] float32 ->
    y [.., T, Hd] bf16: the gate-weighted sum of each token's k expert rows."""
    Hd = grouped.shape[-1]
    n_inst = grouped.shape[0] if grouped.dim() == 3 else 1
    _check("ep_combine", _lib.ep_combine(_ptr(grouped), T, k, Hd, n_inst, _ptr(dst_row),
                                         _ptr(weights), _ptr(y), _ptr(dev_status),
                                         _stream(stream)))


def ep_stage(dom, expert_w, slot_expert, slot_w, prev_slot_expert=None, dev_status=None,
             stream=None):
    """expert_w [E, bytes] or [n_inst, E, bytes] (any dtype, bytes a multiple of
    16) -> slot_w [.., R, S, bytes]: each filled spare slot gets its expert's
    weights (slots already holding their expert are skipped when
    prev_slot_expert is given)."""
    n_inst = slot_expert.numel() // max(1, dom.R * dom.S) if dom.S else 0
    E = dom.E
    nbytes = expert_w.numel() * expert_w.element_size() // max(1, n_inst * E) if n_inst else 0
    _check("ep_stage", _lib.ep_stage(ctypes.byref(dom.c()), n_inst, _ptr(expert_w), nbytes,
                                     _ptr(slot_expert), _ptr(prev_slot_expert), _ptr(slot_w),
                                     _ptr(dev_status), _stream(stream)))


# ------------------------------------------------------------------ buffers
class Buffers:
    """Device buffers of the path for n_inst instances of T tokens (torch only
    allocates; the library never does)."""

    def __init__(self, dom: Domain, T: int, n_inst: int = 1, Hd: int = 0, device="cuda",
                 src_slot: bool = False):
        i32 = dict(dtype=torch.int32, device=device)
        N = T * dom.k
        self.dom, self.T, self.n_inst, self.Hd = dom, T, n_inst, Hd
        self.counts = torch.empty((n_inst, dom.E), **i32)
        self.counts_src = torch.empty((n_inst, dom.R, dom.E), **i32)
        self.dev_status = torch.zeros((1,), **i32)
        ws = ep_count_workspace_bytes(dom, T, n_inst)
        self.workspace = torch.zeros((max(ws, 16) // 4,), **i32)
        self.quota = torch.empty((n_inst, dom.P), **i32)
        self.slot_expert = torch.empty((n_inst, dom.R, dom.S), **i32)
        self.rank_load = torch.empty((n_inst, dom.R), **i32)
        self.inst_ptr = torch.empty((n_inst, dom.E + 1), **i32)
        self.inst_id = torch.full((n_inst, dom.E + dom.R * dom.S), -1, **i32)
        self.inst_cum = torch.full((n_inst, dom.E + dom.R * dom.S), -1, **i32)
        self.n_iter = torch.empty((n_inst,), **i32)
        self.inst_status = torch.empty((n_inst,), **i32)
        self.dst_row = torch.empty((n_inst, N), **i32)
        self.src_slot = torch.full((n_inst, N), -1, **i32) if src_slot else None
        self.inst_offset = torch.empty((n_inst, dom.P + 1), **i32)
        self.grouped = (torch.empty((n_inst, N, Hd), dtype=torch.bfloat16, device=device)
                        if Hd else None)

    def count(self, topk_ids, stream=None):
        ep_count(self.dom, topk_ids, self.counts, self.counts_src, self.dev_status,
                 self.workspace, stream)

    def plan(self, max_iters=0, stream=None, flags=0):
        if flags:
            ep_plan_ex(self.dom, self.counts, flags, self.quota, self.slot_expert,
                       self.rank_load, self.inst_ptr, self.inst_id, self.inst_cum, self.n_iter,
                       self.inst_status, max_iters, stream)
            return
        ep_plan(self.dom, self.counts, self.quota, self.slot_expert, self.rank_load,
                self.inst_ptr, self.inst_id, self.inst_cum, self.n_iter, self.inst_status,
                max_iters, stream)

    def reroute(self, topk_ids, stream=None):
        ep_reroute(self.dom, topk_ids, self.counts_src, self.quota, self.inst_ptr, self.inst_id,
                   self.inst_cum, self.dst_row, self.src_slot, self.inst_offset,
                   self.dev_status, stream)

    def permute(self, hidden, stream=None):
        ep_permute(hidden, self.dom.k, self.dst_row, self.grouped, self.dev_status, stream)

    def balance_fused(self, topk_ids, max_iters=0, stream=None):
        """count -> plan -> reroute through the single chained ep_balance call."""
        ep_balance(self.dom, topk_ids, self, self.dev_status, self.workspace, max_iters, stream)

    def balance(self, topk_ids, hidden=None, stream=None):
        """count -> plan -> reroute (-> permute) for one batch of instances."""
        self.count(topk_ids, stream)
        self.plan(stream=stream)
        self.reroute(topk_ids, stream)
        if hidden is not None:
            self.permute(hidden, stream)
