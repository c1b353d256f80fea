"""The CPU oracle of the UltraEP balancing hot path (numpy view of oracle/liboracle.so).

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's CPU
baseline leg may import this package; the product path never does.  It shares
no code with the CUDA library and imports nothing from it.

Every function here is argument marshalling around the plain C definitions in
ultraep_oracle.c, which cite the pages they follow.
"""
import contextlib
import ctypes
import os

import numpy as np

from . import build as _build

ORACLE_OK = 0
ORACLE_ITER_LIMIT = 2
PLAN_MAX_ITERS = 1 << 16

_lib = None


def lib():
    global _lib
    if _lib is None:
        _lib = _load(_build.build())
    return _lib


@contextlib.contextmanager
def using_library(path):
    """Run the wrappers against another build of the oracle source (used by the
    test that plants mistakes in copies of the oracle)."""
    global _lib
    old = _lib
    _lib = _load(path)
    try:
        yield
    finally:
        _lib = old


def _load(path):
    L = ctypes.CDLL(path)
    i32p = ctypes.POINTER(ctypes.c_int32)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    L.oracle_count.restype = ctypes.c_int64
    L.oracle_count.argtypes = [i32p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                               ctypes.c_int32, i32p, i32p]
    L.oracle_plan.restype = ctypes.c_int
    L.oracle_plan.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                              ctypes.c_int32, i32p, i32p, i32p, i32p, i32p, i32p, i32p]
    L.oracle_plan_variant.restype = ctypes.c_int
    L.oracle_plan_variant.argtypes = [i32p, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                                      ctypes.c_int32, ctypes.c_int32, i32p, i32p, i32p, i32p,
                                      i32p, i32p, i32p]
    L.oracle_reroute.restype = None
    L.oracle_reroute.argtypes = [i32p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32, ctypes.c_int32, i32p, i32p, i32p, i32p,
                                 i32p, i32p, i32p]
    L.oracle_permute.restype = None
    L.oracle_permute.argtypes = [u16p, ctypes.c_int32, ctypes.c_int32, i32p,
                                 ctypes.c_int64, u16p]
    L.oracle_combine.restype = None
    L.oracle_combine.argtypes = [u16p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, i32p,
                                 ctypes.POINTER(ctypes.c_float), u16p]
    L.oracle_stage.restype = None
    L.oracle_stage.argtypes = [ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, i32p, i32p,
                               ctypes.c_int32, ctypes.c_int32, ctypes.c_void_p, i32p,
                               ctypes.POINTER(ctypes.c_int64)]
    L.oracle_unpermute.restype = None
    L.oracle_unpermute.argtypes = [u16p, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                   i32p, u16p]
    return L


def _p(a, ct):
    return a.ctypes.data_as(ctypes.POINTER(ct))


def _i32(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a


def count(ids, R, E):
    """ids: int32 [T, k].  Returns (counts[E], counts_src[R, E], n_invalid)."""
    ids = _i32(ids)
    T, k = ids.shape
    counts = np.zeros(E, np.int32)
    counts_src = np.zeros((R, E), np.int32)
    n_bad = lib().oracle_count(_p(ids, ctypes.c_int32), T, k, R, E,
                               _p(counts, ctypes.c_int32), _p(counts_src, ctypes.c_int32))
    return counts, counts_src, int(n_bad)


# planner variants: None = the base rule's own function; otherwise the flags of
# oracle_plan_variant (1: try the next candidate instead of stopping, 2: release
# replica slots whose quota reaches 0)
PLAN_VARIANTS = {"base": None, "base_flags": 0, "skip": 1, "release": 2, "skip+release": 3}


def plan(counts, R, E, S, max_iters=PLAN_MAX_ITERS, variant="base"):
    """counts: int32 [E].  Returns a dict with the plan outputs.  variant: a key
    of PLAN_VARIANTS."""
    counts = _i32(counts)
    H = E // R
    P = R * (H + S)
    quota = np.zeros(P, np.int32)
    slot_expert = np.zeros(R * S, np.int32)
    rank_load = np.zeros(R, np.int32)
    inst_ptr = np.zeros(E + 1, np.int32)
    inst_id = np.full(E + R * S, -1, np.int32)
    inst_cum = np.full(E + R * S, -1, np.int32)
    n_iter = ctypes.c_int32(0)
    flags = PLAN_VARIANTS[variant]
    if flags is None:
        fn = lib().oracle_plan
        args = (_p(counts, ctypes.c_int32), R, E, S, max_iters)
    else:
        fn = lib().oracle_plan_variant
        args = (_p(counts, ctypes.c_int32), R, E, S, max_iters, flags)
    st = fn(*args,
                           _p(quota, ctypes.c_int32), _p(slot_expert, ctypes.c_int32),
                           _p(rank_load, ctypes.c_int32), _p(inst_ptr, ctypes.c_int32),
                           _p(inst_id, ctypes.c_int32), _p(inst_cum, ctypes.c_int32),
                           ctypes.byref(n_iter))
    return dict(quota=quota, slot_expert=slot_expert.reshape(R, S), rank_load=rank_load,
                inst_ptr=inst_ptr, inst_id=inst_id, inst_cum=inst_cum,
                n_iter=int(n_iter.value), status=int(st))


def reroute(ids, R, E, S, pl):
    """ids: int32 [T, k]; pl: a plan dict.  Returns (dst_row[N], src_slot[N], inst_offset[P+1])."""
    ids = _i32(ids)
    T, k = ids.shape
    N = T * k
    H = E // R
    P = R * (H + S)
    dst_row = np.zeros(N, np.int32)
    src_slot = np.full(N, -1, np.int32)
    inst_offset = np.zeros(P + 1, np.int32)
    q = _i32(pl["quota"])
    ip = _i32(pl["inst_ptr"])
    ii = _i32(pl["inst_id"])
    ic = _i32(pl["inst_cum"])
    lib().oracle_reroute(_p(ids, ctypes.c_int32), T, k, R, E, S, _p(q, ctypes.c_int32),
                         _p(ip, ctypes.c_int32), _p(ii, ctypes.c_int32), _p(ic, ctypes.c_int32),
                         _p(dst_row, ctypes.c_int32), _p(src_slot, ctypes.c_int32),
                         _p(inst_offset, ctypes.c_int32))
    return dst_row, src_slot, inst_offset


def permute(hidden_u16, k, src_slot, n_rows):
    """hidden_u16: uint16 [T, Hd] (bf16 bit patterns).  Returns uint16 [n_rows, Hd]."""
    hidden_u16 = np.ascontiguousarray(hidden_u16, dtype=np.uint16)
    Hd = hidden_u16.shape[1]
    src_slot = _i32(src_slot)
    out = np.zeros((n_rows, Hd), np.uint16)
    lib().oracle_permute(_p(hidden_u16, ctypes.c_uint16), k, Hd, _p(src_slot, ctypes.c_int32),
                         n_rows, _p(out, ctypes.c_uint16))
    return out


def unpermute(grouped_u16, T, k, dst_row):
    """grouped_u16: uint16 [rows, Hd].  Returns uint16 [T, k, Hd]."""
    grouped_u16 = np.ascontiguousarray(grouped_u16, dtype=np.uint16)
    Hd = grouped_u16.shape[1]
    dst_row = _i32(dst_row)
    y = np.zeros((T, k, Hd), np.uint16)
    lib().oracle_unpermute(_p(grouped_u16, ctypes.c_uint16), T, k, Hd,
                           _p(dst_row, ctypes.c_int32), _p(y, ctypes.c_uint16))
    return y


def combine(grouped_u16, T, k, dst_row, weights):
    """grouped_u16: uint16 [rows, Hd] (bf16 bits); dst_row int32 [T*k]; weights
    float32 [T, k].  Returns uint16 [T, Hd]: the gate-weighted sum of each
    token's k expert rows, float32 in ascending j, rounded to bf16."""
    grouped_u16 = np.ascontiguousarray(grouped_u16, dtype=np.uint16)
    Hd = grouped_u16.shape[1]
    dst_row = _i32(dst_row)
    w = np.ascontiguousarray(weights, dtype=np.float32)
    y = np.zeros((T, Hd), np.uint16)
    lib().oracle_combine(_p(grouped_u16, ctypes.c_uint16), T, k, Hd,
                         _p(dst_row, ctypes.c_int32), _p(w, ctypes.c_float),
                         _p(y, ctypes.c_uint16))
    return y


def stage(expert_w, slot_expert, R, S, slot_w, prev=None):
    """expert_w: uint8 [E, expert_bytes]; slot_expert int32 [R*S]; slot_w uint8
    [R*S, expert_bytes], updated in place (a copy is returned).  Returns
    (slot_w, n_copied, n_bad)."""
    expert_w = np.ascontiguousarray(expert_w, dtype=np.uint8)
    E, nb = expert_w.shape
    se = _i32(np.asarray(slot_expert).reshape(-1))
    out = np.ascontiguousarray(slot_w, dtype=np.uint8).copy()
    pv = None if prev is None else _i32(np.asarray(prev).reshape(-1))
    n_copied = ctypes.c_int32(0)
    n_bad = ctypes.c_int64(0)
    lib().oracle_stage(expert_w.ctypes.data, E, nb, _p(se, ctypes.c_int32),
                       None if pv is None else _p(pv, ctypes.c_int32), R, S, out.ctypes.data,
                       ctypes.byref(n_copied), ctypes.byref(n_bad))
    return out, int(n_copied.value), int(n_bad.value)
