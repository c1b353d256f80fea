"""The C-ABI library loads on a machine without a GPU, exports every entry point
include/ultraep.h declares, and rejects bad arguments on the host before any
CUDA call (no call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

from moe_expert_load_id_b300 import build as libbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ultraep.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(libbuild.LIB):
        libbuild.build()
    return ctypes.CDLL(libbuild.LIB)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ep_[a-z_]+)\s*\(", text)))


def test_header_declares_the_path():
    names = declared_functions()
    for n in ("ep_count", "ep_plan", "ep_reroute", "ep_permute", "ep_unpermute"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


class Dom(ctypes.Structure):
    _fields_ = [("R", ctypes.c_int32), ("E", ctypes.c_int32), ("S", ctypes.c_int32),
                ("k", ctypes.c_int32)]


def _setup(lib):
    vp = ctypes.c_void_p
    lib.ep_count_workspace_bytes.restype = ctypes.c_size_t
    lib.ep_count_workspace_bytes.argtypes = [ctypes.POINTER(Dom), ctypes.c_int64, ctypes.c_int32]
    lib.ep_count.argtypes = [ctypes.POINTER(Dom), vp, ctypes.c_int64, ctypes.c_int32, vp, vp, vp,
                             vp, ctypes.c_size_t, vp]
    lib.ep_plan.argtypes = [ctypes.POINTER(Dom), vp, ctypes.c_int32, ctypes.c_int32] + [vp] * 9
    lib.ep_permute.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                               vp, vp, vp, vp]
    lib.ep_status_str.restype = ctypes.c_char_p


@pytest.mark.parametrize("R,E,S,k,ok", [(8, 32, 1, 4, True), (64, 128, 1, 8, True),
                                        (64, 256, 2, 8, True), (40, 160, 1, 8, True),
                                        (0, 32, 1, 4, False), (65, 130, 1, 8, False),
                                        (8, 30, 1, 4, False), (8, 32, -1, 4, False),
                                        (8, 32, 1, 0, False), (8, 32, 1, 33, False),
                                        (4, 8, 1, 9, False), (2, 62, 2, 8, False)])
def test_domain_validation(lib, R, E, S, k, ok):
    _setup(lib)
    d = Dom(R, E, S, k)
    ws = lib.ep_count_workspace_bytes(ctypes.byref(d), 4096, 4)
    assert (ws > 0) == ok


def test_host_rejections_need_no_gpu(lib):
    _setup(lib)
    d = Dom(8, 32, 1, 4)
    fake = ctypes.c_void_p(0x10000)       # never dereferenced: every call below fails validation
    # null domain, bad domain, negative T, T*k >= 2^31
    assert lib.ep_count(None, fake, 16, 1, fake, fake, None, fake, 1 << 20, None) == 1
    assert lib.ep_count(ctypes.byref(Dom(8, 30, 1, 4)), fake, 16, 1, fake, fake, None, fake,
                        1 << 20, None) == 1
    assert lib.ep_count(ctypes.byref(d), fake, -1, 1, fake, fake, None, fake, 1 << 20, None) == 1
    assert lib.ep_count(ctypes.byref(d), fake, 1 << 29, 1, fake, fake, None, fake, 1 << 20,
                        None) == 1
    # missing outputs, misaligned pointer, too-small workspace
    assert lib.ep_count(ctypes.byref(d), fake, 16, 1, None, fake, None, fake, 1 << 20, None) == 1
    assert lib.ep_count(ctypes.byref(d), ctypes.c_void_p(0x10002), 16, 1, fake, fake, None,
                        fake, 1 << 20, None) == 1
    assert lib.ep_count(ctypes.byref(d), fake, 16, 1, fake, fake, None, fake, 4, None) == 4
    # zero instances: nothing to do, nothing launched
    assert lib.ep_count(ctypes.byref(d), None, 16, 0, None, None, None, None, 0, None) == 0
    assert lib.ep_plan(ctypes.byref(d), None, 0, 0, *([None] * 9)) == 0
    # permute: Hd not a multiple of 8, misaligned row pointers, k out of range
    assert lib.ep_permute(fake, 4, 2, 12, 1, fake, fake, None, None) == 1
    assert lib.ep_permute(ctypes.c_void_p(0x10008), 4, 2, 16, 1, fake, fake, None, None) == 1
    assert lib.ep_permute(fake, 4, 0, 16, 1, fake, fake, None, None) == 1
    assert lib.ep_permute(fake, 0, 2, 16, 1, None, fake, None, None) == 0
    assert lib.ep_status_str(0) == b"EP_OK"
    assert b"workspace" in lib.ep_status_str(4)


class BalanceOut(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in (
        "counts", "counts_src", "quota", "slot_expert", "rank_load", "inst_ptr", "inst_id",
        "inst_cum", "n_iter", "inst_status", "dst_row", "src_slot", "inst_offset")]


def test_balance_host_rejections_need_no_gpu(lib):
    vp = ctypes.c_void_p
    lib.ep_balance.argtypes = [ctypes.POINTER(Dom), vp, ctypes.c_int64, ctypes.c_int32,
                               ctypes.c_int32, ctypes.POINTER(BalanceOut), vp, vp,
                               ctypes.c_size_t, vp]
    d = Dom(8, 32, 1, 4)
    fake = 0x10000                        # never dereferenced: every call below fails validation
    full = BalanceOut(*([fake] * 10), fake, None, fake)
    ws = vp(fake)
    # no output struct, bad domain, T*k >= 2^31
    assert lib.ep_balance(ctypes.byref(d), vp(fake), 16, 1, 0, None, None, ws, 1 << 20, None) == 1
    assert lib.ep_balance(ctypes.byref(Dom(8, 30, 1, 4)), vp(fake), 16, 1, 0, ctypes.byref(full),
                          None, ws, 1 << 20, None) == 1
    assert lib.ep_balance(ctypes.byref(d), vp(fake), 1 << 29, 1, 0, ctypes.byref(full), None, ws,
                          1 << 20, None) == 1
    # a missing output array, a misaligned one, a workspace that is too small
    missing = BalanceOut(*([fake] * 10), None, None, fake)
    assert lib.ep_balance(ctypes.byref(d), vp(fake), 16, 1, 0, ctypes.byref(missing), None, ws,
                          1 << 20, None) == 1
    skew = BalanceOut(fake + 2, *([fake] * 9), fake, None, fake)
    assert lib.ep_balance(ctypes.byref(d), vp(fake), 16, 1, 0, ctypes.byref(skew), None, ws,
                          1 << 20, None) == 1
    assert lib.ep_balance(ctypes.byref(d), vp(fake), 16, 1, 0, ctypes.byref(full), None, ws, 4,
                          None) == 4
    # zero instances: nothing to do
    empty = BalanceOut(*([None] * 13))
    assert lib.ep_balance(ctypes.byref(d), None, 16, 0, 0, ctypes.byref(empty), None, None, 0,
                          None) == 0


def test_stage_host_rejections_need_no_gpu(lib):
    vp = ctypes.c_void_p
    lib.ep_stage.argtypes = [ctypes.POINTER(Dom), ctypes.c_int32, vp, ctypes.c_int64, vp, vp,
                             vp, vp, vp]
    d = Dom(8, 32, 1, 4)
    fake = vp(0x10000)                    # never dereferenced: every call below fails validation
    assert lib.ep_stage(ctypes.byref(d), 1, fake, 24, fake, None, fake, None, None) == 1  # 24 % 16
    assert lib.ep_stage(ctypes.byref(d), 1, vp(0x10008), 32, fake, None, fake, None, None) == 1
    assert lib.ep_stage(ctypes.byref(d), 1, fake, 32, None, None, fake, None, None) == 1
    assert lib.ep_stage(ctypes.byref(Dom(8, 30, 1, 4)), 1, fake, 32, fake, None, fake, None,
                        None) == 1
    # nothing to copy: no instances, no spare slots, empty experts
    assert lib.ep_stage(ctypes.byref(d), 0, None, 32, None, None, None, None, None) == 0
    assert lib.ep_stage(ctypes.byref(Dom(8, 32, 0, 4)), 1, None, 32, None, None, None, None,
                        None) == 0
    assert lib.ep_stage(ctypes.byref(d), 1, None, 0, None, None, None, None, None) == 0


def test_plan_ex_rejects_unknown_flags(lib):
    vp = ctypes.c_void_p
    lib.ep_plan_ex.argtypes = [ctypes.POINTER(Dom), vp, ctypes.c_int32, ctypes.c_int32,
                               ctypes.c_int32] + [vp] * 9
    d = Dom(8, 32, 1, 4)
    fake = vp(0x10000)                    # never dereferenced: every call below fails validation
    assert lib.ep_plan_ex(ctypes.byref(d), fake, 1, 0, 4, *([fake] * 8), None) == 1
    assert lib.ep_plan_ex(ctypes.byref(d), fake, 1, 0, -1, *([fake] * 8), None) == 1
    assert lib.ep_plan_ex(ctypes.byref(d), None, 0, 0, 3, *([None] * 8), None) == 0


def test_reroute_host_rejections_need_no_gpu(lib):
    vp = ctypes.c_void_p
    lib.ep_reroute.argtypes = [ctypes.POINTER(Dom), vp, ctypes.c_int64, ctypes.c_int32] + [vp] * 10
    d = Dom(8, 32, 1, 4)
    f = vp(0x10000)                       # never dereferenced: every call below fails validation
    odd = vp(0x10002)
    #                         ids T   n  counts_src quota ptr id cum dst src off status stream
    assert lib.ep_reroute(ctypes.byref(Dom(8, 30, 1, 4)), f, 16, 1, f, f, f, f, f, f, None, f,
                          None, None) == 1                                   # E % R != 0
    assert lib.ep_reroute(ctypes.byref(d), f, 16, -1, f, f, f, f, f, f, None, f, None,
                          None) == 1                                         # n_inst < 0
    assert lib.ep_reroute(ctypes.byref(d), f, 1 << 29, 1, f, f, f, f, f, f, None, f, None,
                          None) == 1                                         # T*k >= 2^31
    assert lib.ep_reroute(ctypes.byref(d), f, 16, 1, f, None, f, f, f, f, None, f, None,
                          None) == 1                                         # no quota
    assert lib.ep_reroute(ctypes.byref(d), f, 16, 1, f, f, f, f, f, odd, None, f, None,
                          None) == 1                                         # misaligned dst_row
    assert lib.ep_reroute(ctypes.byref(d), f, 16, 1, f, f, f, f, f, f, odd, f, None,
                          None) == 1                                         # misaligned src_slot
    assert lib.ep_reroute(ctypes.byref(d), f, 16, 1, f, f, f, f, f, f, None, f, odd,
                          None) == 1                                         # misaligned status
    assert lib.ep_reroute(ctypes.byref(d), None, 16, 0, *([None] * 10)) == 0  # nothing to do


def test_unpermute_and_combine_host_rejections_need_no_gpu(lib):
    vp = ctypes.c_void_p
    lib.ep_unpermute.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32, vp, vp, vp, vp]
    lib.ep_combine.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                               vp, vp, vp, vp, vp]
    f = vp(0x10000)                       # never dereferenced: every call below fails validation
    # unpermute: grouped, T, k, Hd, n_inst, dst_row, y, status, stream
    assert lib.ep_unpermute(f, 4, 2, 12, 1, f, f, None, None) == 1          # Hd % 8 != 0
    assert lib.ep_unpermute(f, 4, 0, 16, 1, f, f, None, None) == 1          # k < 1
    assert lib.ep_unpermute(f, 4, 33, 16, 1, f, f, None, None) == 1         # k > 32
    assert lib.ep_unpermute(vp(0x10008), 4, 2, 16, 1, f, f, None, None) == 1  # rows not 16-aligned
    assert lib.ep_unpermute(f, 4, 2, 16, 1, f, None, None, None) == 1       # no output
    assert lib.ep_unpermute(f, 4, 2, 16, 1, None, f, None, None) == 1       # no dst_row
    assert lib.ep_unpermute(f, 4, 2, 16, -1, f, f, None, None) == 1         # n_inst < 0
    assert lib.ep_unpermute(None, 0, 2, 16, 1, None, None, None, None) == 0  # no rows
    # combine: grouped, T, k, Hd, n_inst, dst_row, weights, y, status, stream
    assert lib.ep_combine(f, 4, 2, 16, 1, f, None, f, None, None) == 1      # no weights
    assert lib.ep_combine(f, 4, 2, 16, 1, f, vp(0x10002), f, None, None) == 1  # misaligned weights
    assert lib.ep_combine(f, 4, 2, 20, 1, f, f, f, None, None) == 1         # Hd % 8 != 0
    assert lib.ep_combine(f, 4, 2, 16, 1, f, f, vp(0x10004), None, None) == 1  # y not 16-aligned
    assert lib.ep_combine(None, 4, 2, 16, 0, None, None, None, None, None) == 0  # no instances


def test_row_calls_reject_rows_past_one_gib(lib):
    # Hd above 2^29 would make the row size (2 * Hd bytes) overflow an int
    vp = ctypes.c_void_p
    _setup(lib)
    lib.ep_unpermute.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32,
                                 ctypes.c_int32, vp, vp, vp, vp]
    lib.ep_combine.argtypes = [vp, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, ctypes.c_int32,
                               vp, vp, vp, vp, vp]
    f = vp(0x10000)                       # never dereferenced: every call below fails validation
    for hd in ((1 << 29) + 8, (1 << 30), (1 << 31) - 8):
        assert lib.ep_permute(f, 4, 2, hd, 1, f, f, None, None) == 1
        assert lib.ep_unpermute(f, 4, 2, hd, 1, f, f, None, None) == 1
        assert lib.ep_combine(f, 4, 2, hd, 1, f, f, f, None, None) == 1
    # the largest accepted row with no rows to move: nothing is launched
    assert lib.ep_permute(f, 0, 2, 1 << 29, 1, None, f, None, None) == 0


def test_count_noalloc_host_rejections_need_no_gpu(lib):
    vp = ctypes.c_void_p
    lib.ep_count_noalloc.argtypes = [ctypes.POINTER(Dom), vp, ctypes.c_int64, ctypes.c_int32,
                                     vp, vp, vp, vp]
    f = vp(0x10000)                       # never dereferenced: every call below fails validation
    d = Dom(64, 128, 1, 8)
    assert lib.ep_count_noalloc(ctypes.byref(Dom(8, 30, 1, 4)), f, 16, 1, f, f, None,
                                None) == 1                                   # bad domain
    assert lib.ep_count_noalloc(ctypes.byref(d), f, 16, 1, None, f, None, None) == 1  # no counts
    # more instances than the library's fixed array holds tickets for: refused
    # before any CUDA call; 16384 tickets fill the 64 KiB exactly, 16385 do not fit
    assert lib.ep_count_noalloc(ctypes.byref(d), f, 1, 20000, f, f, None, None) == 4
    assert lib.ep_count_noalloc(ctypes.byref(d), f, 1, 16385, f, f, None, None) == 4
    lib.ep_count_workspace_bytes.restype = ctypes.c_size_t
    lib.ep_count_workspace_bytes.argtypes = [ctypes.POINTER(Dom), ctypes.c_int64, ctypes.c_int32]
    assert lib.ep_count_workspace_bytes(ctypes.byref(d), 1, 16384) == 64 << 10
    assert lib.ep_count_workspace_bytes(ctypes.byref(d), 1, 16385) > 64 << 10
    assert lib.ep_count_noalloc(ctypes.byref(d), None, 16, 0, None, None, None, None) == 0
