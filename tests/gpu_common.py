"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and the oracle on the same seeded inputs, and compare them.

Every output buffer the tests hand to the library is allocated through a
``Guard``: 4 KiB past its end hold a fixed byte pattern, and ``Guard.check``
asserts after the calls that no kernel wrote there.  compute-sanitizer is not
available on the GPU machines these tests run on; the guard tails are how the
tests see a write past the end of an output."""
import math

import numpy as np
import torch

import oracle
from moe_expert_load_id_b300 import ultraep as U

GUARD_BYTES = 4096
_PATTERN = ((np.arange(GUARD_BYTES, dtype=np.uint32) * 37 + 0xA5) & 0xFF).astype(np.uint8)


class Guard:
    """Allocates output tensors with a guard tail and checks the tails later."""

    def __init__(self, device="cuda"):
        self.device = device
        self.items = []
        self.pattern = torch.from_numpy(_PATTERN).to(device)

    def alloc(self, name, shape, dtype, fill=None):
        n = math.prod(shape)
        esize = torch.empty((), dtype=dtype).element_size()
        extra = GUARD_BYTES // esize
        base = torch.empty(n + extra, dtype=dtype, device=self.device)
        raw = base.view(torch.uint8)
        raw[n * esize:].copy_(self.pattern)
        t = base[:n].view(shape)
        if fill is not None:
            t.fill_(fill)
        self.items.append((name, raw, n * esize))
        return t

    def check(self):
        torch.cuda.synchronize()
        for name, raw, off in self.items:
            tail = raw[off:]
            if not torch.equal(tail, self.pattern):
                bad = int((tail != self.pattern).nonzero()[0].item())
                raise AssertionError(f"{name}: write past the end (guard byte {bad} changed)")


def guarded_buffers(dom, T, n_inst=1, Hd=0, src_slot=False, guard=None, device="cuda"):
    """U.Buffers whose every output (and the count workspace) carries a guard tail."""
    g = guard if guard is not None else Guard(device)
    b = U.Buffers(dom, T, n_inst, Hd=0, device=device, src_slot=False)
    i32 = torch.int32
    N = T * dom.k
    specs = {"counts": ((n_inst, dom.E), None), "counts_src": ((n_inst, dom.R, dom.E), None),
             "dev_status": ((1,), 0), "quota": ((n_inst, dom.P), None),
             "slot_expert": ((n_inst, dom.R, dom.S), None), "rank_load": ((n_inst, dom.R), None),
             "inst_ptr": ((n_inst, dom.E + 1), None),
             "inst_id": ((n_inst, dom.E + dom.R * dom.S), -1),
             "inst_cum": ((n_inst, dom.E + dom.R * dom.S), -1), "n_iter": ((n_inst,), None),
             "inst_status": ((n_inst,), None), "dst_row": ((n_inst, N), None),
             "inst_offset": ((n_inst, dom.P + 1), None)}
    for name, (shape, fill) in specs.items():
        setattr(b, name, g.alloc(name, shape, i32, fill))
    b.workspace = g.alloc("workspace", tuple(b.workspace.shape), i32, 0)
    if src_slot:
        b.src_slot = g.alloc("src_slot", (n_inst, N), i32, -1)
    if Hd:
        b.Hd = Hd
        b.grouped = g.alloc("grouped", (n_inst, N, Hd), torch.bfloat16)
    b.guard = g
    return b


def dom_of(R, E, S, k):
    return U.Domain(R, E, S, k)


def gpu_run(dom, ids_np, hidden_u16=None, src_slot=True, max_iters=0, unpermute=True,
            fused=False, flags=0):
    """ids_np [n_inst, T, k] int32 (host).  Returns host numpy views of every output.
    fused: count -> plan -> reroute through the single ep_balance call."""
    n_inst, T, k = ids_np.shape
    dev = "cuda"
    ids = torch.from_numpy(np.ascontiguousarray(ids_np, dtype=np.int32)).to(dev)
    Hd = 0 if hidden_u16 is None else hidden_u16.shape[-1]
    b = guarded_buffers(dom, T, n_inst, Hd=Hd, src_slot=src_slot, device=dev)
    if fused:
        b.balance_fused(ids, max_iters=max_iters)
    else:
        b.count(ids)
        b.plan(max_iters=max_iters, flags=flags)
        b.reroute(ids)
    out = {}
    if hidden_u16 is not None:
        hid = torch.from_numpy(np.ascontiguousarray(hidden_u16).view(np.int16)).to(dev)
        hid = hid.view(torch.bfloat16).reshape(n_inst, T, Hd)
        b.grouped.zero_()
        b.permute(hid)
        if unpermute:
            y = b.guard.alloc("y", (n_inst, T, k, Hd), torch.bfloat16)
            U.ep_unpermute(b.grouped, T, k, b.dst_row, y, b.dev_status)
            out["y"] = y.view(torch.int16).cpu().numpy().view(np.uint16)
        out["grouped"] = b.grouped.view(torch.int16).cpu().numpy().view(np.uint16)
    b.guard.check()
    for name in ("counts", "counts_src", "quota", "slot_expert", "rank_load", "inst_ptr",
                 "inst_id", "inst_cum", "n_iter", "inst_status", "dst_row", "inst_offset",
                 "dev_status", "workspace"):
        out[name] = getattr(b, name).cpu().numpy()
    if src_slot:
        out["src_slot"] = b.src_slot.cpu().numpy()
    return out


def oracle_run(R, E, S, ids_np, hidden_u16=None, max_iters=oracle.PLAN_MAX_ITERS,
               variant="base"):
    """Per instance oracle outputs, same layout as gpu_run."""
    n_inst, T, k = ids_np.shape
    res = {key: [] for key in ("counts", "counts_src", "n_bad", "quota", "slot_expert",
                               "rank_load", "inst_ptr", "inst_id", "inst_cum", "n_iter",
                               "inst_status", "dst_row", "src_slot", "inst_offset", "grouped",
                               "y")}
    for g in range(n_inst):
        c, cs, nb = oracle.count(ids_np[g], R, E)
        pl = oracle.plan(c, R, E, S, max_iters=max_iters, variant=variant)
        dst, src, off = oracle.reroute(ids_np[g], R, E, S, pl)
        res["counts"].append(c)
        res["counts_src"].append(cs)
        res["n_bad"].append(nb)
        for key in ("quota", "slot_expert", "rank_load", "inst_ptr", "inst_id", "inst_cum"):
            res[key].append(pl[key])
        res["n_iter"].append(pl["n_iter"])
        res["inst_status"].append(pl["status"])
        res["dst_row"].append(dst)
        res["src_slot"].append(src)
        res["inst_offset"].append(off)
        if hidden_u16 is not None:
            n_rows = int(off[-1])
            grouped = oracle.permute(hidden_u16[g], k, src, n_rows)
            res["grouped"].append(grouped)
            full = np.zeros((T * k, hidden_u16.shape[-1]), np.uint16)
            full[:n_rows] = grouped
            res["y"].append(oracle.unpermute(full, T, k, dst))
    return res


def assert_equal(name, got, want):
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, f"{name}: shape {got.shape} != {want.shape}"
    if not np.array_equal(got, want):
        bad = np.argwhere(got != want)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {len(bad)} mismatches, first at {i}: "
                             f"gpu {got[i]} oracle {want[i]}")


def compare(R, E, S, g_out, o_out, check_rows=True):
    """Element-by-element comparison of every output (bit-exact)."""
    n_inst = len(o_out["counts"])
    for g in range(n_inst):
        assert_equal(f"counts[{g}]", g_out["counts"][g], o_out["counts"][g])
        assert_equal(f"counts_src[{g}]", g_out["counts_src"][g], o_out["counts_src"][g])
        for key in ("quota", "rank_load", "inst_ptr"):
            assert_equal(f"{key}[{g}]", g_out[key][g], o_out[key][g])
        assert_equal(f"slot_expert[{g}]", g_out["slot_expert"][g].reshape(-1),
                     o_out["slot_expert"][g].reshape(-1))
        m = int(o_out["inst_ptr"][g][E])
        assert_equal(f"inst_id[{g}]", g_out["inst_id"][g][:m], o_out["inst_id"][g][:m])
        assert_equal(f"inst_cum[{g}]", g_out["inst_cum"][g][:m], o_out["inst_cum"][g][:m])
        assert int(g_out["n_iter"][g]) == o_out["n_iter"][g], f"n_iter[{g}]"
        assert int(g_out["inst_status"][g]) == o_out["inst_status"][g], f"status[{g}]"
        assert_equal(f"dst_row[{g}]", g_out["dst_row"][g], o_out["dst_row"][g])
        assert_equal(f"inst_offset[{g}]", g_out["inst_offset"][g], o_out["inst_offset"][g])
        n_rows = int(o_out["inst_offset"][g][-1])
        if "src_slot" in g_out:
            assert_equal(f"src_slot[{g}]", g_out["src_slot"][g][:n_rows],
                         o_out["src_slot"][g][:n_rows])
        if check_rows and "grouped" in g_out and o_out["grouped"]:
            assert_equal(f"grouped[{g}]", g_out["grouped"][g][:n_rows], o_out["grouped"][g])
            if "y" in g_out:
                assert_equal(f"y[{g}]", g_out["y"][g], o_out["y"][g])
    n_tickets = n_inst  # one ticket per instance
    assert (g_out["workspace"][:n_tickets] == 0).all(), "count tickets not returned to zero"
