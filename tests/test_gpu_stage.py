"""ep_stage (replica weight staging) against the CPU oracle, byte for byte:
random expert tables of several sizes (one 16-byte vector; a ragged 257
vectors; several 64 KB chunks), slots that are empty, invalid, new or already
holding their expert, two instances, a slot buffer whose untouched slots must
keep their old bytes, and slot contents taken from a real ep_plan output."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_load_id_b300 import workload as W

pytestmark = pytest.mark.gpu


def U():
    from moe_expert_load_id_b300 import ultraep
    return ultraep


def G():
    import gpu_common
    return gpu_common


@pytest.mark.parametrize("nbytes", [16, 4112, 200000])
@pytest.mark.parametrize("with_prev", [False, True])
def test_stage_matches_oracle(nbytes, with_prev):
    R, E, S, k, n_inst = 8, 32, 2, 4, 2
    rng = np.random.default_rng(nbytes + with_prev)
    ew = rng.integers(0, 256, size=(n_inst, E, nbytes), dtype=np.uint8)
    sw0 = rng.integers(0, 256, size=(n_inst, R * S, nbytes), dtype=np.uint8)
    se = rng.integers(-1, E, size=(n_inst, R * S)).astype(np.int32)
    se[0, 3] = E + 4                                        # invalid: flagged, left alone
    prev = np.where(rng.random((n_inst, R * S)) < 0.3, se, rng.integers(0, E, (n_inst, R * S)))
    prev = prev.astype(np.int32)
    dom = U().Domain(R, E, S, k)
    ew_d = torch.from_numpy(ew).cuda()
    guard = G().Guard()
    sw_d = guard.alloc("slot_w", tuple(sw0.shape), torch.uint8)
    sw_d.copy_(torch.from_numpy(sw0))
    st = guard.alloc("dev_status", (1,), torch.int32, 0)
    U().ep_stage(dom, ew_d, torch.from_numpy(se).cuda(), sw_d,
                 torch.from_numpy(prev).cuda() if with_prev else None, st)
    guard.check()
    got = sw_d.cpu().numpy()
    for g in range(n_inst):
        want, _, _ = oracle.stage(ew[g], se[g], R, S, sw0[g], prev=prev[g] if with_prev else None)
        assert np.array_equal(got[g], want), f"instance {g}"
    assert int(st.item()) & U().EP_DEV_BAD_ID


def test_stage_from_a_real_plan():
    w = W.WORKLOADS["tiny"]
    dom = U().Domain(w.R, w.E, w.S, w.k)
    ids = W.topk_ids(w, 1, 0, device="cuda")[None]
    b = G().guarded_buffers(dom, w.T, 1)
    b.count(ids)
    b.plan()
    nbytes = 3 * 256 * 64 * 2                               # a small bf16 expert: 3 matrices
    gen = torch.Generator(device="cuda").manual_seed(3)
    ew = torch.randint(0, 256, (w.E, nbytes), dtype=torch.uint8, device="cuda", generator=gen)
    sw = b.guard.alloc("slot_w", (w.R, w.S, nbytes), torch.uint8, 0)
    U().ep_stage(dom, ew, b.slot_expert, sw, None, b.dev_status)
    b.guard.check()
    se = b.slot_expert.cpu().numpy().reshape(-1)
    want, n, bad = oracle.stage(ew.cpu().numpy(), se, w.R, w.S,
                                np.zeros((w.R * w.S, nbytes), np.uint8))
    assert np.array_equal(sw.cpu().numpy().reshape(w.R * w.S, nbytes), want)
    assert n == int((se >= 0).sum()) and bad == 0 and int(b.dev_status.item()) == 0
