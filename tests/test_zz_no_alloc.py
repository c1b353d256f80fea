"""ep_count_noalloc: the count step for callers that cannot allocate device memory.

Such callers (for example a plugin inside an inference engine whose device
memory all belongs to the engine's pool) cannot pass ep_count a workspace;
ep_count_noalloc keeps that workspace in a fixed array inside the library.
This file checks, through the C ABI, that it returns exactly what ep_count
returns, on two calls in a row (the second call finds the array holding the
first call's leftovers), and that it refuses shapes larger than its array.
The counts are also compared with the CPU oracle directly, and the array's
capacity is exercised at its exact limit (16384 instances, 64 KiB of tickets)
and one past it.  Every output carries a guard tail that must stay unchanged.
It is collected last so that a run stopping at the first failure has already
run every other test.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def G():
    import gpu_common
    return gpu_common


def _ids(n_inst, T, k, E, seed):
    rng = np.random.default_rng(seed)
    p = 1.0 / (rng.permutation(E) + 1.0) ** 1.2
    p /= p.sum()
    ids = np.stack([rng.choice(E, size=(T, k), p=p) for _ in range(n_inst)]).astype(np.int32)
    ids[0, 3, 0] = E + 5          # one out-of-range id: both entry points flag and skip it
    return torch.from_numpy(ids).cuda()


@pytest.mark.parametrize("R,E,S,k,T,n_inst", [
    (8, 32, 1, 4, 16384, 1),       # several chunks per source rank: partials in the array
    (64, 128, 1, 8, 131072, 1),    # the Qwen3-235B-like layer, as the benchmark calls it
    (64, 128, 1, 8, 4096, 94),     # many instances in one call
])
def test_noalloc_matches_ep_count_twice(R, E, S, k, T, n_inst):
    from moe_expert_load_id_b300 import ultraep as U
    dom = U.Domain(R, E, S, k)
    ws = U.ep_count_workspace_bytes(dom, T, n_inst)
    assert 0 < ws <= U.EP_COUNT_NOALLOC_SCRATCH_BYTES
    i32 = dict(dtype=torch.int32, device="cuda")
    ref_counts = torch.empty((n_inst, E), **i32)
    ref_src = torch.empty((n_inst, R, E), **i32)
    ref_status = torch.zeros(1, **i32)
    workspace = torch.zeros(ws // 4, **i32)
    guard = G().Guard()
    for call in range(2):
        ids = _ids(n_inst, T, k, E, seed=100 * call + T)
        U.ep_count(dom, ids, ref_counts, ref_src, ref_status, workspace)
        counts = guard.alloc(f"counts{call}", (n_inst, E), torch.int32, -7)
        src = guard.alloc(f"counts_src{call}", (n_inst, R, E), torch.int32, -7)
        status = guard.alloc(f"status{call}", (1,), torch.int32, 0)
        U.ep_count_noalloc(dom, ids, counts, src, status)
        guard.check()
        assert torch.equal(counts, ref_counts), f"counts differ on call {call}"
        assert torch.equal(src, ref_src), f"counts_src differ on call {call}"
        assert int(status.item()) == int(ref_status.item()) == U.EP_DEV_BAD_ID
        ids_h = ids.cpu().numpy()
        c_h, s_h = counts.cpu().numpy(), src.cpu().numpy()
        for g in range(0, n_inst, max(1, n_inst // 8)):
            oc, osrc, n_bad = oracle.count(ids_h[g], R, E)
            assert np.array_equal(c_h[g], oc) and np.array_equal(s_h[g], osrc), (call, g)
            assert n_bad == (1 if g == 0 else 0)


def test_noalloc_at_its_capacity():
    # 16384 instances need exactly the array's 64 KiB of tickets: accepted and
    # counted right; one more instance is refused
    from moe_expert_load_id_b300 import ultraep as U
    R, E, S, k, T, n_inst = 2, 4, 1, 2, 8, 16384
    dom = U.Domain(R, E, S, k)
    assert U.ep_count_workspace_bytes(dom, T, n_inst) == U.EP_COUNT_NOALLOC_SCRATCH_BYTES
    rng = np.random.default_rng(9)
    ids_h = rng.integers(0, E, size=(n_inst + 1, T, k)).astype(np.int32)
    ids = torch.from_numpy(ids_h).cuda()
    guard = G().Guard()
    counts = guard.alloc("counts", (n_inst + 1, E), torch.int32, -7)
    src = guard.alloc("counts_src", (n_inst + 1, R, E), torch.int32, -7)
    status = guard.alloc("status", (1,), torch.int32, 0)
    for _ in range(2):
        U.ep_count_noalloc(dom, ids[:n_inst], counts[:n_inst], src[:n_inst], status)
        guard.check()
        want = np.stack([np.bincount(ids_h[g].reshape(-1), minlength=E) for g in range(n_inst)])
        assert np.array_equal(counts[:n_inst].cpu().numpy(), want)
        for g in (0, 1, n_inst // 2, n_inst - 1):
            oc, osrc, _ = oracle.count(ids_h[g], R, E)
            assert np.array_equal(counts[g].cpu().numpy(), oc)
            assert np.array_equal(src[g].cpu().numpy(), osrc)
    assert int(status.item()) == 0
    assert (counts[n_inst].cpu().numpy() == -7).all()       # the row past the call untouched
    with pytest.raises(U.EpError) as err:
        U.ep_count_noalloc(dom, ids, counts, src, status)
    assert err.value.status == U.EP_ERR_WORKSPACE


def test_noalloc_rejects_shapes_beyond_its_array():
    from moe_expert_load_id_b300 import ultraep as U
    dom = U.Domain(64, 128, 1, 8)
    n_inst, T = 20000, 1
    assert U.ep_count_workspace_bytes(dom, T, n_inst) > U.EP_COUNT_NOALLOC_SCRATCH_BYTES
    i32 = dict(dtype=torch.int32, device="cuda")
    ids = torch.zeros((n_inst, T, 8), **i32)
    counts = torch.zeros((n_inst, 128), **i32)
    src = torch.zeros((n_inst, 64, 128), **i32)
    with pytest.raises(U.EpError) as err:
        U.ep_count_noalloc(dom, ids, counts, src, None)
    assert err.value.status == U.EP_ERR_WORKSPACE
