"""ep_combine (the gate-weighted combine fused with the gather) against the
CPU oracle, bit for bit: seeded bf16 rows with NaN, inf, -0 and subnormal
values mixed in, float32 weights of both signs and zeros, slots without a row,
several k (one and two batches of rows in flight, the maximum 32) and widths
(a ragged last warp chunk, 4096), several instances, and one full-size
Qwen3-235B-like layer checked on a seeded sample of tokens."""
import numpy as np
import pytest
import torch

import oracle
from moe_expert_load_id_b300 import workload as W

pytestmark = pytest.mark.gpu


def U():
    from moe_expert_load_id_b300 import ultraep
    return ultraep


def _rows(rng, n, Hd):
    x = rng.standard_normal((n, Hd)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)          # truncated: any bf16 is fine
    special = np.array([0x7FC1, 0xFF80, 0x7F80, 0x8000, 0x0001, 0x807F, 0x0000], np.uint16)
    m = rng.random((n, Hd)) < 0.01
    bits[m] = rng.choice(special, size=int(m.sum()))
    return bits


def G():
    import gpu_common
    return gpu_common


def _case(T, k, Hd, n_inst, seed):
    rng = np.random.default_rng(seed)
    N = T * k
    grouped = np.stack([_rows(rng, N, Hd) for _ in range(n_inst)])
    dst = np.stack([rng.permutation(N).astype(np.int32) for _ in range(n_inst)])
    if N:
        dst[:, rng.integers(0, N, size=max(1, N // 50))] = -1     # slots without a row
    w = rng.standard_normal((n_inst, T, k)).astype(np.float32)
    w[rng.random((n_inst, T, k)) < 0.05] = 0.0
    return grouped, dst, w


def _gpu_combine(grouped, dst, w, T, k):
    n_inst, N, Hd = grouped.shape
    g = torch.from_numpy(grouped.view(np.int16)).cuda().view(torch.bfloat16)
    d = torch.from_numpy(dst).cuda()
    wt = torch.from_numpy(w).cuda()
    guard = G().Guard()
    y = guard.alloc("y", (n_inst, T, Hd), torch.bfloat16, 7.0)
    st = guard.alloc("dev_status", (1,), torch.int32, 0)
    U().ep_combine(g, T, k, d, wt, y, st)
    guard.check()
    return y.view(torch.int16).cpu().numpy().view(np.uint16), int(st.item())


CASES = [
    # T,    k,  Hd,   n_inst
    (300,   8,  264,  1),       # ragged last chunk of a row (33 vectors)
    (1000,  1,  8,    2),
    (64,    11, 512,  1),       # two batches of rows in flight
    (50,    32, 16,   1),       # the largest k
    (512,   8,  4096, 1),
    (40,    3,  72,   3),
]


@pytest.mark.parametrize("T,k,Hd,n_inst", CASES)
def test_combine_matches_oracle(T, k, Hd, n_inst):
    grouped, dst, w = _case(T, k, Hd, n_inst, seed=T * 7 + k + Hd)
    got, st = _gpu_combine(grouped, dst, w, T, k)
    assert st == 0
    for g in range(n_inst):
        want = oracle.combine(grouped[g], T, k, dst[g], w[g])
        assert np.array_equal(got[g], want), f"instance {g}: {np.argwhere(got[g] != want)[:5]}"


def test_combine_empty_and_range_flag():
    grouped, dst, w = _case(16, 4, 8, 1, 3)
    got, st = _gpu_combine(grouped[:, :0], dst[:, :0], w[:, :0], 0, 4)
    assert got.shape == (1, 0, 8) and st == 0
    dst = dst.copy()
    dst[0, 5] = 16 * 4 + 9                                      # past the last row: adds nothing
    got, st = _gpu_combine(grouped, dst, w, 16, 4)
    assert st & U().EP_DEV_ROW_RANGE
    dst[0, 5] = -1
    assert np.array_equal(got[0], oracle.combine(grouped[0], 16, 4, dst[0], w[0]))


def test_combine_full_size_layer_sample():
    # one Qwen3-235B-like layer: permute the real hidden rows, combine them back
    # with seeded weights; 2048 seeded tokens against the oracle
    Uu = U()
    w_ = W.WORKLOADS["qwen3-235b"]
    ids = W.topk_ids(w_, 5, 0, device="cuda")[None]
    hid = W.hidden(w_.T, w_.Hd, w_.seed(5, 0), device="cuda")[None]
    b = G().guarded_buffers(Uu.Domain(w_.R, w_.E, w_.S, w_.k), w_.T, 1, Hd=w_.Hd)
    b.balance(ids, hid)
    gen = torch.Generator(device="cuda").manual_seed(11)
    wts = torch.softmax(torch.randn((1, w_.T, w_.k), device="cuda", generator=gen), -1)
    y = b.guard.alloc("y", (1, w_.T, w_.Hd), torch.bfloat16)
    Uu.ep_combine(b.grouped, w_.T, w_.k, b.dst_row, wts, y, b.dev_status)
    b.guard.check()
    assert int(b.dev_status.item()) == 0
    rng = np.random.default_rng(5)
    toks = np.sort(rng.choice(w_.T, size=2048, replace=False))
    dst = b.dst_row[0].view(w_.T, w_.k)[torch.from_numpy(toks).cuda()].cpu().numpy()
    rows = b.grouped[0][torch.from_numpy(dst.reshape(-1)).cuda()]
    sub = rows.view(torch.int16).cpu().numpy().view(np.uint16)
    want = oracle.combine(sub, len(toks), w_.k, np.arange(len(toks) * w_.k, dtype=np.int32),
                          wts[0][torch.from_numpy(toks).cuda()].cpu().numpy())
    got = y[0][torch.from_numpy(toks).cuda()].view(torch.int16).cpu().numpy().view(np.uint16)
    assert np.array_equal(got, want)


def _fused_differs_case(n_tok, seed):
    """k = 2 tokens whose combine depends on the product being rounded before the
    sum: with a fused multiply-add the bf16 result would differ.  Found by a
    seeded search on the CPU (float64 holds a product of two floats exactly)."""
    rng = np.random.default_rng(seed)
    rows, ws = [], []
    while len(rows) < n_tok:
        a = rng.standard_normal(2).astype(np.float32)
        xb = (a.view(np.uint32) >> 16).astype(np.uint16)
        x = (xb.astype(np.uint32) << 16).view(np.float32)
        w = rng.standard_normal(2).astype(np.float32)
        sep = np.float32(np.float32(w[0] * x[0]) + np.float32(w[1] * x[1]))
        fused = np.float32(np.float64(w[1]) * np.float64(x[1]) + np.float64(np.float32(w[0] * x[0])))
        bs = int(np.array([sep], np.float32).view(np.uint32)[0])
        bfz = int(np.array([fused], np.float32).view(np.uint32)[0])
        to_bf = lambda u: (u >> 16) + (1 if ((u & 0xFFFF) > 0x8000 or ((u & 0xFFFF) == 0x8000 and (u >> 16) & 1)) else 0)
        if to_bf(bs) != to_bf(bfz):
            rows.append(xb)
            ws.append(w)
    T, k = n_tok, 2
    grouped = np.zeros((1, T * k, 8), np.uint16)
    for t_, xb in enumerate(rows):
        grouped[0, 2 * t_, :] = xb[0]
        grouped[0, 2 * t_ + 1, :] = xb[1]
    dst = np.arange(T * k, dtype=np.int32)[None]
    w = np.stack(ws).astype(np.float32)[None]
    return grouped, dst, w


def test_combine_rounds_products_before_sums():
    grouped, dst, w = _fused_differs_case(64, 5)
    got, st = _gpu_combine(grouped, dst, w, 64, 2)
    assert st == 0
    want = oracle.combine(grouped[0], 64, 2, dst[0], w[0])
    assert np.array_equal(got[0], want)
