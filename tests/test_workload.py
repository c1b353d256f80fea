"""The seeded input generators (CPU): the properties the path and the
benchmark rely on, each checked against what the recipe fixes.

- Gumbel-top-k gives every token k distinct ids in [0, E), ordered by
  descending score, the same for the same seed; with k = 1 it is the Gumbel-max
  trick, an exact draw from p, so the top-1 frequencies must match p within
  sampling error (a closed form the sampler is pinned to).
- Zipf popularity: the sorted values stand in the ratio (i+1)^-s over ranks i.
- Dirichlet drift: fixed endpoints per layer, linear in the microbatch.
- Hidden rows: bf16 draws of N(0, 1), the same for the same seed.
"""
import numpy as np
import pytest
import torch

from moe_expert_load_id_b300 import workload as W


@pytest.mark.parametrize("E,k", [(8, 1), (32, 4), (128, 8), (160, 8), (16, 16)])
def test_gumbel_topk_gives_distinct_ids_in_range(E, k):
    p = np.random.default_rng(E * 31 + k).dirichlet(np.full(E, 0.5))
    ids = W.gumbel_topk(p, 3000, k, seed=E + k).numpy()
    assert ids.shape == (3000, k) and ids.dtype == np.int32
    assert ids.min() >= 0 and ids.max() < E
    srt = np.sort(ids, axis=1)
    assert (np.diff(srt, axis=1) > 0).all()  # k distinct ids per token
    again = W.gumbel_topk(p, 3000, k, seed=E + k).numpy()
    assert np.array_equal(ids, again)
    other = W.gumbel_topk(p, 3000, k, seed=E + k + 1).numpy()
    assert not np.array_equal(ids, other)


def test_gumbel_topk_rejects_k_above_E():
    with pytest.raises(ValueError):
        W.gumbel_topk(np.full(4, 0.25), 10, 5, seed=1)


def test_gumbel_max_is_a_draw_from_p():
    # k = 1: P(id = e) = p[e] exactly; 200k draws put every frequency within
    # five standard errors of p (a miss has probability ~1e-5 per expert)
    E, T = 12, 200_000
    p = np.arange(1, E + 1, dtype=np.float64) ** 1.5
    p /= p.sum()
    ids = W.gumbel_topk(p, T, 1, seed=4242).numpy()[:, 0]
    freq = np.bincount(ids, minlength=E) / T
    se = np.sqrt(p * (1 - p) / T)
    assert (np.abs(freq - p) < 5 * se).all(), (freq, p)


def test_first_listed_id_is_the_gumbel_max_draw():
    # ids are listed by descending score, so the first one is the largest
    # score, i.e. the Gumbel-max draw: its frequencies follow p for any k (a
    # different order, e.g. ascending, would not)
    E, T, k = 12, 200_000, 3
    p = 1.0 / (np.arange(E) + 1.0) ** 1.2
    p /= p.sum()
    ids = W.gumbel_topk(p, T, k, seed=77).numpy()
    freq = np.bincount(ids[:, 0], minlength=E) / T
    se = np.sqrt(p * (1 - p) / T)
    assert (np.abs(freq - p) < 5 * se).all(), (freq, p)


@pytest.mark.parametrize("name", ["tiny", "qwen3-235b", "glm-4.5"])
def test_zipf_popularity_has_the_stated_ratios(name):
    w = W.WORKLOADS[name]
    p = W.popularity(w, 3, 1)
    assert p.shape == (w.E,) and (p > 0).all() and abs(p.sum() - 1.0) < 1e-12
    srt = np.sort(p)[::-1]
    ranks = np.arange(1, w.E + 1, dtype=np.float64)
    assert np.allclose(srt / srt[0], ranks ** -w.s, rtol=1e-12)


def test_zipf_redraw_follows_the_workload_flag():
    q = W.WORKLOADS["qwen3-235b"]        # re-drawn every microbatch
    g = W.WORKLOADS["glm-4.5"]           # fixed per layer
    assert not np.array_equal(W.popularity(q, 5, 0), W.popularity(q, 5, 1))
    assert np.array_equal(W.popularity(g, 5, 0), W.popularity(g, 5, 1))
    assert not np.array_equal(W.popularity(g, 5, 0), W.popularity(g, 6, 0))


def test_dirichlet_drift_is_linear_in_the_microbatch():
    w = W.WORKLOADS["deepseek-v3"]
    M = w.microbatches
    p0, pm, pl = (W.popularity(w, 2, m) for m in (0, (M - 1) // 2, M - 1))
    for p in (p0, pm, pl):
        assert (p > 0).all() and abs(p.sum() - 1.0) < 1e-12
    f = ((M - 1) // 2) / (M - 1)
    # p(m) = 0.5 d + 0.5 ((1-f) A + f B) is affine in f
    assert np.allclose(pm, (1 - f) * p0 + f * pl, rtol=0, atol=1e-15)
    assert not np.allclose(p0, pl)


def test_popularity_desc_names_each_model():
    assert "re-drawn every microbatch" in W.WORKLOADS["qwen3-235b"].popularity_desc()
    assert "fixed per layer" in W.WORKLOADS["glm-4.5"].popularity_desc()
    assert "Dirichlet(0.3)" in W.WORKLOADS["deepseek-v3"].popularity_desc()


def test_hidden_rows_are_bf16_standard_normal():
    h = W.hidden(4096, 64, seed=99)
    assert h.shape == (4096, 64) and h.dtype == torch.bfloat16
    x = h.float().numpy().ravel()
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert torch.equal(h, W.hidden(4096, 64, seed=99))
    assert not torch.equal(h, W.hidden(4096, 64, seed=100))
