"""The seeded input generator: deterministic, shaped as the workloads say,
and its paged layout holds the same data as the contiguous one."""
import numpy as np
import torch

from oracle import dustin_oracle as O
from sparse_kv_verification_gb300 import inputs as I


def test_generator_is_deterministic_and_shaped():
    wl = I.WORKLOADS["tiny"]
    q1, k1, v1 = I.target_layer(wl, 0)
    q2, k2, v2 = I.target_layer(wl, 0)
    assert torch.equal(q1, q2) and torch.equal(k1, k2) and torch.equal(v1, v2)
    assert q1.shape == (1, 4, 4, 64) and k1.shape == (1, 2, 256, 64)
    assert q1.dtype == torch.bfloat16
    qd, kd = I.draft_layer(wl, 0)
    assert qd.shape == (1, 2, 3, 64) and kd.shape == (1, 1, 256, 64)
    pt, pd = I.scored_pairs(wl)
    assert len(pt) == wl.p_t and len(pd) == wl.p_d


def test_heavy_hitters_are_planted():
    wl = I.WORKLOADS["tiny"]
    hh = I.heavy_hitter_positions(wl)
    assert hh.shape == (1, round(0.02 * 256))
    q, k, _ = I.target_layer(wl, 0)
    # Planted keys align with the mean query direction.
    mean = q.float()[0, :2].reshape(-1, 64).mean(0)
    dots = k.float()[0, 0] @ (mean / mean.norm())
    assert dots[hh[0]].mean() > dots.mean() + 2.0


def test_paged_layout_round_trip():
    rng_k = torch.randn(2, 3, 50, 8).to(torch.bfloat16)
    rng_v = torch.randn(2, 3, 50, 8).to(torch.bfloat16)
    pool_k, pool_v, table = I.to_paged(rng_k, rng_v, 16, seed=5)
    assert table.shape == (2, 4) and pool_k.shape[1:] == (3, 16, 8)
    for b in range(2):
        for j in range(50):
            pg = int(table[b, j // 16])
            assert torch.equal(pool_k[pg, :, j % 16], rng_k[b, :, j])
            assert torch.equal(pool_v[pg, :, j % 16], rng_v[b, :, j])
    # Page ids are a permutation drawn from a larger pool.
    assert len(set(table.reshape(-1).tolist())) == 8


def test_random_indices_and_scores():
    idx = I.random_sorted_indices(3, 100, 17, seed=1)
    assert idx.shape == (3, 17) and idx.dtype == torch.int32
    assert bool((idx[:, 1:] > idx[:, :-1]).all())
    s = I.synthetic_scores(2, 300, seed=2, ties=True, specials=True)
    assert s.dtype == torch.float32 and s.shape == (2, 300)
    assert torch.isnan(s).any()


def test_tiny_chain_on_oracle():
    """Score -> select -> attend on the tiny workload, all on the oracle:
    the hybrid selection keeps most of the window's attention mass."""
    wl = I.WORKLOADS["tiny"]
    q, k, v = I.target_layer(wl, 0)
    qd, kd = I.draft_layer(wl, 0)
    pt, pd = I.scored_pairs(wl)
    f = lambda t: t.double().numpy()
    s_t = O.score_heads([f(I.historical_query(wl, q, h)) for _, h in pt],
                        [f(k)[:, h // wl.group] for _, h in pt], wl.scale)
    s_d = O.score_heads([f(qd)[:, h] for _, h in pd],
                        [f(kd)[:, h // wl.draft_group] for _, h in pd],
                        wl.draft_scale)
    idx = O.hybrid_select(s_d, s_t, wl.k, wl.n_sink, wl.n_recent, wl.alpha)
    assert idx.shape == (1, 32)
    a = O.attention_weights(f(q)[0, 0], f(k)[0, 0], wl.scale)   # [w][n]
    got = O.windowed_arr(a, idx[0])
    best = O.sd_oracle(a, wl.k)[1]
    assert 0.0 < got <= best + 1e-12
    o, lse = O.verify_attention(f(q), f(k), f(v), idx, wl.scale)
    assert np.all(np.isfinite(o)) and np.all(np.isfinite(lse))
