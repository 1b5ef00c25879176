"""Pins for the CPU oracle: it is checked against hand-derived fixtures,
brute force, closed forms, invariants and library routines, never against
itself or the CUDA path."""
import itertools
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

from oracle import dustin_oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def rand_attention(rng, w, n, peak=2.0):
    return scipy.special.softmax(peak * rng.standard_normal((w, n)), axis=-1)


# ----------------------------------------------------------- ARR, Eq. (1)-(4)

def test_arr_worked_example():
    g = load("arr_window_example.json")
    a = np.array(g["a_window"])
    np.testing.assert_array_equal(O.window_mean_attention(a), g["abar"])
    for case in g["oracle"]:
        chosen, value = O.sd_oracle(a, case["k"])
        assert chosen.tolist() == case["set"]
        assert value == case["arr"]
        assert O.windowed_arr(a, chosen) == case["arr"]
    for case in g["policies"]:
        assert [O.arr(a[s], case["set"]) for s in range(2)] == case["arr_rows"]
        assert O.windowed_arr(a, case["set"]) == case["windowed_arr"]


@pytest.mark.parametrize("seed", range(6))
def test_sd_oracle_is_optimal_by_brute_force(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(5, 13))
    w = int(rng.integers(1, 5))
    a = rand_attention(rng, w, n)
    for k in range(0, min(5, n) + 1):
        best = max(O.windowed_arr(a, s)
                   for s in itertools.combinations(range(n), k))
        chosen, value = O.sd_oracle(a, k)
        assert len(chosen) == k
        assert value == pytest.approx(best, abs=1e-12)
        assert O.windowed_arr(a, chosen) == pytest.approx(best, abs=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_arr_invariants(seed):
    rng = np.random.default_rng(100 + seed)
    w, n = 4, 64
    a = rand_attention(rng, w, n)
    abar = O.window_mean_attention(a)
    assert abs(abar.sum() - 1.0) < 1e-12          # rows of A sum to 1
    prev = -1.0
    for k in range(0, n + 1):
        chosen, value = O.sd_oracle(a, k)
        assert 0.0 <= value <= 1.0 + 1e-12
        assert value >= prev - 1e-15              # nested sets: monotone
        prev = value
    assert O.sd_oracle(a, n)[1] == pytest.approx(1.0, abs=1e-12)
    assert O.windowed_arr(a, []) == 0.0
    # Any policy is bounded by the oracle at the same budget.
    for _ in range(20):
        s = rng.choice(n, size=8, replace=False)
        assert O.windowed_arr(a, s) <= O.sd_oracle(a, 8)[1] + 1e-12


def test_windowed_arr_is_mean_of_rows():
    rng = np.random.default_rng(7)
    a = rand_attention(rng, 3, 20)
    s = [1, 4, 9]
    by_hand = (a[0, s].sum() + a[1, s].sum() + a[2, s].sum()) / 3.0
    assert O.windowed_arr(a, s) == pytest.approx(by_hand, abs=1e-15)


# ----------------------------------------------------------- attention

def test_attention_worked_example():
    g = load("attention_example.json")
    q = np.array(g["q"])[None, None, None, :]
    keys = np.array(g["keys"])[None, None]
    vals = np.array(g["values"])[None, None]
    o, lse = O.full_verify_attention(q, keys, vals, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], g["o"], atol=1e-12)
    assert lse[0, 0, 0] == pytest.approx(g["lse"], abs=1e-12)
    np.testing.assert_allclose(
        O.attention_weights(np.array(g["q"]), np.array(g["keys"]), 1.0),
        g["weights"], atol=1e-12)


@pytest.mark.parametrize("b,hq,hkv,w,n,d", [(2, 4, 2, 3, 37, 16),
                                            (1, 6, 3, 5, 64, 8),
                                            (2, 8, 8, 1, 9, 32)])
def test_dense_attention_matches_torch_sdpa(b, hq, hkv, w, n, d):
    """Library special case: torch's scaled_dot_product_attention in fp64."""
    rng = np.random.default_rng(11)
    q = rng.standard_normal((b, hq, w, d))
    k = rng.standard_normal((b, hkv, n, d))
    v = rng.standard_normal((b, hkv, n, d))
    scale = 1.0 / math.sqrt(d)
    o, lse = O.full_verify_attention(q, k, v, scale)
    group = hq // hkv
    tq = torch.from_numpy(q)
    tk = torch.from_numpy(k).repeat_interleave(group, dim=1)
    tv = torch.from_numpy(v).repeat_interleave(group, dim=1)
    ref = torch.nn.functional.scaled_dot_product_attention(
        tq, tk, tv, scale=scale)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)
    ref_lse = torch.logsumexp(scale * tq @ tk.transpose(-1, -2), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), atol=1e-12)


def test_sparse_attention_is_dense_attention_on_gathered_cache():
    rng = np.random.default_rng(12)
    b, hq, hkv, w, n, d = 2, 4, 2, 3, 50, 16
    q = rng.standard_normal((b, hq, w, d))
    k = rng.standard_normal((b, hkv, n, d))
    v = rng.standard_normal((b, hkv, n, d))
    idx = np.stack([np.sort(rng.choice(n, 11, replace=False))
                    for _ in range(b)])
    o, lse = O.verify_attention(q, k, v, idx, 0.25)
    for bi in range(b):
        tq = torch.from_numpy(q[bi:bi + 1])
        tk = torch.from_numpy(k[bi:bi + 1][:, :, idx[bi]]).repeat_interleave(
            2, dim=1)
        tv = torch.from_numpy(v[bi:bi + 1][:, :, idx[bi]]).repeat_interleave(
            2, dim=1)
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, scale=0.25)
        np.testing.assert_allclose(o[bi:bi + 1], ref.numpy(), atol=1e-12)
    # k = n with the identity index set is the dense call.
    full = np.tile(np.arange(n), (b, 1))
    o1, l1 = O.verify_attention(q, k, v, full, 0.25)
    o2, l2 = O.full_verify_attention(q, k, v, 0.25)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)


# ------------------------------------------------ window self-block merged in

def _window_case(seed, b=2, hq=4, hkv=2, w=4, n=40, d=16, k=9):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((b, hq, w, d))
    kk = rng.standard_normal((b, hkv, n, d))
    vv = rng.standard_normal((b, hkv, n, d))
    kw = rng.standard_normal((b, hkv, w, d))
    vw = rng.standard_normal((b, hkv, w, d))
    idx = np.stack([np.sort(rng.choice(n, k, replace=False)) for _ in range(b)])
    return q, kk, vv, kw, vw, idx


def test_window_attention_matches_sdpa_with_a_causal_window_mask():
    """Library special case: SDPA in fp64 over [K[idx]; K_win] with a mask
    that opens all the selected history and the causal part of the window."""
    q, kk, vv, kw, vw, idx = _window_case(21)
    b, hq, w, d = q.shape
    group = hq // kk.shape[1]
    o, lse = O.verify_attention_window(q, kk, vv, idx, kw, vw, 0.3)
    for bi in range(b):
        ck = np.concatenate([kk[bi][:, idx[bi]], kw[bi]], axis=1)
        cv = np.concatenate([vv[bi][:, idx[bi]], vw[bi]], axis=1)
        tk = torch.from_numpy(ck).repeat_interleave(group, dim=0)[None]
        tv = torch.from_numpy(cv).repeat_interleave(group, dim=0)[None]
        kk_len = idx.shape[1]
        mask = torch.ones((w, kk_len + w), dtype=torch.bool)
        mask[:, kk_len:] = torch.tril(torch.ones((w, w), dtype=torch.bool))
        tq = torch.from_numpy(q[bi:bi + 1])
        ref = torch.nn.functional.scaled_dot_product_attention(
            tq, tk, tv, attn_mask=mask, scale=0.3)
        np.testing.assert_allclose(o[bi:bi + 1], ref.numpy(), atol=1e-12)
        logits = 0.3 * (tq @ tk.transpose(-1, -2))
        ref_lse = torch.logsumexp(logits.masked_fill(~mask, -math.inf), dim=-1)
        np.testing.assert_allclose(lse[bi:bi + 1], ref_lse.numpy(), atol=1e-12)


def test_window_attention_without_history_is_causal_self_attention():
    q, kk, vv, kw, vw, _ = _window_case(22)
    group = q.shape[1] // kk.shape[1]
    empty = np.zeros((q.shape[0], 0), dtype=np.int64)
    o, _ = O.verify_attention_window(q, kk, vv, empty, kw, vw, 0.25)
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q),
        torch.from_numpy(kw).repeat_interleave(group, dim=1),
        torch.from_numpy(vw).repeat_interleave(group, dim=1),
        is_causal=True, scale=0.25)
    np.testing.assert_allclose(o, ref.numpy(), atol=1e-12)


def test_window_attention_is_the_lse_merge_of_history_and_window():
    """Splitting the softmax over a disjoint union: the joint output is the
    two parts' outputs weighted by exp(LSE) (closed form)."""
    q, kk, vv, kw, vw, idx = _window_case(23)
    o, lse = O.verify_attention_window(q, kk, vv, idx, kw, vw, 0.4)
    o_h, l_h = O.verify_attention(q, kk, vv, idx, 0.4)
    b, hq, w, d = q.shape
    group = hq // kk.shape[1]
    for bi in range(b):
        for h in range(hq):
            g = h // group
            for t in range(w):
                lw = 0.4 * (kw[bi, g, :t + 1] @ q[bi, h, t])
                l_w = scipy.special.logsumexp(lw)
                o_w = scipy.special.softmax(lw) @ vw[bi, g, :t + 1]
                m = max(l_h[bi, h, t], l_w)
                a_h, a_w = math.exp(l_h[bi, h, t] - m), math.exp(l_w - m)
                np.testing.assert_allclose(
                    o[bi, h, t], (a_h * o_h[bi, h, t] + a_w * o_w) / (a_h + a_w),
                    atol=1e-12)
                assert lse[bi, h, t] == pytest.approx(
                    m + math.log(a_h + a_w), abs=1e-12)
    # w = 1: the single row sees the history and itself.
    o1, _ = O.verify_attention_window(q[:, :, :1], kk, vv, idx, kw[:, :, :1],
                                      vw[:, :, :1], 0.4)
    np.testing.assert_allclose(o1, o[:, :, :1], atol=1e-12)


def test_attention_closed_forms():
    rng = np.random.default_rng(13)
    d, n = 8, 20
    v = rng.standard_normal((1, 1, n, d))
    idx = np.array([[2, 5, 7, 11]])
    # Identical keys: uniform weights over the selection.
    kr = rng.standard_normal(d)
    k = np.tile(kr, (1, 1, n, 1))
    q = rng.standard_normal((1, 1, 1, d))
    o, lse = O.verify_attention(q, k, v, idx, 0.5)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, idx[0]].mean(axis=0),
                               atol=1e-12)
    assert lse[0, 0, 0] == pytest.approx(0.5 * q[0, 0, 0] @ kr + math.log(4),
                                         abs=1e-12)
    # Zero query: LSE = log k.
    o, lse = O.verify_attention(np.zeros((1, 1, 1, d)), rng.standard_normal(
        (1, 1, n, d)), v, idx, 1.0)
    assert lse[0, 0, 0] == pytest.approx(math.log(4), abs=1e-12)
    # One dominant key: the output is that key's value row.
    k = np.zeros((1, 1, n, d))
    k[0, 0, 7, 0] = 100.0
    q = np.zeros((1, 1, 1, d))
    q[0, 0, 0, 0] = 1.0
    o, lse = O.verify_attention(q, k, v, idx, 1.0)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 7], atol=1e-12)
    assert lse[0, 0, 0] == pytest.approx(100.0, abs=1e-12)
    # Empty selection: O = 0, LSE = -inf.
    o, lse = O.verify_attention(q, k, v, np.zeros((1, 0), np.int64), 1.0)
    assert np.all(o == 0.0) and lse[0, 0, 0] == -np.inf


def test_gqa_head_mapping():
    """Query head h reads kv head h // (hq // hkv): with kv head g's values
    all equal to g, every output of head h equals h // group."""
    b, hq, hkv, w, n, d = 1, 8, 2, 2, 6, 4
    rng = np.random.default_rng(14)
    q = rng.standard_normal((b, hq, w, d))
    k = rng.standard_normal((b, hkv, n, d))
    v = np.zeros((b, hkv, n, d))
    for g in range(hkv):
        v[:, g] = float(g)
    o, _ = O.full_verify_attention(q, k, v, 1.0)
    for h in range(hq):
        np.testing.assert_allclose(o[0, h], h // (hq // hkv), atol=1e-12)


# ----------------------------------------------------------- scoring

def test_score_heads_single_pair_is_library_softmax():
    rng = np.random.default_rng(21)
    b, n, d = 2, 40, 16
    q = rng.standard_normal((b, 1, d))
    k = rng.standard_normal((b, n, d))
    s = O.score_heads([q], [k], 0.3)
    for bi in range(b):
        ref = scipy.special.softmax(0.3 * (k[bi] @ q[bi, 0]))
        np.testing.assert_allclose(s[bi], ref, atol=1e-14)
    g = load("attention_example.json")
    s = O.score_heads([np.array(g["q"])[None, None]],
                      [np.array(g["keys"])[None]], 1.0)
    np.testing.assert_allclose(s[0], g["weights"], atol=1e-12)


def test_score_heads_closed_forms_and_invariants():
    rng = np.random.default_rng(22)
    b, n, d, rows = 2, 33, 8, 3
    qs = [rng.standard_normal((b, rows, d)) for _ in range(4)]
    ks = [rng.standard_normal((b, n, d)) for _ in range(4)]
    s = O.score_heads(qs, ks, 0.5)
    # Each softmax row sums to 1: the vector sums to pairs * rows.
    np.testing.assert_allclose(s.sum(axis=1), 4 * rows, atol=1e-12)
    # Sum over pairs: additive.
    s01 = O.score_heads(qs[:2], ks[:2], 0.5)
    s23 = O.score_heads(qs[2:], ks[2:], 0.5)
    np.testing.assert_allclose(s, s01 + s23, atol=1e-13)
    # Sum over rows: rows scored one at a time add up.
    per_row = sum(O.score_heads([qs[0][:, r:r + 1]], [ks[0]], 0.5)
                  for r in range(rows))
    np.testing.assert_allclose(O.score_heads([qs[0]], [ks[0]], 0.5), per_row,
                               atol=1e-13)
    # A zero query attends uniformly.
    z = O.score_heads([np.zeros((b, rows, d))], [ks[0]], 0.5)
    np.testing.assert_allclose(z, rows / n, atol=1e-15)
    # The scale enters the logits: scale 0 is uniform too.
    np.testing.assert_allclose(O.score_heads([qs[1]], [ks[1]], 0.0), rows / n,
                               atol=1e-15)


# ----------------------------------------------------------- Top-K

def brute_topk(values, k, eligible):
    """The size-k eligible subset with the largest sum; among equal sums the
    one whose ascending position list is lexicographically smallest."""
    pos = [j for j in range(len(values)) if eligible[j]]
    best_key, best = None, None
    for s in itertools.combinations(pos, k):
        total = sum(values[j] for j in s)
        key = (-total, list(s))
        if best_key is None or key < best_key:
            best_key, best = key, s
    return sorted(best)


@pytest.mark.parametrize("seed", range(8))
def test_topk_brute_force_with_ties(seed):
    rng = np.random.default_rng(300 + seed)
    n = int(rng.integers(4, 12))
    values = rng.integers(0, 4, n).astype(np.float64)      # many exact ties
    values[rng.integers(0, n)] = -0.0
    values[rng.integers(0, n)] = np.inf
    eligible = rng.random(n) < 0.8
    for k in range(0, int(eligible.sum()) + 1):
        # Brute force uses exact sums; swap inf for a large finite value.
        finite = np.where(np.isinf(values), 1e6, values)
        got = sorted(O.topk(values, k, eligible).tolist())
        assert got == brute_topk(finite, k, eligible)


def test_topk_special_values():
    v = np.array([np.nan, -np.inf, 0.0, -0.0, 1.0, np.nan, -5.0])
    order = O.rank_order(v).tolist()
    assert order == [4, 2, 3, 6, 1, 0, 5]   # -0 ties +0; NaN below -inf
    assert O.topk(v, 0).size == 0


# ----------------------------------------------------------- selection

def test_hybrid_worked_example():
    g = load("hybrid_example.json")
    sd = np.array(g["s_draft"])
    st = np.array(g["s_target"])
    c = O.hybrid_scores(sd, st, g["alpha"], O.NORM_L1)
    np.testing.assert_array_equal(c, np.array(g["hybrid"], np.float32))
    np.testing.assert_array_equal(O.hybrid_scores(sd, None, 1.0, O.NORM_L1),
                                  np.array(g["normalised_draft"], np.float32))
    np.testing.assert_array_equal(O.hybrid_scores(None, st, 0.0, O.NORM_L1),
                                  np.array(g["normalised_target"], np.float32))
    for case in g["alpha_mode"]:
        got = O.hybrid_select(sd[None], st[None], case["k"], 0, 0,
                              g["alpha"], -1, O.NORM_L1)
        assert got[0].tolist() == case["idx"]
    for case in g["m_mode"]:
        got = O.hybrid_select(sd[None], st[None], case["k"], 0, 0,
                              g["alpha"], case["m"], O.NORM_L1)
        assert got[0].tolist() == case["idx"]
    for case in g["protected"]:
        got = O.protected_positions(case["n"], case["n_sink"],
                                    case["n_recent"])
        assert got.tolist() == case["idx"]


def test_streaming_llm_special_case():
    """k = n_sink + n_recent keeps exactly the protected positions, whatever
    the scores (StreamingLLM-style retention)."""
    rng = np.random.default_rng(40)
    n = 64
    sd = rng.random((3, n))
    st = rng.random((3, n))
    idx = O.hybrid_select(sd, st, 4 + 8, 4, 8, 0.5)
    for row in idx:
        assert row.tolist() == list(range(4)) + list(range(56, 64))


def test_alpha_and_m_extremes_reduce_to_single_signal():
    rng = np.random.default_rng(41)
    n, k, ns, nr = 80, 20, 2, 5
    sd = rng.random((2, n)).astype(np.float32)
    st = rng.random((2, n)).astype(np.float32)
    forced = O.protected_positions(n, ns, nr)
    elig = np.ones(n, bool)
    elig[forced] = False
    for bi in range(2):
        want_d = np.sort(np.concatenate([forced, O.topk(sd[bi], k - 7, elig)]))
        want_t = np.sort(np.concatenate([forced, O.topk(st[bi], k - 7, elig)]))
        assert O.hybrid_select(sd, st, k, ns, nr, 1.0, -1, O.NORM_NONE)[
            bi].tolist() == want_d.tolist()
        assert O.hybrid_select(sd, st, k, ns, nr, 0.0, -1, O.NORM_NONE)[
            bi].tolist() == want_t.tolist()
        assert O.hybrid_select(sd, st, k, ns, nr, 0.5, 0)[bi].tolist() == \
            want_t.tolist()
        assert O.hybrid_select(sd, st, k, ns, nr, 0.5, 100)[bi].tolist() == \
            want_d.tolist()


def test_m_mode_structure():
    rng = np.random.default_rng(42)
    n, k, ns, nr, m = 100, 30, 3, 6, 10
    sd = rng.random((1, n)).astype(np.float32)
    st = rng.random((1, n)).astype(np.float32)
    idx = O.hybrid_select(sd, st, k, ns, nr, 0.5, m)[0]
    forced = O.protected_positions(n, ns, nr)
    assert len(idx) == k and len(set(idx.tolist())) == k
    assert np.all(np.diff(idx) > 0)
    assert set(forced.tolist()) <= set(idx.tolist())
    elig = np.ones(n, bool)
    elig[forced] = False
    draft_pick = O.topk(sd[0], m, elig)
    assert set(draft_pick.tolist()) <= set(idx.tolist())
    rest = sorted(set(idx.tolist()) - set(forced.tolist())
                  - set(draft_pick.tolist()))
    # The remainder is the target's best among what the draft left.
    elig2 = elig.copy()
    elig2[draft_pick] = False
    assert rest == sorted(O.topk(st[0], k - len(forced) - m, elig2).tolist())


def test_select_edge_cases():
    rng = np.random.default_rng(43)
    s = rng.random((2, 10))
    assert O.hybrid_select(s, s, 10, 2, 2)[0].tolist() == list(range(10))
    assert O.hybrid_select(s, s, 50, 2, 2)[1].tolist() == list(range(10))
    with pytest.raises(ValueError):
        O.hybrid_select(s, s, 3, 2, 2)
    # Budget equal to the protected count.
    assert O.hybrid_select(s, s, 4, 2, 2)[0].tolist() == [0, 1, 8, 9]


def test_bf16_rounding_helper():
    x = np.array([1.0, 1.0 + 2 ** -8, 1.0 + 3 * 2 ** -9, -2.5, 0.0, 1e-3])
    torch_round = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    np.testing.assert_array_equal(O.round_to_bf16(x), torch_round)


# --------------------------------------------- Quest page scoring (baseline)

def test_quest_stats_bound_every_key_of_the_page():
    """Invariant: q . k <= score of k's page for every key (the box bound),
    with equality when the page holds one key; stats do not depend on the
    order of the keys inside a page."""
    rng = np.random.default_rng(51)
    b, hq, hkv, n, d, page = 2, 4, 2, 53, 8, 16
    k = rng.standard_normal((b, hkv, n, d))
    q = rng.standard_normal((b, hq, d))
    st = O.quest_page_stats(k, page)
    sc = O.quest_page_scores(q, st)
    assert st.shape == (b, hkv, 4, 2, d) and sc.shape == (b, hq, 4)
    for bi in range(b):
        for h in range(hq):
            dots = k[bi, h // 2] @ q[bi, h]
            for j in range(n):
                assert dots[j] <= sc[bi, h, j // page] + 1e-12
            # the short last page (53 = 3 * 16 + 5) has its own box
            last = k[bi, h // 2, 48:]
            assert np.allclose(st[bi, h // 2, 3, 0], last.min(axis=0))
    perm = np.concatenate([rng.permutation(16) + 16 * p for p in range(3)] +
                          [48 + rng.permutation(5)])
    np.testing.assert_array_equal(O.quest_page_stats(k[:, :, perm], page), st)
    one = O.quest_page_stats(k, 1)
    np.testing.assert_allclose(O.quest_page_scores(q, one)[:, 0],
                               np.einsum("bnd,bd->bn", k[:, 0], q[:, 0]),
                               atol=1e-12)


def test_quest_scores_closed_forms():
    rng = np.random.default_rng(52)
    k = rng.standard_normal((1, 1, 32, 6))
    st = O.quest_page_stats(k, 16)
    for c in range(6):
        e = np.zeros((1, 1, 6))
        e[0, 0, c] = 1.0                     # unit query: the page maximum
        np.testing.assert_allclose(O.quest_page_scores(e, st)[0, 0],
                                   [k[0, 0, :16, c].max(), k[0, 0, 16:, c].max()])
        np.testing.assert_allclose(O.quest_page_scores(-e, st)[0, 0],
                                   [-k[0, 0, :16, c].min(), -k[0, 0, 16:, c].min()])
    # brute force over the box corners: the score is the largest q . x over
    # x in the box, attained at a corner
    q = rng.standard_normal((1, 1, 6))
    lo, hi = st[0, 0, 0, 0], st[0, 0, 0, 1]
    best = max(q[0, 0] @ np.where(np.array(bits), hi, lo)
               for bits in itertools.product([0, 1], repeat=6))
    assert O.quest_page_scores(q, st)[0, 0, 0] == pytest.approx(best, abs=1e-12)


def test_quest_page_selection():
    sc = np.array([[[0.5, 2.0, 2.0, -1.0, 3.0]]])
    np.testing.assert_array_equal(O.quest_select_pages(sc, 3), [[[1, 2, 4]]])
    np.testing.assert_array_equal(O.quest_select_pages(sc, 2), [[[1, 4]]])
    np.testing.assert_array_equal(O.quest_select_pages(sc, 9), [[[0, 1, 2, 3, 4]]])
