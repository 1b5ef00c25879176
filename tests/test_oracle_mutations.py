"""Each plausible mistake planted in the oracle (on the CPU) must make at
least one of its pins fail: this shows the pins constrain every part."""
import numpy as np
import pytest

from oracle import dustin_oracle as O
from tests import test_oracle as pins


def _window_mean_no_division(a_window):
    return np.sum(np.asarray(a_window, np.float64), axis=0)


def _rank_order_high_index_first(values, eligible=None):
    v = np.asarray(values, dtype=np.float64)
    pos = np.arange(v.shape[0])
    if eligible is not None:
        pos = pos[np.asarray(eligible, dtype=bool)]
    vv = v[pos]
    is_nan = np.isnan(vv)
    clean = np.where(is_nan, 0.0, vv) + 0.0
    order = np.lexsort((-pos, -clean, is_nan.astype(np.int8)))
    return pos[order]


def _score_heads_without_scale(queries, keys, scale):
    return ORIG["score_heads"](queries, keys, 1.0)


def _hybrid_alpha_on_target(s_draft, s_target, alpha, norm=O.NORM_L1):
    return ORIG["hybrid_scores"](s_draft, s_target, 1.0 - alpha, norm)


def _protected_off_by_one(n, n_sink, n_recent):
    sink = np.arange(min(max(n_sink, 0), n))
    recent = np.arange(max(n - max(n_recent, 0) - 1, 0), n)
    return np.union1d(sink, recent).astype(np.int64)


def _logsumexp_drops_peak(logits):
    x = np.asarray(logits, dtype=np.float64)
    if x.shape[-1] == 0:
        return np.full(x.shape[:-1], -np.inf)
    peak = np.max(x, axis=-1)
    return np.log(np.sum(np.exp(x - peak[..., None]), axis=-1))


def _verify_attention_wrong_gqa(q, keys, values, idx, scale):
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    b, hq, w, d = q.shape
    hkv = keys.shape[1]
    out = np.zeros((b, hq, w, d))
    lse = np.full((b, hq, w), -np.inf)
    for bi in range(b):
        sel = np.arange(keys.shape[2]) if idx is None else np.asarray(idx[bi])
        if sel.size == 0:
            continue
        for h in range(hq):
            g = h % hkv                                   # transposed mapping
            logits = scale * (q[bi, h] @ keys[bi, g][sel].T)
            lse[bi, h] = O.logsumexp(logits)
            out[bi, h] = O.softmax(logits) @ values[bi, g][sel]
    return out, lse


def _softmax_transposed(logits):
    x = np.asarray(logits, dtype=np.float64)
    if x.ndim < 2 or x.shape[-1] == 0:
        return ORIG["softmax"](x)
    peak = np.max(x, axis=-2, keepdims=True)
    e = np.exp(x - peak)
    return e / np.sum(e, axis=-2, keepdims=True)


def _window_attention_not_causal(q, keys, values, idx, k_win, v_win, scale):
    # the window rows see the whole window, later tokens included
    q = np.asarray(q, np.float64)
    b, hq, w, d = q.shape
    group = hq // np.asarray(keys).shape[1]
    out = np.zeros((b, hq, w, d))
    lse = np.zeros((b, hq, w))
    for bi in range(b):
        sel = np.arange(keys.shape[2]) if idx is None else np.asarray(idx[bi])
        for h in range(hq):
            g = h // group
            kk = np.concatenate([keys[bi, g][sel], k_win[bi, g]])
            vv = np.concatenate([values[bi, g][sel], v_win[bi, g]])
            for t in range(w):
                logits = scale * (kk @ q[bi, h, t])
                out[bi, h, t] = O.softmax(logits) @ vv
                lse[bi, h, t] = O.logsumexp(logits)
    return out, lse


def _quest_scores_max_only(q, stats):
    # uses the channel maxima whatever the sign of q_c
    q = np.asarray(q, np.float64)
    stats = np.asarray(stats, np.float64)
    group = q.shape[1] // stats.shape[1]
    out = np.zeros((q.shape[0], q.shape[1], stats.shape[2]))
    for h in range(q.shape[1]):
        out[:, h] = (q[:, h][:, None, :] * stats[:, h // group, :, 1]).sum(axis=-1)
    return out


ORIG = {name: getattr(O, name) for name in (
    "score_heads", "hybrid_scores", "softmax")}

MUTATIONS = [
    ("window_mean_attention", _window_mean_no_division,
     [pins.test_arr_worked_example]),
    ("rank_order", _rank_order_high_index_first,
     [lambda: pins.test_topk_brute_force_with_ties(0),
      pins.test_hybrid_worked_example]),
    ("score_heads", _score_heads_without_scale,
     [pins.test_score_heads_single_pair_is_library_softmax,
      pins.test_score_heads_closed_forms_and_invariants]),
    ("hybrid_scores", _hybrid_alpha_on_target,
     [pins.test_hybrid_worked_example]),
    ("protected_positions", _protected_off_by_one,
     [pins.test_hybrid_worked_example, pins.test_streaming_llm_special_case]),
    ("logsumexp", _logsumexp_drops_peak,
     [pins.test_attention_closed_forms]),
    ("verify_attention", _verify_attention_wrong_gqa,
     [pins.test_gqa_head_mapping]),
    ("verify_attention_window", _window_attention_not_causal,
     [pins.test_window_attention_matches_sdpa_with_a_causal_window_mask,
      pins.test_window_attention_without_history_is_causal_self_attention]),
    ("quest_page_scores", _quest_scores_max_only,
     [pins.test_quest_stats_bound_every_key_of_the_page,
      pins.test_quest_scores_closed_forms]),
    ("softmax", _softmax_transposed,
     [lambda: pins.test_dense_attention_matches_torch_sdpa(2, 4, 2, 3, 37, 16)]),
]


@pytest.mark.parametrize("name,mutant,checks", MUTATIONS,
                         ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, mutant, checks):
    monkeypatch.setattr(O, name, mutant)
    if name == "verify_attention":
        monkeypatch.setattr(O, "full_verify_attention",
                            lambda q, k, v, s: mutant(q, k, v, None, s))
    caught = False
    for check in checks:
        try:
            check()
        except (AssertionError, ValueError):
            caught = True
            break
    assert caught, f"no pin caught the planted mistake in {name}"
