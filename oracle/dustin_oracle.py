"""CPU oracle for Dustin's draft-augmented sparse verification.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
the ``cpu_baseline`` / reference leg of ``bench.py`` may import or call this
module.  It shares no code with the CUDA library and imports nothing from it.

Plain, slow, obviously-correct restatement in float64 (numpy), following the
pages in their own order and notation.  Library primitives (matmul, exp,
sort) serve as steps; there is no blocking, fusion or reordering.

Sources cited below:

* [Paper] "Dustin: Draft-Augmented Sparse Verification for Efficient
  Long-Context Generation with Speculative Decoding" (arXiv 2606.24957), HTML
  translation page: section 3.1 gives Eq. (1)-(4), section 3.2 the
  historical-attention policy.
* [Notes] the "dustin-long-context" paper-notes page: section 2.2 (hybrid
  attention aggregation, S_Draft / S_Target, one global index set, Fig. 5),
  section 2.3 (verification set: sink, window, draft top-m, target fills the
  rest), section 2.4 (SRH sparse estimation on a few heads, Fig. 6).
* [Summary] the newx.sg abstract page (importance scoring restricted to a
  small subset of heads).

Where the pages leave a step open, the reading taken is stated at the
function.  Inputs are float64 arrays holding exact bf16 values.

Parity status: every function here is pinned by a CPU test against brute
force, closed forms, invariants or a library routine (``tests/test_oracle.py``).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

NORM_NONE = 0
NORM_L1 = 1


# ------------------------------------------------------------ attention

def softmax(logits: np.ndarray) -> np.ndarray:
    """Normalised attention weights along the last axis (they sum to 1, as
    [Paper] section 3.1 requires of A_{i,j})."""
    x = np.asarray(logits, dtype=np.float64)
    if x.shape[-1] == 0:
        return x.copy()
    peak = np.max(x, axis=-1, keepdims=True)
    e = np.exp(x - peak)
    return e / np.sum(e, axis=-1, keepdims=True)


def logsumexp(logits: np.ndarray) -> np.ndarray:
    """Natural-log normaliser of the attention row (-inf for an empty row)."""
    x = np.asarray(logits, dtype=np.float64)
    if x.shape[-1] == 0:
        return np.full(x.shape[:-1], -np.inf)
    peak = np.max(x, axis=-1)
    return peak + np.log(np.sum(np.exp(x - peak[..., None]), axis=-1))


def attention_weights(q: np.ndarray, keys: np.ndarray, scale: float
                      ) -> np.ndarray:
    """A_{i,j} = softmax_j(scale * q_i . K_j) for query rows q [..., d] over
    keys [n, d]: the full-cache attention of [Paper] section 3.1."""
    return softmax(scale * (np.asarray(q, np.float64) @ np.asarray(
        keys, np.float64).T))


# ------------------------------------------------------------ ARR, Eq. (1)-(4)

def arr(a_row: np.ndarray, selected: Iterable[int]) -> float:
    """ARR_i(pi) = sum over j in K_i^pi of A_{i,j}  ([Paper] Eq. (1))."""
    sel = np.asarray(sorted(set(int(j) for j in selected)), dtype=np.int64)
    return float(np.sum(np.asarray(a_row, np.float64)[sel])) if sel.size \
        else 0.0


def windowed_arr(a_window: np.ndarray, selected: Iterable[int]) -> float:
    """ARR_i^(w)(pi) = (1/w) sum_{s=0}^{w-1} ARR_{i+s}(pi)  ([Paper] Eq. (2)).

    a_window holds the w future attention rows A_{i+s,.} as [w][n]; the one
    selected set is scored against every row of the window."""
    a = np.asarray(a_window, np.float64)
    sel = list(selected)
    w = a.shape[0]
    return sum(arr(a[s], sel) for s in range(w)) / w


def window_mean_attention(a_window: np.ndarray) -> np.ndarray:
    """A-bar_{i,j}^(w) = (1/w) sum_s A_{i+s,j}  ([Paper] Eq. (3), left)."""
    a = np.asarray(a_window, np.float64)
    return np.sum(a, axis=0) / a.shape[0]


def sd_oracle(a_window: np.ndarray, k: int) -> Tuple[np.ndarray, float]:
    """SD oracle: K = TopK_k(A-bar) and its windowed ARR, the sum of A-bar
    over K  ([Paper] Eq. (3) right and Eq. (4)).  Returns (ascending K, ARR).
    Ties in A-bar go to the lower position (see ``topk``)."""
    abar = window_mean_attention(a_window)
    chosen = np.sort(topk(abar, k))
    return chosen, float(np.sum(abar[chosen])) if chosen.size else 0.0


# ------------------------------------------------------------ Top-K

def rank_order(values: np.ndarray, eligible: Optional[np.ndarray] = None
               ) -> np.ndarray:
    """Eligible positions in selection order.

    Reading (the pages do not say how TopK breaks ties): a total order with
    the higher value first and, among equal values, the lower position
    first; -0.0 equals +0.0; NaN ranks below every number, -inf included."""
    v = np.asarray(values, dtype=np.float64)
    pos = np.arange(v.shape[0])
    if eligible is not None:
        pos = pos[np.asarray(eligible, dtype=bool)]
    vv = v[pos]
    is_nan = np.isnan(vv)
    clean = np.where(is_nan, 0.0, vv) + 0.0        # folds -0.0 onto +0.0
    # np.lexsort: the last key is the primary key.
    order = np.lexsort((pos, -clean, is_nan.astype(np.int8)))
    return pos[order]


def topk(values: np.ndarray, k: int, eligible: Optional[np.ndarray] = None
         ) -> np.ndarray:
    """TopK_k: the first k eligible positions of ``rank_order`` (rank order,
    not sorted by position)."""
    if k <= 0:
        return np.zeros(0, dtype=np.int64)
    return rank_order(values, eligible)[:k]


# ------------------------------------------------------------ scoring

def score_heads(queries: Sequence[np.ndarray], keys: Sequence[np.ndarray],
                scale: float) -> np.ndarray:
    """Global token-importance vector over the history, [b][n].

    [Notes] section 2.2: S_Draft sums the draft's attention over its heads,
    layers and Gamma lookahead queries; S_Target sums the target's attention
    of its latest token over its heads and layers.  [Notes] section 2.4 /
    Fig. 6 and [Summary]: only a small subset of (layer, head) pairs is
    recomputed.  Reading: a plain, unweighted sum over the scored pairs and
    their query rows of the softmax over history positions [0, n).

    queries[p]: [b][rows][d] for scored pair p; keys[p]: [b][n][d], the key
    cache of that pair's layer at kv head q_head // group."""
    b, n = keys[0].shape[0], keys[0].shape[1]
    s = np.zeros((b, n), dtype=np.float64)
    for q, kk in zip(queries, keys):
        for bi in range(b):
            a = attention_weights(q[bi], kk[bi], scale)     # [rows][n]
            s[bi] += np.sum(a, axis=0)
    return s


# ------------------------------------------------------------ selection

def protected_positions(n: int, n_sink: int, n_recent: int) -> np.ndarray:
    """I_sink union I_window ([Notes] section 2.3 and Fig. 5: attention sinks
    and the recent window are always kept).  Reading: the first n_sink and
    the last n_recent history positions, overlap counted once."""
    sink = np.arange(min(max(n_sink, 0), n))
    recent = np.arange(max(n - max(n_recent, 0), 0), n)
    return np.union1d(sink, recent).astype(np.int64)


def hybrid_scores(s_draft: Optional[np.ndarray],
                  s_target: Optional[np.ndarray], alpha: float,
                  norm: int = NORM_L1) -> np.ndarray:
    """c = alpha * S_Draft-hat + (1 - alpha) * S_Target-hat for one sequence.

    Reading ([Notes] section 2.2 names the hybrid of the two vectors without
    its formula): each vector is normalised by its own sum (L1; NONE leaves
    it as is) and alpha weighs the draft signal, so alpha = 1 is the
    draft-only "Dustin-D" and alpha = 0 the target-only "Dustin-T" of
    [Notes] Table 3.

    Precision: this score decides which positions are selected, so it is
    evaluated in the selection kernel's precision.  The per-vector sum is
    taken in float64; each coefficient (alpha / sum) is rounded once to
    float32; c_j = fl32(fl32(a_D * S_D[j]) + fl32(a_T * S_T[j])) with every
    operation rounded to nearest even.  A term whose weight is 0 or whose
    vector is absent is left out; a sum that is not positive and finite
    leaves the vector unscaled."""
    terms = []
    for vec, weight in ((s_draft, alpha), (s_target, 1.0 - alpha)):
        if vec is None or weight == 0.0:
            continue
        v32 = np.asarray(vec, dtype=np.float32)
        coef = float(weight)
        if norm == NORM_L1:
            total = float(np.sum(v32.astype(np.float64)))
            if total > 0.0 and math.isfinite(total):
                coef = coef / total
        terms.append(np.float32(coef) * v32)
    if not terms:
        ref = s_draft if s_draft is not None else s_target
        return np.zeros(np.asarray(ref).shape, dtype=np.float32)
    c = terms[0]
    for t in terms[1:]:
        c = (c + t).astype(np.float32)
    return c.astype(np.float32)


def hybrid_select(s_draft: Optional[np.ndarray],
                  s_target: Optional[np.ndarray], k: int, n_sink: int,
                  n_recent: int, alpha: float = 0.5, m: int = -1,
                  norm: int = NORM_L1) -> np.ndarray:
    """The global verification index set I_verify per sequence, [b][min(k,n)]
    ascending int64 ([Notes] sections 2.2 and 2.3).

    * One set per sequence, shared by every layer and head ([Notes] 2.2).
    * k counts every kept position, protected ones included.
    * alpha mode (m < 0): protected positions, then the top
      (k - |protected|) of ``hybrid_scores`` over the other positions.
    * m mode (m >= 0, the budget split of [Notes] 2.3): protected positions,
      then the top-m of S_Draft over the unprotected positions, then the top
      (k - |protected| - m) of S_Target over what is left.  A positive
      per-vector scale cannot change an ordering, so m mode ranks the raw
      vectors (in float32, the selection kernel's precision).
    * k >= n keeps all n positions.  More protected positions than k (with
      k < n) is an error."""
    ref = s_draft if s_draft is not None else s_target
    ref = np.atleast_2d(np.asarray(ref))
    b, n = ref.shape
    sd = None if s_draft is None else np.atleast_2d(np.asarray(s_draft))
    st = None if s_target is None else np.atleast_2d(np.asarray(s_target))
    rows = []
    for bi in range(b):
        if k >= n:
            rows.append(np.arange(n, dtype=np.int64))
            continue
        forced = protected_positions(n, n_sink, n_recent)
        if forced.size > k:
            raise ValueError("protected positions exceed the budget k")
        eligible = np.ones(n, dtype=bool)
        eligible[forced] = False
        budget = k - forced.size
        if m < 0:
            c = hybrid_scores(None if sd is None else sd[bi],
                              None if st is None else st[bi], alpha, norm)
            picked = topk(c, budget, eligible)
        else:
            m_eff = min(m, budget)
            if m_eff > 0 and sd is None:
                raise ValueError("m mode needs S_Draft")
            if budget - m_eff > 0 and st is None:
                raise ValueError("m mode needs S_Target")
            p_d = topk(sd[bi].astype(np.float32), m_eff, eligible) \
                if m_eff > 0 else np.zeros(0, np.int64)
            rest = eligible.copy()
            rest[p_d] = False
            p_t = topk(st[bi].astype(np.float32), budget - m_eff, rest) \
                if budget - m_eff > 0 else np.zeros(0, np.int64)
            picked = np.concatenate([p_d, p_t])
        rows.append(np.sort(np.concatenate([forced, picked])))
    return np.stack(rows) if rows else np.zeros((0, 0), np.int64)


# ------------------------------------------------------------ verification

def verify_attention(q: np.ndarray, keys: np.ndarray, values: np.ndarray,
                     idx: Optional[np.ndarray], scale: float
                     ) -> Tuple[np.ndarray, np.ndarray]:
    """Sparse verification attention ([Notes] section 2.2 Fig. 5, Stage 2:
    the target verifies the draft tokens over the compressed KV only).

    q [b][hq][w][d]; keys, values [b][hkv][n][d]; idx [b][k] positions (None
    means all n positions: full-cache verification).  Query head h reads kv
    head h // (hq // hkv) (grouped-query attention).  For each row:
    O = softmax(scale * q . K[idx]^T) V[idx] and LSE = log sum exp(scale *
    q . K[idx]^T) (natural log).  Reading: the w rows attend to the selected
    history with no causal mask; the window's own causal block is merged by
    the caller through LSE.  An empty selection gives O = 0, LSE = -inf.
    Returns (O [b][hq][w][d], LSE [b][hq][w]) in float64."""
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    b, hq, w, d = q.shape
    hkv = keys.shape[1]
    group = hq // hkv
    out = np.zeros((b, hq, w, d), dtype=np.float64)
    lse = np.full((b, hq, w), -np.inf, dtype=np.float64)
    for bi in range(b):
        sel = np.arange(keys.shape[2]) if idx is None else \
            np.asarray(idx[bi], dtype=np.int64)
        if sel.size == 0:
            continue
        for h in range(hq):
            g = h // group
            kk = keys[bi, g][sel]
            vv = values[bi, g][sel]
            logits = scale * (q[bi, h] @ kk.T)            # [w][k]
            lse[bi, h] = logsumexp(logits)
            out[bi, h] = softmax(logits) @ vv
    return out, lse


def verify_attention_window(q: np.ndarray, keys: np.ndarray,
                            values: np.ndarray, idx: Optional[np.ndarray],
                            k_win: np.ndarray, v_win: np.ndarray, scale: float
                            ) -> Tuple[np.ndarray, np.ndarray]:
    """Verification attention of the w window rows over the selected history
    and, causally, over the window itself ([Notes] section 2.2 Fig. 5,
    Stage 2: the target scores its w draft positions in one pass; the draft
    tokens follow the history, so row t sees every selected history position
    and the window positions 0..t, as in ordinary causal decoding).

    q [b][hq][w][d]; keys, values [b][hkv][n][d]; idx [b][k] (None: all n);
    k_win, v_win [b][hkv][w][d], the window tokens' own keys and values.
    For row t of head h (kv head g = h // (hq // hkv)):
      logits = scale * q . [K[g][idx], K_win[g][0..t]]
      O = softmax(logits) [V[g][idx], V_win[g][0..t]],  LSE = log sum exp.
    Returns (O [b][hq][w][d], LSE [b][hq][w]) in float64."""
    q = np.asarray(q, np.float64)
    keys = np.asarray(keys, np.float64)
    values = np.asarray(values, np.float64)
    k_win = np.asarray(k_win, np.float64)
    v_win = np.asarray(v_win, np.float64)
    b, hq, w, d = q.shape
    hkv = keys.shape[1]
    group = hq // hkv
    out = np.zeros((b, hq, w, d), dtype=np.float64)
    lse = np.zeros((b, hq, w), dtype=np.float64)
    for bi in range(b):
        sel = np.arange(keys.shape[2]) if idx is None else \
            np.asarray(idx[bi], dtype=np.int64)
        for h in range(hq):
            g = h // group
            for t in range(w):
                kk = np.concatenate([keys[bi, g][sel], k_win[bi, g, :t + 1]])
                vv = np.concatenate([values[bi, g][sel], v_win[bi, g, :t + 1]])
                logits = scale * (kk @ q[bi, h, t])
                p = softmax(logits)
                out[bi, h, t] = p @ vv
                lse[bi, h, t] = logsumexp(logits)
    return out, lse


def full_verify_attention(q, keys, values, scale):
    """Full-cache verification (the dense baseline of [Notes] section 3,
    Fig. 7): ``verify_attention`` over every history position."""
    return verify_attention(q, keys, values, None, scale)


# ---------------------------------------------- Quest page scoring (baseline)

def quest_page_stats(keys: np.ndarray, page: int) -> np.ndarray:
    """Per-page key statistics of the Quest baseline ([Notes] section 1 and
    related work: query-aware selection that scores KV pages from cheap
    per-channel min/max key statistics instead of the exact q K^T).

    keys [b][hkv][n][d]; pages of `page` consecutive positions (the last one
    may be short).  Returns [b][hkv][P][2][d]: channel-wise minimum, then
    maximum, over the page's positions."""
    keys = np.asarray(keys, np.float64)
    b, hkv, n, d = keys.shape
    n_pages = (n + page - 1) // page
    out = np.zeros((b, hkv, n_pages, 2, d))
    for p in range(n_pages):
        blk = keys[:, :, p * page:min(n, (p + 1) * page)]
        out[:, :, p, 0] = blk.min(axis=2)
        out[:, :, p, 1] = blk.max(axis=2)
    return out


def quest_page_scores(q: np.ndarray, stats: np.ndarray) -> np.ndarray:
    """Quest's page score for each query head: the largest value q . k can
    take for a key inside the page's channel-wise box,
      score[b][h][p] = sum_c max(q_c * min_c, q_c * max_c),
    with the stats of kv head h // (hq // hkv).  q [b][hq][d]; stats as
    ``quest_page_stats``.  Returns [b][hq][P]."""
    q = np.asarray(q, np.float64)
    stats = np.asarray(stats, np.float64)
    b, hq, d = q.shape
    hkv = stats.shape[1]
    group = hq // hkv
    out = np.zeros((b, hq, stats.shape[2]))
    for h in range(hq):
        st = stats[:, h // group]                       # [b][P][2][d]
        qh = q[:, h][:, None, :]                        # [b][1][d]
        out[:, h] = np.maximum(qh * st[:, :, 0], qh * st[:, :, 1]).sum(axis=-1)
    return out


def quest_select_pages(scores: np.ndarray, n_pages_kept: int) -> np.ndarray:
    """Top pages per (sequence, head), in ascending page order ([b][hq][m]),
    with the tie order of ``rank_order``."""
    scores = np.asarray(scores, np.float64)
    b, hq, n_pages = scores.shape
    m = min(n_pages_kept, n_pages)
    out = np.zeros((b, hq, m), dtype=np.int64)
    for bi in range(b):
        for h in range(hq):
            out[bi, h] = np.sort(topk(scores[bi, h], m))
    return out


def round_to_bf16(x: np.ndarray) -> np.ndarray:
    """Round float64 values to the nearest bf16 (ties to even), returned as
    float64.  Used only to present oracle outputs in the output precision."""
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                   # x = m * 2**e, 0.5 <= |m| < 1
    scaled = np.ldexp(m, 8)              # 8 significant bits
    r = np.round(scaled)                 # numpy rounds half to even
    return np.where(np.isfinite(x), np.ldexp(r, e - 8), x)
