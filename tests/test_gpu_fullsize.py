"""Parity at the full Qwen2.5-72B-shaped sizes (b16, n32768, h_q64/h_kv8,
d128, w5, k2048, 4 + 4 scored pairs), in the launch configuration bench.py
times: the whole batch runs on the GPU and sampled sequences are checked
against the CPU oracle one by one."""
import numpy as np
import pytest
import torch

from oracle import dustin_oracle as O
from sparse_kv_verification_gb300 import build, inputs as I, native as N
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = "cuda"
SAMPLED = (0, 11)


@pytest.fixture(scope="module")
def step():
    build.build()
    N.load()
    wl = I.WORKLOADS["72b"]
    inp = I.step_inputs(wl, DEV, n_layers=2)
    s_t = H.score(inp.q_t, inp.k_t, inp.kvh_t, wl.scale, wl.n)
    s_d = H.score(inp.q_d, inp.k_d, inp.kvh_d, wl.draft_scale, wl.n)
    idx = H.select(s_d, s_t, wl.k, wl.n_sink, wl.n_recent, wl.alpha, -1, 1)
    yield wl, inp, s_t, s_d, idx
    del inp
    torch.cuda.empty_cache()


def oracle_scores(wl, inp, b):
    q_t = [H.f64(inp.q_t[p, b:b + 1]) for p in range(wl.p_t)]
    k_t = [H.f64(k[b:b + 1, h]) for k, h in zip(inp.k_t, inp.kvh_t)]
    q_d = [H.f64(inp.q_d[p, b:b + 1]) for p in range(wl.p_d)]
    k_d = [H.f64(k[b:b + 1, h]) for k, h in zip(inp.k_d, inp.kvh_d)]
    return (O.score_heads(q_t, k_t, wl.scale),
            O.score_heads(q_d, k_d, wl.draft_scale))


def test_scores_full_size(step):
    wl, inp, s_t, s_d, _ = step
    for b in SAMPLED:
        ref_t, ref_d = oracle_scores(wl, inp, b)
        np.testing.assert_allclose(H.f64(s_t[b:b + 1]), ref_t, rtol=2e-4,
                                   atol=1e-7)
        np.testing.assert_allclose(H.f64(s_d[b:b + 1]), ref_d, rtol=2e-4,
                                   atol=1e-7)
    sums = H.f64(s_t).sum(axis=1)
    np.testing.assert_allclose(sums, wl.p_t, rtol=1e-4)


def test_select_full_size_bit_exact():
    wl = I.WORKLOADS["72b"]
    sd = I.synthetic_scores(wl.b, wl.n, seed=72, specials=True)
    st = I.synthetic_scores(wl.b, wl.n, seed=73)
    got = H.select(sd.to(DEV), st.to(DEV), wl.k, wl.n_sink, wl.n_recent,
                   wl.alpha, -1, 1)
    want = O.hybrid_select(sd.numpy(), st.numpy(), wl.k, wl.n_sink,
                           wl.n_recent, wl.alpha, -1, O.NORM_L1)
    np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_selection_quality_matches_oracle_arr(step):
    """Indices from GPU scores against indices from oracle scores: windowed
    ARR of the timed layer (mean over heads) agrees within 1e-5."""
    wl, inp, _, _, idx = step
    idx_h = idx.cpu().numpy()
    assert np.all(np.diff(idx_h, axis=1) > 0) and idx_h.shape == (wl.b, wl.k)
    forced = O.protected_positions(wl.n, wl.n_sink, wl.n_recent)
    for b in SAMPLED:
        assert set(forced.tolist()) <= set(idx_h[b].tolist())
        ref_t, ref_d = oracle_scores(wl, inp, b)
        ref_idx = O.hybrid_select(ref_d, ref_t, wl.k, wl.n_sink, wl.n_recent,
                                  wl.alpha, -1, O.NORM_L1)[0]
        q = H.f64(inp.q[0][b])
        k = H.f64(inp.k[0][b])
        got, want = [], []
        for h in range(wl.hq):
            a = O.attention_weights(q[h], k[h // wl.group], wl.scale)
            got.append(O.windowed_arr(a, idx_h[b]))
            want.append(O.windowed_arr(a, ref_idx))
        assert abs(np.mean(got) - np.mean(want)) <= H.ARR_TOL
        # Better than a uniform random subset (expected ARR k / n), and at
        # most the SD oracle (Eq. 3-4) of every head's window.
        assert np.mean(got) > wl.k / wl.n
        best = [O.sd_oracle(O.attention_weights(q[h], k[h // wl.group],
                                                wl.scale), wl.k)[1]
                for h in range(0, wl.hq, 8)]
        assert all(g <= s + 1e-12 for g, s in zip(got[::8], best))


def test_sparse_attention_full_size(step):
    wl, inp, _, _, idx = step
    q, k, v = inp.q[1], inp.k[1], inp.v[1]
    o, lse = H.sparse_attn(q, k, v, idx, wl.scale)
    for b in SAMPLED:
        o_ref, l_ref = O.verify_attention(
            H.f64(q[b:b + 1]), H.f64(k[b:b + 1]), H.f64(v[b:b + 1]),
            idx[b:b + 1].cpu().numpy(), wl.scale)
        H.assert_attn_close(o[b:b + 1], lse[b:b + 1], o_ref, l_ref)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_full_attention_full_size(step):
    wl, inp, _, _, _ = step
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    o, lse = H.full_attn(q, k, v, wl.scale)
    for b in SAMPLED:
        o_ref, l_ref = O.full_verify_attention(
            H.f64(q[b:b + 1]), H.f64(k[b:b + 1]), H.f64(v[b:b + 1]), wl.scale)
        H.assert_attn_close(o[b:b + 1], lse[b:b + 1], o_ref, l_ref)
