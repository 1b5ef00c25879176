"""Parity on the other workload shapes: the Qwen2.5-7B-shaped (b4, n8192,
h_q28/h_kv4, w4, k512) and 32B-shaped (b16, n16384, h_q40/h_kv8, w5, k1024,
heavy hitters drifted by up to 64 positions) steps, and a point of the
72B-shape sweep on a paged cache (page 16, seeded random page table).
The whole batch runs on the GPU; the first and last sequences are checked
against the CPU oracle one by one."""
import numpy as np
import pytest
import torch

from oracle import dustin_oracle as O
from sparse_kv_verification_gb300 import build, inputs as I, native as N
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _run_step(wl, page_size=None):
    """GPU scores, indices, sparse and dense attention of one layer."""
    inp = I.step_inputs(wl, DEV, n_layers=1)
    tables_t = tables_d = None
    k_t, k_d = inp.k_t, inp.k_d
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    table = None
    if page_size:
        paged_t = [I.to_paged(kk, None, page_size, seed=10 + i)
                   for i, kk in enumerate(inp.k_t)]
        paged_d = [I.to_paged(kk, None, page_size, seed=20 + i)
                   for i, kk in enumerate(inp.k_d)]
        k_t = [p[0].to(DEV) for p in paged_t]
        tables_t = [p[2].to(DEV) for p in paged_t]
        k_d = [p[0].to(DEV) for p in paged_d]
        tables_d = [p[2].to(DEV) for p in paged_d]
        pk, pv, table = I.to_paged(k, v, page_size, seed=30)
        k_att, v_att, table = pk.to(DEV), pv.to(DEV), table.to(DEV)
    else:
        k_att, v_att = k, v
    s_t = H.score(inp.q_t, k_t, inp.kvh_t, wl.scale, wl.n, page_tables=tables_t)
    s_d = H.score(inp.q_d, k_d, inp.kvh_d, wl.draft_scale, wl.n,
                  page_tables=tables_d)
    idx = H.select(s_d, s_t, wl.k, wl.n_sink, wl.n_recent, wl.alpha, wl.m, 1)
    o_s, l_s = H.sparse_attn(q, k_att, v_att, idx, wl.scale, n=wl.n,
                             page_table=table)
    o_f, l_f = H.full_attn(q, k_att, v_att, wl.scale, n=wl.n, page_table=table)
    return dict(wl=wl, inp=inp, s_t=s_t, s_d=s_d, idx=idx,
                sparse=(o_s, l_s), full=(o_f, l_f))


CASES = {
    "7b": lambda: (I.WORKLOADS["7b"], None),
    "32b_drift": lambda: (I.WORKLOADS["32b"], None),
    "sweep_paged": lambda: (I.sweep_workload(8192, 4, 8, 1024, 16), 16),
}


@pytest.fixture(scope="module", params=list(CASES))
def step(request):
    build.build()
    N.load()
    wl, page = CASES[request.param]()
    r = _run_step(wl, page)
    yield r
    del r
    torch.cuda.empty_cache()


def _sampled(wl):
    return sorted({0, wl.b - 1})


def _oracle_scores(wl, inp, b):
    q_t = [H.f64(inp.q_t[p, b:b + 1]) for p in range(wl.p_t)]
    k_t = [H.f64(k[b:b + 1, h]) for k, h in zip(inp.k_t, inp.kvh_t)]
    q_d = [H.f64(inp.q_d[p, b:b + 1]) for p in range(wl.p_d)]
    k_d = [H.f64(k[b:b + 1, h]) for k, h in zip(inp.k_d, inp.kvh_d)]
    return (O.score_heads(q_t, k_t, wl.scale),
            O.score_heads(q_d, k_d, wl.draft_scale))


def test_scores(step):
    wl, inp = step["wl"], step["inp"]
    for b in _sampled(wl):
        ref_t, ref_d = _oracle_scores(wl, inp, b)
        np.testing.assert_allclose(H.f64(step["s_t"][b:b + 1]), ref_t,
                                   rtol=2e-4, atol=1e-7)
        np.testing.assert_allclose(H.f64(step["s_d"][b:b + 1]), ref_d,
                                   rtol=2e-4, atol=1e-7)
    np.testing.assert_allclose(H.f64(step["s_t"]).sum(axis=1), wl.p_t, rtol=1e-4)
    np.testing.assert_allclose(H.f64(step["s_d"]).sum(axis=1),
                               wl.p_d * wl.gamma, rtol=1e-4)


def test_select_bit_exact_on_gpu_scores(step):
    """The oracle's selection over the GPU's own score vectors."""
    wl = step["wl"]
    want = O.hybrid_select(H.f64(step["s_d"]).astype(np.float32),
                           H.f64(step["s_t"]).astype(np.float32), wl.k,
                           wl.n_sink, wl.n_recent, wl.alpha, wl.m, O.NORM_L1)
    np.testing.assert_array_equal(step["idx"].cpu().numpy(), want)


def test_selection_quality(step):
    """Windowed ARR of GPU indices against indices from oracle scores."""
    wl, inp = step["wl"], step["inp"]
    idx_h = step["idx"].cpu().numpy()
    q, k = H.f64(inp.q[0]), H.f64(inp.k[0])
    for b in _sampled(wl):
        ref_t, ref_d = _oracle_scores(wl, inp, b)
        ref_idx = O.hybrid_select(ref_d, ref_t, wl.k, wl.n_sink, wl.n_recent,
                                  wl.alpha, wl.m, O.NORM_L1)[0]
        got, want = [], []
        for h in range(wl.hq):
            a = O.attention_weights(q[b, h], k[b, h // wl.group], wl.scale)
            got.append(O.windowed_arr(a, idx_h[b]))
            want.append(O.windowed_arr(a, ref_idx))
        assert abs(np.mean(got) - np.mean(want)) <= H.ARR_TOL
        assert np.mean(got) > wl.k / wl.n


def test_sparse_attention(step):
    wl, inp = step["wl"], step["inp"]
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    o, lse = step["sparse"]
    idx = step["idx"].cpu().numpy()
    for b in _sampled(wl):
        o_ref, l_ref = O.verify_attention(H.f64(q[b:b + 1]), H.f64(k[b:b + 1]),
                                          H.f64(v[b:b + 1]), idx[b:b + 1],
                                          wl.scale)
        H.assert_attn_close(o[b:b + 1], lse[b:b + 1], o_ref, l_ref)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()


def test_full_attention(step):
    wl, inp = step["wl"], step["inp"]
    q, k, v = inp.q[0], inp.k[0], inp.v[0]
    o, lse = step["full"]
    for b in _sampled(wl):
        o_ref, l_ref = O.full_verify_attention(H.f64(q[b:b + 1]),
                                               H.f64(k[b:b + 1]),
                                               H.f64(v[b:b + 1]), wl.scale)
        H.assert_attn_close(o[b:b + 1], lse[b:b + 1], o_ref, l_ref)


@pytest.mark.parametrize("k", [8192, 16384])
def test_attention_at_the_longest_context(k):
    """n = 65536 (the longest supported context), 72B head shape, k up to
    a quarter of it: sparse and dense attention against the oracle."""
    build.build()
    N.load()
    b, hq, hkv, d, w, n = 2, 64, 8, 128, 5, 65536
    g = I.generator(k)
    q = torch.randn((b, hq, w, d), generator=g).to(torch.bfloat16)
    kk = torch.randn((b, hkv, n, d), generator=g).to(torch.bfloat16)
    v = torch.randn((b, hkv, n, d), generator=g).to(torch.bfloat16)
    idx = I.random_sorted_indices(b, n, k, seed=k + 1)
    scale = d ** -0.5
    o, lse = H.sparse_attn(q.to(DEV), kk.to(DEV), v.to(DEV), idx.to(DEV), scale)
    o_f, l_f = H.full_attn(q.to(DEV), kk.to(DEV), v.to(DEV), scale)
    assert N.dustin_device_status() == 0
    for bb in range(b):
        o_ref, l_ref = O.verify_attention(H.f64(q[bb:bb + 1]), H.f64(kk[bb:bb + 1]),
                                          H.f64(v[bb:bb + 1]), idx[bb:bb + 1].numpy(),
                                          scale)
        H.assert_attn_close(o[bb:bb + 1], lse[bb:bb + 1], o_ref, l_ref)
    o_ref, l_ref = O.full_verify_attention(H.f64(q[:1]), H.f64(kk[:1]), H.f64(v[:1]),
                                           scale)
    H.assert_attn_close(o_f[:1], l_f[:1], o_ref, l_ref)
