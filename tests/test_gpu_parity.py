"""GPU parity: the CUDA path (through the C-ABI) against the CPU oracle on
the same seeded inputs, at sizes the oracle finishes in seconds that span
several tiles, ragged tails, every kernel variant and the edge cases."""
import numpy as np
import pytest
import torch

from oracle import dustin_oracle as O
from sparse_kv_verification_gb300 import build, inputs as I, native as N
from tests import gpu_harness as H

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module", autouse=True)
def lib():
    build.build()
    return N.load()


def qkv(b, hq, hkv, d, w, n, seed):
    g = I.generator(seed)
    q = torch.randn((b, hq, w, d), generator=g).to(torch.bfloat16)
    k = torch.randn((b, hkv, n, d), generator=g).to(torch.bfloat16)
    v = torch.randn((b, hkv, n, d), generator=g).to(torch.bfloat16)
    return q, k, v


# (b, h_q, h_kv, d, w, n, k): 16-row tiles 1..4, two row blocks, d 64/128,
# ragged n and k; one unit cut into ~70 position splits (sparse) or spread
# over ~80 CTAs one tile each (dense); k past the 2048-row offset table of
# one CTA; more units than resident CTAs (dense CTA ranges that hold the end
# of one unit, whole units and the start of another).
SHAPES = [
    (1, 4, 2, 64, 4, 256, 32),
    (2, 28, 4, 128, 4, 700, 131),
    (3, 40, 8, 128, 5, 1000, 333),
    (2, 64, 8, 128, 5, 3000, 1100),
    (1, 64, 8, 128, 8, 2048, 600),
    (1, 64, 4, 64, 5, 900, 450),
    (1, 8, 1, 128, 3, 5000, 4500),
    (4, 14, 2, 64, 4, 129, 65),
    (48, 32, 8, 128, 2, 600, 300),
    (40, 16, 4, 64, 3, 400, 130),
    # k past 4096 with enough units for one CTA each: one row table of
    # 5000 positions per CTA (d 128) and 7000 (d 64, two row tiles)
    (16, 16, 8, 128, 2, 6000, 5000),
    (12, 56, 8, 64, 4, 7500, 7000),
]


@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_sparse_attention_parity(shape):
    b, hq, hkv, d, w, n, k = shape
    q, kk, v = qkv(b, hq, hkv, d, w, n, seed=sum(shape))
    idx = I.random_sorted_indices(b, n, k, seed=k + n)
    scale = d ** -0.5
    o, lse = H.sparse_attn(q.to(DEV), kk.to(DEV), v.to(DEV), idx.to(DEV), scale)
    o_ref, lse_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                        idx.numpy(), scale)
    H.assert_attn_close(o, lse, o_ref, lse_ref)


DENSE_SHAPES = SHAPES[:6] + SHAPES[8:10]


@pytest.mark.parametrize("shape", DENSE_SHAPES, ids=[str(s) for s in DENSE_SHAPES])
def test_full_attention_parity(shape):
    b, hq, hkv, d, w, n, _ = shape
    q, kk, v = qkv(b, hq, hkv, d, w, n, seed=sum(shape) + 1)
    scale = d ** -0.5
    o, lse = H.full_attn(q.to(DEV), kk.to(DEV), v.to(DEV), scale)
    o_ref, lse_ref = O.full_verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                             scale)
    H.assert_attn_close(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("shape", [SHAPES[6], SHAPES[8]], ids=["one-unit", "many-units"])
def test_reused_workspace_gives_identical_results(shape):
    """Dense units shared between CTAs are merged through per-unit counters
    kept in the workspace.  A workspace full of 0xff bytes, reused over
    several calls (sparse and dense alternating), must give bit-identical
    outputs: the merge order is fixed whichever CTA finishes a unit last."""
    b, hq, hkv, d, w, n, k = shape
    q, kk, v = (t.to(DEV) for t in qkv(b, hq, hkv, d, w, n, seed=77))
    idx = I.random_sorted_indices(b, n, k, seed=78).to(DEV)
    desc = N.kv_desc(kk, v)
    nbytes = max(N.dustin_sparse_verify_attn_workspace_size(b, hq, hkv, d, w, k),
                 N.dustin_full_verify_attn_workspace_size(b, hq, hkv, d, w, n))
    ws = N.workspace(nbytes, DEV)
    ws.fill_(255)
    outs = []
    for rep in range(3):
        o = torch.full_like(q, float("nan"))
        lse = torch.full((b, hq, w), float("nan"), device=DEV)
        N.dustin_sparse_verify_attn(q, desc, hkv, n, idx, 0.1, o, lse, ws)
        fo = torch.full_like(q, float("nan"))
        flse = torch.full((b, hq, w), float("nan"), device=DEV)
        N.dustin_full_verify_attn(q, desc, hkv, n, 0.1, fo, flse, ws)
        H.sync()
        outs.append((o, lse, fo, flse))
    assert N.dustin_device_status() == 0
    for later in outs[1:]:
        assert all(torch.equal(x, y) for x, y in zip(outs[0], later))
    o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                      idx.cpu().numpy(), 0.1)
    H.assert_attn_close(outs[0][0], outs[0][1], o_ref, l_ref)


@pytest.mark.parametrize("case", ["contiguous", "paged", "split"])
def test_kv_ready_launch_overlap_gives_identical_results(case):
    """DUSTIN_ATTN_KV_READY lets a launch gather K/V while the kernel before
    it on the stream still runs.  Consecutive layers over one index set
    (layer 0 after a kernel that writes idx, so without the flag), back to
    back on one stream, must give the same bits as calls without it."""
    b, hq, hkv, d, w, n, k = {"contiguous": (4, 32, 4, 128, 5, 3000, 700),
                              "paged": (2, 16, 2, 128, 4, 1000, 300),
                              "split": (1, 8, 1, 128, 3, 5000, 4500)}[case]
    layers = 4
    idx = I.random_sorted_indices(b, n, k, seed=21).to(DEV)
    qs, descs, keep = [], [], []
    for l in range(layers):
        q, kk, v = qkv(b, hq, hkv, d, w, n, seed=100 + l)
        if case == "paged":
            kk, v, table = I.to_paged(kk, v, 16, seed=200 + l)
            table = table.to(DEV)
        else:
            table = None
        q, kk, v = q.to(DEV), kk.to(DEV), v.to(DEV)
        keep += [kk, v, table]
        qs.append(q)
        descs.append(N.kv_desc(kk, v, table))
    ws_s = N.workspace(N.dustin_sparse_verify_attn_workspace_size(b, hq, hkv, d, w, k), DEV)
    ws_f = N.workspace(N.dustin_full_verify_attn_workspace_size(b, hq, hkv, d, w, n), DEV)

    def run(ready):
        outs = []
        for dense in (False, True):
            for l in range(layers):
                o = torch.full_like(qs[l], float("nan"))
                lse = torch.full((b, hq, w), float("nan"), device=DEV)
                flags = N.DUSTIN_ATTN_KV_READY if ready and l > 0 else 0
                if dense:
                    N.dustin_full_verify_attn(qs[l], descs[l], hkv, n, 0.1, o, lse,
                                              ws_f, flags=flags)
                else:
                    N.dustin_sparse_verify_attn(qs[l], descs[l], hkv, n, idx, 0.1,
                                                o, lse, ws_s, flags=flags)
                outs.append((o, lse))
        H.sync()
        return outs

    plain, ready = run(False), run(True)
    assert N.dustin_device_status() == 0
    for (o1, l1), (o2, l2) in zip(plain, ready):
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


# ------------------------------------------- window causal block merged in

WINDOW_SHAPES = [SHAPES[0], SHAPES[2], SHAPES[4], SHAPES[6], SHAPES[9],
                 (2, 16, 2, 128, 4, 40, 0), SHAPES[10]]


@pytest.mark.parametrize("shape", WINDOW_SHAPES, ids=[str(s) for s in WINDOW_SHAPES])
def test_window_attention_parity(shape):
    """History over idx (sparse) or all n (dense) plus the window's own
    causal block, in one launch, against the oracle.  Covers several row
    blocks, position splits, the dense stream-K ranges and k = 0."""
    b, hq, hkv, d, w, n, k = shape
    q, kk, v = qkv(b, hq, hkv, d, w, n, seed=sum(shape) + 7)
    _, kw, vw = qkv(b, hq, hkv, d, w, w, seed=sum(shape) + 8)
    idx = I.random_sorted_indices(b, n, k, seed=k + n + 1) if k else \
        torch.zeros((b, 0), dtype=torch.int32)
    dq, dk, dv, dkw, dvw = (t.to(DEV) for t in (q, kk, v, kw, vw))
    scale = d ** -0.5
    o, lse = H.sparse_attn_window(dq, dk, dv, idx.to(DEV), dkw, dvw, scale)
    o_ref, l_ref = O.verify_attention_window(H.f64(q), H.f64(kk), H.f64(v),
                                             idx.numpy(), H.f64(kw), H.f64(vw),
                                             scale)
    H.assert_attn_close(o, lse, o_ref, l_ref)
    if k:   # the dense call (k = 0 is a sparse-only case)
        o, lse = H.full_attn_window(dq, dk, dv, dkw, dvw, scale)
        o_ref, l_ref = O.verify_attention_window(H.f64(q), H.f64(kk), H.f64(v),
                                                 None, H.f64(kw), H.f64(vw),
                                                 scale)
        H.assert_attn_close(o, lse, o_ref, l_ref)
    assert N.dustin_device_status() == 0


def test_window_attention_paged_and_kv_ready():
    b, hq, hkv, d, w, n, k = 2, 16, 2, 128, 4, 1000, 300
    q, kk, v = qkv(b, hq, hkv, d, w, n, seed=31)
    _, kw, vw = qkv(b, hq, hkv, d, w, w, seed=32)
    pk, pv, table = I.to_paged(kk, v, 16, seed=33)
    idx = I.random_sorted_indices(b, n, k, seed=34).to(DEV)
    dq, dkw, dvw = q.to(DEV), kw.to(DEV), vw.to(DEV)
    o_c, l_c = H.sparse_attn_window(dq, kk.to(DEV), v.to(DEV), idx, dkw, dvw, 0.1)
    o_p, l_p = H.sparse_attn_window(dq, pk.to(DEV), pv.to(DEV), idx, dkw, dvw, 0.1,
                                    n=n, page_table=table.to(DEV),
                                    flags=N.DUSTIN_ATTN_KV_READY)
    assert torch.equal(o_c, o_p) and torch.equal(l_c, l_p)
    f_c, fl_c = H.full_attn_window(dq, kk.to(DEV), v.to(DEV), dkw, dvw, 0.1)
    f_p, fl_p = H.full_attn_window(dq, pk.to(DEV), pv.to(DEV), dkw, dvw, 0.1, n=n,
                                   page_table=table.to(DEV),
                                   flags=N.DUSTIN_ATTN_KV_READY)
    assert torch.equal(f_c, f_p) and torch.equal(fl_c, fl_p)
    o_ref, l_ref = O.verify_attention_window(H.f64(q), H.f64(kk), H.f64(v),
                                             idx.cpu().numpy(), H.f64(kw),
                                             H.f64(vw), 0.1)
    H.assert_attn_close(o_p, l_p, o_ref, l_ref)
    assert N.dustin_device_status() == 0


# ---------------------------------------- several layers in one launch

@pytest.mark.parametrize("shape,layers,paged", [
    ((2, 28, 4, 128, 4, 700, 131), 3, False),
    ((3, 40, 8, 128, 5, 1000, 333), 4, True),
    ((1, 64, 4, 64, 5, 900, 450), 2, False),
    ((4, 14, 2, 64, 4, 129, 0), 2, False),
    ((48, 32, 8, 128, 2, 600, 300), 3, False),
], ids=["3x-rows4", "4x-paged", "2x-d64", "k0", "many-units"])
def test_multi_layer_launch_matches_per_layer_calls(shape, layers, paged):
    """Every layer of the persistent multi-layer launch gives the same bits
    as its own per-layer call (same tiles, same math and merge order), and
    matches the oracle."""
    b, hq, hkv, d, w, n, k = shape
    idx = (I.random_sorted_indices(b, n, k, seed=41) if k else
           torch.zeros((b, 0), dtype=torch.int32)).to(DEV)
    qs, descs, keep, host = [], [], [], []
    for l in range(layers):
        q, kk, v = qkv(b, hq, hkv, d, w, n, seed=300 + l)
        host.append((q, kk, v))
        table = None
        if paged:
            kk, v, table = I.to_paged(kk, v, 16, seed=400 + l)
            table = table.to(DEV)
        q, kk, v = q.to(DEV), kk.to(DEV), v.to(DEV)
        keep += [kk, v, table]
        qs.append(q)
        descs.append(N.kv_desc(kk, v, table))
    os = [torch.full_like(q, float("nan")) for q in qs]
    lses = [torch.full((b, hq, w), float("nan"), device=DEV) for _ in qs]
    N.dustin_sparse_verify_attn_layers(qs, descs, hkv, n, idx, 0.1, os, lses)
    H.sync()
    assert N.dustin_device_status() == 0
    ws = N.workspace(N.dustin_sparse_verify_attn_workspace_size(b, hq, hkv, d, w, k), DEV)
    for l in range(layers):
        o1 = torch.full_like(qs[l], float("nan"))
        l1 = torch.full((b, hq, w), float("nan"), device=DEV)
        N.dustin_sparse_verify_attn(qs[l], descs[l], hkv, n, idx, 0.1, o1, l1, ws)
        H.sync()
        if k == 0 or N.dustin_sparse_verify_attn_workspace_size(b, hq, hkv, d, w, k) <= 1:
            assert torch.equal(os[l], o1) and torch.equal(lses[l], l1)
        q, kk, v = host[l]
        o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                          idx.cpu().numpy(), 0.1)
        H.assert_attn_close(os[l], lses[l], o_ref, l_ref)


# ---------------------------------------- Quest page scoring (baseline)

@pytest.mark.parametrize("b,hq,hkv,d,n,page", [(2, 8, 2, 128, 1000, 16),
                                               (3, 14, 2, 64, 777, 32),
                                               (1, 64, 8, 128, 4096, 16)])
def test_quest_page_scoring_parity(b, hq, hkv, d, n, page):
    """Stats are exact (min/max of bf16 values); scores within fp32
    rounding; the top pages picked by the selection kernel from the GPU
    scores equal the oracle's page selection on the same scores; paged keys
    give the same stats bits."""
    g = I.generator(n + page)
    k = (2.0 * torch.randn((b, hkv, n, d), generator=g)).to(torch.bfloat16)
    q = torch.randn((b, hq, d), generator=g).to(torch.bfloat16)
    dk, dq = k.to(DEV), q.to(DEV)
    st = N.dustin_quest_page_stats(N.kv_desc(dk), b, hkv, d, n, page, device=DEV)
    sc = N.dustin_quest_page_scores(dq, st, n, page)
    H.sync()
    st_ref = O.quest_page_stats(H.f64(k), page)
    np.testing.assert_array_equal(H.f64(st), st_ref)
    sc_ref = O.quest_page_scores(H.f64(q), st_ref)
    np.testing.assert_allclose(H.f64(sc), sc_ref, rtol=1e-5, atol=1e-4)
    n_pages = st.shape[2]
    keep = max(1, n_pages // 8)
    rows = sc.reshape(b * hq, n_pages).contiguous()
    got = H.select(rows, None, keep, 0, 0, 1.0, -1, 0)
    want = O.quest_select_pages(H.f64(sc), keep).reshape(b * hq, -1)
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    pk, _, table = I.to_paged(k, None, 16, seed=5)
    dpk, dtable = pk.to(DEV), table.to(DEV)     # alive while the kernel runs
    st_p = N.dustin_quest_page_stats(N.kv_desc(dpk, None, dtable), b,
                                     hkv, d, n, page, device=DEV)
    H.sync()
    assert torch.equal(st, st_p)
    assert N.dustin_device_status() == 0


def test_multi_layer_launch_beyond_one_launch_of_layers():
    """More layers than one launch carries (128): the call splits them into
    launches; every layer still matches its own per-layer call bit for bit."""
    b, hq, hkv, d, w, n, k, layers = 1, 4, 2, 64, 2, 100, 30, 130
    idx = I.random_sorted_indices(b, n, k, seed=43).to(DEV)
    g = I.generator(44)
    qs = [torch.randn((b, hq, w, d), generator=g).to(torch.bfloat16).to(DEV)
          for _ in range(layers)]
    ks = [torch.randn((b, hkv, n, d), generator=g).to(torch.bfloat16).to(DEV)
          for _ in range(layers)]
    vs = [torch.randn((b, hkv, n, d), generator=g).to(torch.bfloat16).to(DEV)
          for _ in range(layers)]
    descs = [N.kv_desc(kk, vv) for kk, vv in zip(ks, vs)]
    os = [torch.full_like(q, float("nan")) for q in qs]
    lses = [torch.full((b, hq, w), float("nan"), device=DEV) for _ in qs]
    N.dustin_sparse_verify_attn_layers(qs, descs, hkv, n, idx, 0.2, os, lses)
    H.sync()
    ws = N.workspace(N.dustin_sparse_verify_attn_workspace_size(b, hq, hkv, d, w, k), DEV)
    for l in (0, 1, 127, 128, 129):
        o1 = torch.full_like(qs[l], float("nan"))
        l1 = torch.full((b, hq, w), float("nan"), device=DEV)
        N.dustin_sparse_verify_attn(qs[l], descs[l], hkv, n, idx, 0.2, o1, l1, ws)
        H.sync()
        if N.dustin_sparse_verify_attn_workspace_size(b, hq, hkv, d, w, k) <= 1:
            assert torch.equal(os[l], o1) and torch.equal(lses[l], l1)
        else:
            assert (os[l].float() - o1.float()).abs().max().item() <= 1e-2
    assert N.dustin_device_status() == 0


def test_sparse_with_all_positions_matches_full():
    b, hq, hkv, d, w, n = 2, 16, 2, 128, 4, 777
    q, kk, v = qkv(b, hq, hkv, d, w, n, seed=5)
    q, kk, v = q.to(DEV), kk.to(DEV), v.to(DEV)
    idx = torch.arange(n, dtype=torch.int32, device=DEV).repeat(b, 1)
    o1, l1 = H.sparse_attn(q, kk, v, idx.contiguous(), 0.1)
    o2, l2 = H.full_attn(q, kk, v, 0.1)
    assert (o1.float() - o2.float()).abs().max().item() <= 1e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


@pytest.mark.parametrize("page,shape", [(16, (2, 16, 2, 128, 4, 1000, 300)),
                                        (32, (2, 16, 2, 128, 4, 1000, 300)),
                                        (16, (16, 16, 8, 128, 2, 6000, 5000))],
                         ids=["p16", "p32", "p16-k5000"])
def test_paged_layout_matches_contiguous_and_oracle(page, shape):
    b, hq, hkv, d, w, n, k = shape
    q, kk, v = qkv(b, hq, hkv, d, w, n, seed=page)
    pk, pv, table = I.to_paged(kk, v, page, seed=page + 1)
    idx = I.random_sorted_indices(b, n, k, seed=3).to(DEV)
    qd = q.to(DEV)
    o_c, l_c = H.sparse_attn(qd, kk.to(DEV), v.to(DEV), idx, 0.1)
    o_p, l_p = H.sparse_attn(qd, pk.to(DEV), pv.to(DEV), idx, 0.1, n=n,
                             page_table=table.to(DEV))
    assert torch.equal(o_c, o_p) and torch.equal(l_c, l_p)
    o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                      idx.cpu().numpy(), 0.1)
    H.assert_attn_close(o_p, l_p, o_ref, l_ref)
    f_c, fl_c = H.full_attn(qd, kk.to(DEV), v.to(DEV), 0.1)
    f_p, fl_p = H.full_attn(qd, pk.to(DEV), pv.to(DEV), 0.1, n=n,
                            page_table=table.to(DEV))
    assert torch.equal(f_c, f_p) and torch.equal(fl_c, fl_p)


def test_attention_edge_cases():
    q, kk, v = qkv(2, 8, 2, 64, 3, 50, seed=9)
    q, kk, v = q.to(DEV), kk.to(DEV), v.to(DEV)
    # k = 0: empty selection gives O = 0, LSE = -inf.
    o, lse = H.sparse_attn(q, kk, v, torch.zeros((2, 0), dtype=torch.int32,
                                                 device=DEV), 0.2)
    assert torch.all(o == 0) and torch.all(lse == float("-inf"))
    # n smaller than one tile, k = n.
    idx = torch.arange(50, dtype=torch.int32, device=DEV).repeat(2, 1)
    o, lse = H.sparse_attn(q, kk, v, idx.contiguous(), 0.2)
    o_ref, l_ref = O.full_verify_attention(H.f64(q), H.f64(kk), H.f64(v), 0.2)
    H.assert_attn_close(o, lse, o_ref, l_ref)
    # One position only.
    one = torch.tensor([[7], [49]], dtype=torch.int32, device=DEV)
    o, lse = H.sparse_attn(q, kk, v, one, 0.2)
    o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                      one.cpu().numpy(), 0.2)
    H.assert_attn_close(o, lse, o_ref, l_ref)


def test_bounded_wait_gives_up_and_leaves_the_context_usable():
    """A wait that nothing ends (an mbarrier no thread arrives at), with the
    bounded wait every pipeline of the library uses: it gives up after its
    limit, raises the timeout flag, and the next call runs normally."""
    N.dustin_device_status()                     # clear old flags
    N.dustin_wait_selftest(2_000_000)            # about a millisecond
    assert N.dustin_device_status() == 4         # DUSTIN_DEVFLAG_WAIT_TIMEOUT
    assert N.dustin_device_status() == 0         # read clears
    q, kk, v = qkv(1, 4, 1, 64, 2, 100, seed=12)
    idx = torch.tensor([[3, 10, 50]], dtype=torch.int32)
    o, lse = H.sparse_attn(q.to(DEV), kk.to(DEV), v.to(DEV), idx.to(DEV), 0.2)
    assert N.dustin_device_status() == 0
    o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                      idx.numpy(), 0.2)
    H.assert_attn_close(o, lse, o_ref, l_ref)


def test_out_of_range_index_is_flagged_not_faulted():
    """The kernel's own bounds check: an index >= n is left out of the
    attention and raises a device flag; no access goes out of bounds."""
    q, kk, v = qkv(1, 4, 1, 64, 2, 100, seed=11)
    N.dustin_device_status()                     # clear old flags
    idx = torch.tensor([[3, 10, 200, 50]], dtype=torch.int32)
    o, lse = H.sparse_attn(q.to(DEV), kk.to(DEV), v.to(DEV), idx.to(DEV), 0.2)
    flags = N.dustin_device_status()
    assert flags & 1
    o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(kk), H.f64(v),
                                      np.array([[3, 10, 50]]), 0.2)
    H.assert_attn_close(o, lse, o_ref, l_ref)
    assert N.dustin_device_status() == 0          # read clears


# ---------------------------------------------------------------- scoring

@pytest.mark.parametrize("p,b,rows,d,n", [(4, 2, 1, 128, 3000),
                                          (3, 2, 4, 64, 1000),
                                          (2, 1, 16, 128, 200),
                                          (1, 3, 3, 64, 4097)])
def test_score_heads_parity(p, b, rows, d, n):
    g = I.generator(p * 100 + n)
    q = torch.randn((p, b, rows, d), generator=g).to(torch.bfloat16)
    hkv = 3
    keys = [(2.0 * torch.randn((b, hkv, n, d), generator=g)).to(torch.bfloat16)
            for _ in range(p)]
    heads = [i % hkv for i in range(p)]
    scale = d ** -0.5
    s = H.score(q.to(DEV), [k.to(DEV) for k in keys], heads, scale, n)
    ref = O.score_heads([H.f64(q[i]) for i in range(p)],
                        [H.f64(keys[i][:, heads[i]]) for i in range(p)], scale)
    np.testing.assert_allclose(H.f64(s), ref, rtol=2e-4, atol=1e-7)
    np.testing.assert_allclose(H.f64(s).sum(axis=1), p * rows, rtol=1e-4)


@pytest.mark.parametrize("pairs,hkv,rows,d,n,b", [(64, 8, 1, 128, 8192, 2),
                                                  (14, 2, 4, 64, 8192, 3)],
                         ids=["target-all-heads", "draft-all-heads"])
def test_score_heads_naive_estimator_shapes(pairs, hkv, rows, d, n, b):
    """The naive estimator ([Paper] section 1, [Notes] section 3 Fig. 8)
    scores every query head of a layer: 64 target heads with the latest
    token's row, or the draft's 14 heads with its lookahead rows.  The
    pairs then share their kv heads' keys (pairs // hkv siblings each),
    which selects the kernel's shared-keys L2 policy; every element against
    the oracle at the scoring tolerance."""
    g = I.generator(pairs * 1000 + n)
    keys = (2.0 * torch.randn((b, hkv, n, d), generator=g)).to(torch.bfloat16)
    q = torch.randn((pairs, b, rows, d), generator=g).to(torch.bfloat16)
    group = pairs // hkv
    heads = [h // group for h in range(pairs)]
    scale = d ** -0.5
    dk = keys.to(DEV)
    s = H.score(q.to(DEV), [dk] * pairs, heads, scale, n)
    ref = O.score_heads([H.f64(q[i]) for i in range(pairs)],
                        [H.f64(keys[:, heads[i]]) for i in range(pairs)], scale)
    np.testing.assert_allclose(H.f64(s), ref, rtol=2e-4, atol=1e-7)
    np.testing.assert_allclose(H.f64(s).sum(axis=1), pairs * rows, rtol=1e-4)
    assert N.dustin_device_status() == 0


@pytest.mark.parametrize("page,d,rows", [(16, 128, 2), (32, 128, 1), (64, 64, 4),
                                          (16, 64, 5), (48, 128, 2), (128, 64, 3)])
def test_score_heads_paged_matches_contiguous(page, d, rows):
    """Paged keys give the contiguous scores bit for bit (page sizes 16, 32
    and 64 load one page per TMA box; 48 and 128 go to the cp.async
    kernel)."""
    p, b, n = 2, 2, 1500
    g = I.generator(77 + page + d)
    q = torch.randn((p, b, rows, d), generator=g).to(torch.bfloat16).to(DEV)
    keys = [torch.randn((b, 2, n, d), generator=g).to(torch.bfloat16)
            for _ in range(p)]
    paged = [I.to_paged(k, None, page, seed=i) for i, k in enumerate(keys)]
    s_c = H.score(q, [k.to(DEV) for k in keys], [0, 1], 0.1, n)
    s_p = H.score(q, [pk.to(DEV) for pk, _, _ in paged], [0, 1], 0.1, n,
                  page_tables=[t.to(DEV) for _, _, t in paged])
    assert torch.equal(s_c, s_p)
    assert N.dustin_device_status() == 0


@pytest.mark.parametrize("page", [16, 48])
def test_score_heads_bad_page_left_out(page):
    """A page id outside the pool raises flag 0x2 and its positions are left
    out: they score 0 and the rest is the softmax over the other positions."""
    p, b, rows, d, n = 1, 2, 3, 128, 700
    g = I.generator(500 + page)
    q = torch.randn((p, b, rows, d), generator=g).to(torch.bfloat16)
    k = torch.randn((b, 1, n, d), generator=g).to(torch.bfloat16)
    pk, _, table = I.to_paged(k, None, page, seed=9)
    bad_seq, bad_page = 1, 3
    table[bad_seq, bad_page] = pk.shape[0] + 5
    s = H.score(q.to(DEV), [pk.to(DEV)], [0], 0.1, n, page_tables=[table.to(DEV)])
    assert N.dustin_device_status() & 2
    gone = np.arange(bad_page * page, min(n, (bad_page + 1) * page))
    keep = np.setdiff1d(np.arange(n), gone)
    for bb in range(b):
        kb = H.f64(k[bb:bb + 1, 0])
        cols = keep if bb == bad_seq else np.arange(n)
        ref = np.zeros(n)
        ref[cols] = O.score_heads([H.f64(q[0, bb:bb + 1])], [kb[:, cols]], 0.1)[0]
        np.testing.assert_allclose(H.f64(s[bb]), ref, rtol=2e-4, atol=1e-7)


def test_score_heads_unaligned_output():
    """S at an address that is 4- but not 16-byte aligned: the same bits."""
    p, b, rows, d, n = 2, 3, 5, 64, 2048
    g = I.generator(91)
    q = torch.randn((p, b, rows, d), generator=g).to(torch.bfloat16).to(DEV)
    keys = [torch.randn((b, 2, n, d), generator=g).to(torch.bfloat16).to(DEV)
            for _ in range(p)]
    s_a = H.score(q, keys, [0, 1], 0.125, n)
    buf = torch.full((b * n + 4,), float("nan"), device=DEV)
    s_u = H.score(q, keys, [0, 1], 0.125, n, out=buf[1:1 + b * n].view(b, n))
    assert torch.equal(s_a, s_u)
    assert torch.isnan(buf[0]) and torch.isnan(buf[1 + b * n:]).all()


def test_score_heads_workspace_alignment_and_reuse():
    """The logits pass keeps its fp32 logits in L2 and the second pass drops
    them after reading only when n is a multiple of 32 and the workspace
    starts on a 128-byte boundary.  A workspace that is 16- but not
    128-byte aligned takes the path that leaves them in memory: the same S
    bits either way, twice in a row over the same workspaces."""
    p, b, rows, d, n = 3, 2, 4, 64, 8192
    g = I.generator(97)
    q = torch.randn((p, b, rows, d), generator=g).to(torch.bfloat16).to(DEV)
    keys = [torch.randn((b, 2, n, d), generator=g).to(torch.bfloat16).to(DEV)
            for _ in range(p)]
    descs = [N.kv_desc(k) for k in keys]
    need = N.dustin_score_heads_workspace_size(b, n, p, rows)
    ws_a = N.workspace(need, DEV)                         # 256-byte aligned
    raw = torch.empty(need + 256, dtype=torch.uint8, device=DEV)
    ws_u = raw[16:16 + need]                              # 16-, not 128-byte aligned
    assert ws_a.data_ptr() % 128 == 0 and ws_u.data_ptr() % 128 == 16
    outs = []
    for ws in (ws_a, ws_u, ws_a, ws_u):
        s = torch.full((b, n), float("nan"), device=DEV)
        N.dustin_score_heads(q, descs, [0, 1, 1], 0.125, s, ws, n)
        H.sync()
        outs.append(s)
    assert all(torch.equal(outs[0], o) for o in outs[1:])
    ref = O.score_heads([H.f64(q[i]) for i in range(p)],
                        [H.f64(keys[i][:, h]) for i, h in enumerate([0, 1, 1])], 0.125)
    np.testing.assert_allclose(H.f64(outs[0]), ref, rtol=2e-4, atol=1e-7)
    assert N.dustin_device_status() == 0


# ---------------------------------------------------------------- selection

SELECT_CASES = [
    # b, n, k, n_sink, n_recent, alpha, m, norm, specials
    (3, 1000, 100, 4, 64, 0.5, -1, 1, False),
    (2, 32768, 2048, 4, 64, 0.5, -1, 1, True),
    (4, 5000, 700, 0, 0, 1.0, -1, 0, True),
    (2, 4096, 300, 2, 8, 0.0, -1, 1, False),
    (2, 3000, 500, 4, 16, 0.25, -1, 0, True),
    (2, 3000, 500, 4, 16, 0.5, 100, 1, False),
    (2, 3000, 500, 4, 16, 0.5, 0, 1, True),
    (2, 3000, 500, 4, 16, 0.5, 1000, 1, False),
    (1, 100, 100, 2, 2, 0.5, -1, 1, False),
    (1, 100, 250, 2, 2, 0.5, -1, 1, False),
    (2, 100, 12, 4, 8, 0.5, -1, 1, False),
    (1, 1, 1, 0, 0, 0.5, -1, 1, False),
    (3, 17, 5, 0, 0, 0.5, -1, 1, False),
    (2, 65536, 8192, 4, 64, 0.5, -1, 1, True),
    # one 8-CTA cluster per sequence: m mode, ragged segments, and rows too
    # long for the keys to stay in shared memory
    (2, 32768, 2048, 4, 64, 0.5, 512, 1, True),
    (2, 12345, 1500, 3, 17, 0.3, -1, 1, True),
    (1, 400000, 4000, 4, 64, 0.5, -1, 1, False),
    (1, 400000, 4000, 4, 64, 0.5, 1000, 1, False),
    # 16 sequences: 8-CTA clusters do not all fit at once, so each sequence
    # gets a smaller cluster
    (16, 32768, 2048, 4, 64, 0.5, -1, 1, True),
    (16, 20000, 3000, 2, 8, 0.7, 600, 1, True),
    # many short rows (at least 304 of at most 4096 positions): the
    # 256-thread CTAs, one per row
    (400, 2048, 128, 0, 0, 1.0, -1, 0, True),
    (320, 3000, 500, 4, 16, 0.5, -1, 1, True),
    (310, 1000, 100, 2, 8, 0.5, 50, 1, False),
    (304, 4096, 700, 4, 64, 0.3, -1, 1, True),
    (303, 2048, 128, 0, 0, 1.0, -1, 0, True),
]


@pytest.mark.parametrize("case", SELECT_CASES, ids=[str(c) for c in SELECT_CASES])
def test_select_bit_exact(case):
    b, n, k, ns, nr, alpha, m, norm, specials = case
    sd = I.synthetic_scores(b, n, seed=n + k, specials=specials)
    st = I.synthetic_scores(b, n, seed=n + k + 1, specials=specials)
    got = H.select(sd.to(DEV), st.to(DEV), k, ns, nr, alpha, m, norm)
    want = O.hybrid_select(sd.numpy(), st.numpy(), k, ns, nr, alpha, m, norm)
    np.testing.assert_array_equal(got.cpu().numpy(), want)


@pytest.mark.parametrize("n", [32768, 20000])
def test_select_ties_across_the_cluster(n):
    """Equal scores spread over every CTA of a sequence's cluster: the tie
    rule (lower position first) must hold across CTA boundaries."""
    g = I.generator(n)
    sd = torch.where(torch.rand((2, n), generator=g) < 0.5, 1.0, 0.5).float()
    st = torch.ones((2, n))
    for k in (1000, n // 2 + 7, n - 100):
        got = H.select(sd.to(DEV), st.to(DEV), k, 4, 64, 0.5, -1, 1)
        want = O.hybrid_select(sd.numpy(), st.numpy(), k, 4, 64, 0.5, -1, 1)
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def _planted(n, top, seed, lo, hi):
    """Two rows of n scores in [0.25, 0.5) with the values `top` written at
    random positions in [lo, hi) (the same values, shuffled, in each row)."""
    g = I.generator(seed)
    s = 0.25 + 0.25 * torch.rand((2, n), generator=g, dtype=torch.float64)
    for r in range(2):
        pos = lo + torch.randperm(hi - lo, generator=g)[: len(top)]
        s[r, pos] = torch.as_tensor(top, dtype=torch.float64)[torch.randperm(len(top), generator=g)]
    return s.float()


@pytest.mark.parametrize("n", [32768, 3000])
def test_select_bucket_holds_exactly_the_rest(n):
    """Scores built so that the bucket holding the budget-th key holds
    exactly the keys still needed after the first, the second or only the
    third radix digit (top bits: sign, exponent, 2 mantissa bits; then 11
    mantissa bits; then the last 10): the set must not depend on where the
    count first matches, and must equal the oracle's."""
    ns, nr = 4, 64
    k = min(2048, n // 4)
    budget = k - ns - nr
    # first digit: budget equal values far above the rest
    a = _planted(n, [4.0] * budget, seed=n + 1, lo=ns, hi=n - nr)
    # second digit: budget + 68 distinct values sharing the first digit
    b = _planted(n, [1.0 + i * 2.0 ** -13 for i in range(budget + 68)], seed=n + 2, lo=ns, hi=n - nr)
    # third digit: pairs that share the first two digits (an odd budget
    # leaves one key of a pair to the third digit)
    pairs = [1.0 + ((i // 2) * 1024 + (i % 2)) * 2.0 ** -23 for i in range(2 * budget)]
    c = _planted(n, pairs, seed=n + 3, lo=ns, hi=n - nr)
    for sd, kk in ((a, k), (b, k), (c, k), (c, k + 1)):
        got = H.select(sd.to(DEV), None, kk, ns, nr, 1.0, -1, 0)
        want = O.hybrid_select(sd.numpy(), None, kk, ns, nr, 1.0, -1, 0)
        np.testing.assert_array_equal(got.cpu().numpy(), want)
    # two rounds (draft quota, then target) with the match at different digits
    for sd, st in ((a, b), (b, c), (c, a)):
        got = H.select(sd.to(DEV), st.to(DEV), k, ns, nr, 0.5, k // 4 + 1, 1)
        want = O.hybrid_select(sd.numpy(), st.numpy(), k, ns, nr, 0.5, k // 4 + 1, 1)
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_select_bucket_holds_exactly_the_rest_short_rows():
    """The same early stop on the instance for many short rows (one
    256-thread CTA per row): 320 rows of 2048 scores built so that, over the
    two budgets, rows stop after the first, the second and the third
    digit."""
    rows, n, k = 320, 2048, 128
    ns, nr = 2, 8
    budget = k - ns - nr
    a = _planted(n, [4.0] * budget, seed=71, lo=ns, hi=n - nr)
    b = _planted(n, [1.0 + i * 2.0 ** -13 for i in range(budget + 40)], seed=72,
                 lo=ns, hi=n - nr)
    pairs = [1.0 + ((i // 2) * 1024 + (i % 2)) * 2.0 ** -23 for i in range(2 * budget)]
    c = _planted(n, pairs, seed=73, lo=ns, hi=n - nr)
    planted = torch.cat([a, b, c])                      # 6 distinct rows
    sd = planted[torch.arange(rows) % planted.shape[0]].contiguous()
    for kk in (k, k + 1):
        got = H.select(sd.to(DEV), None, kk, ns, nr, 1.0, -1, 0)
        want = O.hybrid_select(sd.numpy(), None, kk, ns, nr, 1.0, -1, 0)
        np.testing.assert_array_equal(got.cpu().numpy(), want)


def test_select_single_vector():
    sd = I.synthetic_scores(2, 2000, seed=1)
    got = H.select(sd.to(DEV), None, 100, 4, 4, 1.0, -1, 0)
    want = O.hybrid_select(sd.numpy(), None, 100, 4, 4, 1.0, -1, 0)
    np.testing.assert_array_equal(got.cpu().numpy(), want)
    # alpha = 1, NONE, no target: the vector passes through unchanged, so
    # the result is the Top-K of the raw vector.
    forced = O.protected_positions(2000, 4, 4)
    elig = np.ones(2000, bool)
    elig[forced] = False
    for r in range(2):
        raw = np.sort(np.concatenate([forced, O.topk(sd[r].numpy(), 92, elig)]))
        np.testing.assert_array_equal(got[r].cpu().numpy(), raw)
    st = I.synthetic_scores(2, 2000, seed=2)
    got = H.select(None, st.to(DEV), 100, 4, 4, 0.0, -1, 1)
    want = O.hybrid_select(None, st.numpy(), 100, 4, 4, 0.0, -1, 1)
    np.testing.assert_array_equal(got.cpu().numpy(), want)


# ---------------------------------------------------------------- the chain

def test_tiny_chain_score_select_attend():
    """The tiny workload end to end: scores match, the index set equals the
    oracle's, attention matches, windowed ARR agrees."""
    wl = I.WORKLOADS["tiny"]
    st_in = I.step_inputs(wl, "cpu")
    s_t = H.score(st_in.q_t.to(DEV), [k.to(DEV) for k in st_in.k_t],
                  st_in.kvh_t, wl.scale, wl.n)
    s_d = H.score(st_in.q_d.to(DEV), [k.to(DEV) for k in st_in.k_d],
                  st_in.kvh_d, wl.draft_scale, wl.n)
    ref_t = O.score_heads([H.f64(st_in.q_t[i]) for i in range(wl.p_t)],
                          [H.f64(k[:, h]) for k, h in zip(st_in.k_t,
                                                          st_in.kvh_t)],
                          wl.scale)
    ref_d = O.score_heads([H.f64(st_in.q_d[i]) for i in range(wl.p_d)],
                          [H.f64(k[:, h]) for k, h in zip(st_in.k_d,
                                                          st_in.kvh_d)],
                          wl.draft_scale)
    np.testing.assert_allclose(H.f64(s_t), ref_t, rtol=2e-4, atol=1e-7)
    np.testing.assert_allclose(H.f64(s_d), ref_d, rtol=2e-4, atol=1e-7)
    idx = H.select(s_d, s_t, wl.k, wl.n_sink, wl.n_recent, wl.alpha, -1, 1)
    idx_ref = O.hybrid_select(ref_d, ref_t, wl.k, wl.n_sink, wl.n_recent,
                              wl.alpha, -1, 1)
    np.testing.assert_array_equal(idx.cpu().numpy(), idx_ref)
    q, k, v = st_in.q[0], st_in.k[0], st_in.v[0]
    o, lse = H.sparse_attn(q.to(DEV), k.to(DEV), v.to(DEV), idx, wl.scale)
    o_ref, l_ref = O.verify_attention(H.f64(q), H.f64(k), H.f64(v), idx_ref,
                                      wl.scale)
    H.assert_attn_close(o, lse, o_ref, l_ref)
    a = np.stack([O.attention_weights(H.f64(q)[0, h], H.f64(k)[0, h // 2],
                                      wl.scale) for h in range(wl.hq)])
    got = np.mean([O.windowed_arr(a[h], idx.cpu().numpy()[0])
                   for h in range(wl.hq)])
    want = np.mean([O.windowed_arr(a[h], idx_ref[0]) for h in range(wl.hq)])
    assert abs(got - want) <= H.ARR_TOL
