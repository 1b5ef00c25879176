"""The C-ABI library builds, loads and exports every symbol its header
declares; host-side validation rejects bad calls before any launch.  None of
these calls reaches a kernel: each case fails validation first (or is a
no-op), so they run without a GPU."""
import ctypes
import os
import re

import pytest

from sparse_kv_verification_gb300 import build, native

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include",
                      "dustin.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return native.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dustin_[a-z0-9_]+)\s*\(", text)))


def test_header_and_binding_agree():
    assert sorted(native.EXPORTS) == declared_functions()


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.dustin_status_string(0) == b"ok"
    for s in range(1, 8):
        assert lib.dustin_status_string(s) not in (b"", b"unknown status")
    assert lib.dustin_status_string(99) == b"unknown status"
    assert lib.dustin_version() >= 100


FAKE = 0x10000   # never dereferenced: every call below fails validation


def kv(stride_n=128, d=128, page_table=None, page_size=0, ppseq=0, pages=0,
       base=FAKE):
    desc = native.DustinKV()
    desc.k = base
    desc.v = base
    desc.stride_b, desc.stride_h, desc.stride_n = 8 * 4096 * d, 4096 * d, stride_n
    desc.page_table = page_table
    desc.page_size = page_size
    desc.pages_per_seq = ppseq
    desc.num_pages = pages
    return desc


def sparse(lib, **kw):
    args = dict(b=1, hq=8, hkv=2, d=128, w=4, n=256, k=32, q=FAKE,
                kv=kv(), idx=FAKE, scale=0.1, o=FAKE, lse=FAKE, ws=None,
                ws_bytes=0, flags=0)
    args.update(kw)
    r = lib.dustin_sparse_verify_attn(
        args["b"], args["hq"], args["hkv"], args["d"], args["w"], args["n"],
        args["k"], args["q"], ctypes.byref(args["kv"]), args["idx"],
        args["scale"], args["o"], args["lse"], args["ws"], args["ws_bytes"],
        args["flags"], None)
    return r, lib.dustin_last_error().decode()


def test_attention_validation(lib):
    assert sparse(lib, d=96)[0] == 3
    assert sparse(lib, k=300)[0] == 2
    assert sparse(lib, k=-1)[0] == 2
    assert sparse(lib, hq=7)[0] == 2
    assert sparse(lib, w=0)[0] == 2
    assert sparse(lib, q=None)[0] == 1
    assert sparse(lib, idx=None)[0] == 1
    assert sparse(lib, q=FAKE + 8)[0] == 5
    assert sparse(lib, kv=kv(stride_n=100))[0] == 2
    assert sparse(lib, kv=kv(stride_n=132))[0] == 5
    assert sparse(lib, kv=kv(base=FAKE + 4))[0] == 5
    assert sparse(lib, scale=float("nan"))[0] == 1
    assert sparse(lib, scale=0.0)[0] == 1
    assert sparse(lib, scale=-0.5)[0] == 1
    assert sparse(lib, flags=2)[0] == 1           # unknown flag bit
    assert sparse(lib, kv=kv(page_table=FAKE, page_size=8, ppseq=32,
                             pages=64))[0] == 3
    assert sparse(lib, kv=kv(page_table=FAKE, page_size=16, ppseq=4,
                             pages=64))[0] == 2
    r, msg = sparse(lib, d=96)
    assert "d=96" in msg
    # b == 0 is a no-op that touches nothing.
    assert sparse(lib, b=0, q=None, o=None, lse=None)[0] == 0


def test_multi_layer_validation(lib):
    qa = (ctypes.c_void_p * 2)(FAKE, FAKE)
    ka = (native.DustinKV * 2)(kv(), kv())
    la = (ctypes.c_void_p * 2)(FAKE, FAKE)

    def call(k=32, kvs=ka, n_layers=2):
        return lib.dustin_sparse_verify_attn_layers(
            n_layers, 1, 8, 2, 128, 4, 4096, k, ctypes.addressof(qa),
            ctypes.addressof(kvs), FAKE, 0.1, ctypes.addressof(qa),
            ctypes.addressof(la), 0, None)
    assert call(k=3000) == 3                     # k above 2048
    mixed = (native.DustinKV * 2)(kv(), kv(page_table=FAKE, page_size=16, ppseq=256,
                                       pages=64))
    assert call(kvs=mixed) == 1                  # paged and contiguous mixed
    assert call(n_layers=0) == 0                 # nothing to do


def test_score_and_select_validation(lib):
    heads = (ctypes.c_int32 * 1)(0)
    arr = (native.DustinKV * 1)(kv())
    call = lambda **kw: lib.dustin_score_heads(
        kw.get("b", 1), kw.get("n", 64), kw.get("d", 128), kw.get("p", 1),
        kw.get("rows", 1), kw.get("q", FAKE), ctypes.addressof(arr),
        ctypes.addressof(heads), 0.1, kw.get("s", FAKE), kw.get("ws", None),
        kw.get("wsb", 0), None)
    assert call(d=80) == 3
    assert call(rows=17) == 3
    assert call(p=65) == 3
    assert call(q=None) == 1
    assert call(ws=None) == 4
    assert call(b=0) == 0
    assert call(n=0) == 0
    assert lib.dustin_score_heads_workspace_size(2, 100, 3, 4) >= 2 * 100 * 12 * 4
    sel = lambda **kw: lib.dustin_hybrid_topk(
        kw.get("b", 1), kw.get("n", 100), kw.get("k", 10), kw.get("ns", 2),
        kw.get("nr", 2), kw.get("alpha", 0.5), kw.get("m", -1),
        kw.get("norm", 1), kw.get("sd", FAKE), kw.get("st", FAKE),
        kw.get("idx", FAKE), None)
    assert sel(k=3) == 2                  # 4 protected > k
    assert sel(norm=5) == 1
    assert sel(sd=None, st=None) == 1
    assert sel(idx=None) == 1
    assert sel(alpha=float("inf")) == 1
    assert sel(m=3, sd=None) == 1
    assert sel(n=(1 << 20) + 1) == 3
    assert sel(b=0) == 0 and sel(k=0) == 0


def test_noalloc_checks_arguments_before_the_array_size(lib):
    """The no-allocation scoring call gives the statuses of dustin_score_heads
    for bad arguments even when their scratch would also overflow the
    built-in array, and WORKSPACE only for valid calls that need more."""
    assert lib.dustin_score_heads_noalloc_capacity() == native.noalloc_scratch_bytes()
    cap = lib.dustin_score_heads_noalloc_capacity()
    heads = (ctypes.c_int32 * 64)(*([0] * 64))
    arr = (native.DustinKV * 64)(*([kv(stride_n=128)] * 64))
    call = lambda b=16, n=32768, d=128, p=64, rows=1: lib.dustin_score_heads_noalloc(
        b, n, d, p, rows, FAKE, ctypes.addressof(arr), ctypes.addressof(heads), 0.1,
        FAKE, None)
    assert lib.dustin_score_heads_workspace_size(16, 32768, 64, 1) > cap
    assert call(d=96) == 3
    assert call(rows=17) == 3
    assert call(p=65) == 3
    assert call(b=-1) == 2
    assert call() == 4
    assert str(cap) in lib.dustin_last_error().decode()
    assert call(b=0) == 0


def test_quest_and_window_validation(lib):
    pst = lambda **kw: lib.dustin_quest_page_stats(
        kw.get("b", 1), kw.get("hkv", 2), kw.get("d", 128), kw.get("n", 256),
        kw.get("page", 16), ctypes.byref(kw.get("kv", kv())), kw.get("st", FAKE), None)
    assert pst(d=96) == 3
    assert pst(page=0) == 2
    assert pst(st=FAKE + 4) == 5
    assert pst(b=0) == 0
    psc = lambda **kw: lib.dustin_quest_page_scores(
        kw.get("b", 1), kw.get("hq", 8), kw.get("hkv", 2), kw.get("d", 128),
        kw.get("n", 256), kw.get("page", 16), kw.get("q", FAKE), kw.get("st", FAKE),
        kw.get("sc", FAKE), None)
    assert psc(hq=130, hkv=2) == 3          # more than 64 query heads per kv head
    assert psc(hq=7) == 2                    # not a multiple of h_kv
    assert psc(q=None) == 1
    assert psc(st=FAKE + 8) == 5
    assert psc(d=80) == 3
    assert lib.dustin_quest_stats_size(2, 4, 128, 1000, 16) == 2 * 4 * 63 * 2 * 128 * 2
    win = kv(stride_n=128)
    wcall = lambda **kw: lib.dustin_sparse_verify_attn_window(
        1, 8, 2, 128, 4, 256, 32, FAKE, ctypes.byref(kv()), FAKE,
        ctypes.byref(kw.get("win", win)) if kw.get("win", win) is not None else None,
        0.1, FAKE, FAKE, None, 0, kw.get("flags", 0), None)
    assert wcall(win=None) == 1
    assert wcall(win=kv(stride_n=100)) == 2
    assert wcall(flags=4) == 1


def test_wait_selftest_limit_is_checked_before_launch(lib):
    """The self-test's limit is validated on the host: an out-of-range limit
    launches nothing (no GPU needed)."""
    assert lib.dustin_wait_selftest(0, None) == 2
    assert lib.dustin_wait_selftest(-5, None) == 2
    assert lib.dustin_wait_selftest((1 << 31) + 1, None) == 2
