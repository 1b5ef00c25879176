"""Python binding of libdustin.so (the C-ABI in include/dustin.h).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  The functions carry the C names and take torch tensors that live on
a CUDA device; shapes are read from the tensors.  A non-zero status raises
``DustinError``.  Loading fails loudly if the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Sequence

import torch

from . import build as _build

DUSTIN_OK = 0
DUSTIN_NORM_NONE = 0
DUSTIN_NORM_L1 = 1
DUSTIN_ATTN_KV_READY = 1

EXPORTS = (
    "dustin_status_string", "dustin_last_error", "dustin_version",
    "dustin_launch_count", "dustin_device_status", "dustin_wait_selftest",
    "dustin_score_heads_workspace_size", "dustin_score_heads",
    "dustin_score_heads_noalloc", "dustin_score_heads_noalloc_capacity",
    "dustin_hybrid_topk",
    "dustin_sparse_verify_attn_workspace_size", "dustin_sparse_verify_attn",
    "dustin_sparse_verify_attn_window",
    "dustin_full_verify_attn_workspace_size", "dustin_full_verify_attn",
    "dustin_full_verify_attn_window",
    "dustin_sparse_verify_attn_layers",
    "dustin_quest_stats_size", "dustin_quest_page_stats",
    "dustin_quest_page_scores",
)


class DustinError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"dustin status {status}: {message}")
        self.status = status


class DustinKV(ctypes.Structure):
    """Mirror of ``dustin_kv``."""
    _fields_ = [
        ("k", ctypes.c_void_p),
        ("v", ctypes.c_void_p),
        ("stride_b", ctypes.c_int64),
        ("stride_h", ctypes.c_int64),
        ("stride_n", ctypes.c_int64),
        ("page_table", ctypes.c_void_p),
        ("page_size", ctypes.c_int32),
        ("pages_per_seq", ctypes.c_int32),
        ("num_pages", ctypes.c_int32),
    ]


_LIB: Optional[ctypes.CDLL] = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False, path: Optional[str] = None
         ) -> ctypes.CDLL:
    """Loads libdustin.so (or the library at `path`, which then replaces the
    loaded one); raises if it is missing (there is no fallback)."""
    global _LIB
    if _LIB is not None and path is None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        if not build_if_missing:
            raise RuntimeError(
                f"{path} is missing: build it with "
                "`python -m sparse_kv_verification_gb300.build`")
        _build.build()
    lib = ctypes.CDLL(path)
    P, I, F, D, S, U = (ctypes.c_void_p, ctypes.c_int, ctypes.c_float,
                        ctypes.c_double, ctypes.c_size_t, ctypes.c_uint)
    sig = {
        "dustin_status_string": (ctypes.c_char_p, [I]),
        "dustin_last_error": (ctypes.c_char_p, []),
        "dustin_version": (I, []),
        "dustin_launch_count": (ctypes.c_uint64, []),
        "dustin_device_status": (I, [P]),
        "dustin_wait_selftest": (I, [ctypes.c_int64, P]),
        "dustin_score_heads_workspace_size": (S, [I, I, I, I]),
        "dustin_score_heads": (I, [I, I, I, I, I, P, P, P, F, P, P, S, P]),
        "dustin_score_heads_noalloc": (I, [I, I, I, I, I, P, P, P, F, P, P]),
        "dustin_score_heads_noalloc_capacity": (S, []),
        "dustin_hybrid_topk": (I, [I, I, I, I, I, D, I, I, P, P, P, P]),
        "dustin_sparse_verify_attn_workspace_size": (S, [I, I, I, I, I, I]),
        "dustin_sparse_verify_attn": (I, [I, I, I, I, I, I, I, P, P, P, F, P, P,
                                          P, S, U, P]),
        "dustin_full_verify_attn_workspace_size": (S, [I, I, I, I, I, I]),
        "dustin_full_verify_attn": (I, [I, I, I, I, I, I, P, P, F, P, P, P, S,
                                        U, P]),
        "dustin_sparse_verify_attn_window": (I, [I, I, I, I, I, I, I, P, P, P, P,
                                                 F, P, P, P, S, U, P]),
        "dustin_full_verify_attn_window": (I, [I, I, I, I, I, I, P, P, P, F, P, P,
                                               P, S, U, P]),
        "dustin_sparse_verify_attn_layers": (I, [I, I, I, I, I, I, I, I, P, P, P, F,
                                                 P, P, U, P]),
        "dustin_quest_stats_size": (S, [I, I, I, I, I]),
        "dustin_quest_page_stats": (I, [I, I, I, I, I, P, P, P]),
        "dustin_quest_page_scores": (I, [I, I, I, I, I, I, P, P, P, P]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def _check(status: int) -> None:
    if status != DUSTIN_OK:
        lib = load()
        raise DustinError(status, lib.dustin_last_error().decode())


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(stream, device) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream


def _need_cuda(*ts: Optional[torch.Tensor]) -> None:
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("tensors must live on a CUDA device")


def kv_desc(k: torch.Tensor, v: Optional[torch.Tensor] = None,
            page_table: Optional[torch.Tensor] = None) -> DustinKV:
    """Describes a KV cache.  Contiguous: k (and v) [b][h_kv][n][d].
    Paged: k (and v) are pools [pages][h_kv][page_size][d] and page_table is
    int32 [b][pages_per_seq].  K and V must share strides."""
    if k.dtype != torch.bfloat16 or k.dim() != 4 or k.stride(3) != 1:
        raise ValueError("k must be a bf16 4-D tensor with a contiguous last dim")
    if v is not None and (v.shape != k.shape or v.stride() != k.stride()
                          or v.dtype != k.dtype):
        raise ValueError("v must match k in shape, strides and dtype")
    desc = DustinKV()
    desc.k = k.data_ptr()
    desc.v = v.data_ptr() if v is not None else None
    desc.stride_b, desc.stride_h, desc.stride_n = (k.stride(0), k.stride(1),
                                                   k.stride(2))
    if page_table is not None:
        if page_table.dtype != torch.int32 or page_table.dim() != 2:
            raise ValueError("page_table must be int32 [b][pages_per_seq]")
        if page_table.stride(1) != 1:
            raise ValueError("page_table rows must be contiguous")
        desc.page_table = page_table.data_ptr()
        desc.page_size = k.shape[2]
        desc.pages_per_seq = page_table.stride(0)
        desc.num_pages = k.shape[0]
    return desc


def workspace(nbytes: int, device) -> torch.Tensor:
    """A caller-owned scratch buffer (uint8, 256-byte aligned by torch)."""
    return torch.empty(max(int(nbytes), 1), dtype=torch.uint8, device=device)


# ------------------------------------------------------------------ scoring

def dustin_score_heads_workspace_size(b: int, n: int, n_pairs: int,
                                      rows: int) -> int:
    return int(load().dustin_score_heads_workspace_size(b, n, n_pairs, rows))


def dustin_score_heads(q: torch.Tensor, kvs: Sequence[DustinKV],
                       kv_heads: Sequence[int], scale: float,
                       s_out: torch.Tensor, ws: torch.Tensor, n: int,
                       stream=None) -> None:
    """q bf16 [n_pairs][b][rows][d]; kvs[p] the pair's key cache; s_out fp32
    [b][n] (overwritten with the summed softmax of every pair and row)."""
    _need_cuda(q, s_out, ws)
    n_pairs, b, rows, d = q.shape
    if len(kvs) != n_pairs or len(kv_heads) != n_pairs:
        raise ValueError("one kv descriptor and kv head per scored pair")
    if not q.is_contiguous() or s_out.dtype != torch.float32:
        raise ValueError("q must be contiguous; s_out fp32")
    arr = (DustinKV * n_pairs)(*kvs)
    heads = (ctypes.c_int32 * n_pairs)(*[int(h) for h in kv_heads])
    with torch.cuda.device(q.device):
        _check(load().dustin_score_heads(
            b, n, d, n_pairs, rows, q.data_ptr(), ctypes.addressof(arr),
            ctypes.addressof(heads), float(scale), s_out.data_ptr(), ws.data_ptr(),
            ws.numel(), _stream(stream, q.device)))


def noalloc_scratch_bytes() -> int:
    """Size of the library's built-in scoring scratch array."""
    return int(load().dustin_score_heads_noalloc_capacity())


def dustin_score_heads_noalloc(q: torch.Tensor, kvs: Sequence[DustinKV],
                               kv_heads: Sequence[int], scale: float,
                               s_out: torch.Tensor, n: int,
                               stream=None) -> None:
    """dustin_score_heads with the library's built-in scratch array instead
    of a workspace: for callers that cannot allocate device memory.  Calls
    share the array and must not overlap on the GPU."""
    _need_cuda(q, s_out)
    n_pairs, b, rows, d = q.shape
    if len(kvs) != n_pairs or len(kv_heads) != n_pairs:
        raise ValueError("one kv descriptor and kv head per scored pair")
    if not q.is_contiguous() or s_out.dtype != torch.float32:
        raise ValueError("q must be contiguous; s_out fp32")
    arr = (DustinKV * n_pairs)(*kvs)
    heads = (ctypes.c_int32 * n_pairs)(*[int(h) for h in kv_heads])
    # The library finds the array of the current device: make it q's.
    with torch.cuda.device(q.device):
        _check(load().dustin_score_heads_noalloc(
            b, n, d, n_pairs, rows, q.data_ptr(), ctypes.addressof(arr),
            ctypes.addressof(heads), float(scale), s_out.data_ptr(),
            _stream(stream, q.device)))


# ------------------------------------------------------------------ selection

def dustin_hybrid_topk(s_draft: Optional[torch.Tensor],
                       s_target: Optional[torch.Tensor], k: int, n_sink: int,
                       n_recent: int, alpha: float, m: int, norm: int,
                       idx: torch.Tensor, stream=None) -> None:
    """idx int32 [b][min(k, n)] receives ascending kept positions."""
    ref = s_draft if s_draft is not None else s_target
    if ref is None:
        raise ValueError("need at least one score vector")
    _need_cuda(s_draft, s_target, idx)
    for s in (s_draft, s_target):
        if s is not None and (s.dtype != torch.float32 or not s.is_contiguous()
                              or s.shape != ref.shape):
            raise ValueError("score vectors: contiguous fp32 [b][n]")
    b, n = ref.shape
    if idx.dtype != torch.int32 or not idx.is_contiguous() or \
            tuple(idx.shape) != (b, min(k, n)):
        raise ValueError("idx must be contiguous int32 [b][min(k, n)]")
    _check(load().dustin_hybrid_topk(
        b, n, k, n_sink, n_recent, float(alpha), m, norm, _ptr(s_draft),
        _ptr(s_target), idx.data_ptr(), _stream(stream, ref.device)))


# ------------------------------------------------------------------ attention

def dustin_sparse_verify_attn_workspace_size(b, h_q, h_kv, d, w, k) -> int:
    return int(load().dustin_sparse_verify_attn_workspace_size(
        b, h_q, h_kv, d, w, k))


def dustin_full_verify_attn_workspace_size(b, h_q, h_kv, d, w, n) -> int:
    return int(load().dustin_full_verify_attn_workspace_size(
        b, h_q, h_kv, d, w, n))


def _attn_checks(q, o, lse):
    _need_cuda(q, o, lse)
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or q.dim() != 4:
        raise ValueError("q must be contiguous bf16 [b][h_q][w][d]")
    if o.shape != q.shape or o.dtype != torch.bfloat16 or not o.is_contiguous():
        raise ValueError("o must be contiguous bf16 shaped like q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != tuple(q.shape[:3]) \
            or not lse.is_contiguous():
        raise ValueError("lse must be contiguous fp32 [b][h_q][w]")


def dustin_sparse_verify_attn(q: torch.Tensor, kv: DustinKV, h_kv: int,
                              n: int, idx: torch.Tensor, scale: float,
                              o: torch.Tensor, lse: torch.Tensor,
                              ws: Optional[torch.Tensor], stream=None,
                              flags: int = 0) -> None:
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    if idx.dtype != torch.int32 or not idx.is_contiguous() or idx.dim() != 2 \
            or idx.shape[0] != b:
        raise ValueError("idx must be contiguous int32 [b][k]")
    k = idx.shape[1]
    _check(load().dustin_sparse_verify_attn(
        b, h_q, h_kv, d, w, n, k, q.data_ptr(), ctypes.byref(kv),
        idx.data_ptr(), float(scale), o.data_ptr(), lse.data_ptr(),
        _ptr(ws), 0 if ws is None else ws.numel(), int(flags),
        _stream(stream, q.device)))


def dustin_full_verify_attn(q: torch.Tensor, kv: DustinKV, h_kv: int, n: int,
                            scale: float, o: torch.Tensor, lse: torch.Tensor,
                            ws: Optional[torch.Tensor], stream=None,
                            flags: int = 0) -> None:
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    _check(load().dustin_full_verify_attn(
        b, h_q, h_kv, d, w, n, q.data_ptr(), ctypes.byref(kv), float(scale),
        o.data_ptr(), lse.data_ptr(), _ptr(ws), 0 if ws is None else ws.numel(),
        int(flags), _stream(stream, q.device)))


def dustin_sparse_verify_attn_window(q: torch.Tensor, kv: DustinKV, h_kv: int,
                                     n: int, idx: torch.Tensor, win: DustinKV,
                                     scale: float, o: torch.Tensor,
                                     lse: torch.Tensor,
                                     ws: Optional[torch.Tensor], stream=None,
                                     flags: int = 0) -> None:
    """dustin_sparse_verify_attn with the window's causal block merged in;
    win describes the window tokens' K/V [b][h_kv][w][d] (kv_desc)."""
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    if idx.dtype != torch.int32 or not idx.is_contiguous() or idx.dim() != 2 \
            or idx.shape[0] != b:
        raise ValueError("idx must be contiguous int32 [b][k]")
    _check(load().dustin_sparse_verify_attn_window(
        b, h_q, h_kv, d, w, n, idx.shape[1], q.data_ptr(), ctypes.byref(kv),
        idx.data_ptr(), ctypes.byref(win), float(scale), o.data_ptr(),
        lse.data_ptr(), _ptr(ws), 0 if ws is None else ws.numel(), int(flags),
        _stream(stream, q.device)))


def dustin_full_verify_attn_window(q: torch.Tensor, kv: DustinKV, h_kv: int,
                                   n: int, win: DustinKV, scale: float,
                                   o: torch.Tensor, lse: torch.Tensor,
                                   ws: Optional[torch.Tensor], stream=None,
                                   flags: int = 0) -> None:
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    _check(load().dustin_full_verify_attn_window(
        b, h_q, h_kv, d, w, n, q.data_ptr(), ctypes.byref(kv), ctypes.byref(win),
        float(scale), o.data_ptr(), lse.data_ptr(), _ptr(ws),
        0 if ws is None else ws.numel(), int(flags), _stream(stream, q.device)))


def _layers_args(qs, kvs, idx, os, lses):
    n_layers = len(qs)
    if not (len(kvs) == len(os) == len(lses) == n_layers) or n_layers == 0:
        raise ValueError("one q, kv, o and lse per layer")
    for q, o, lse in zip(qs, os, lses):
        _attn_checks(q, o, lse)
        if q.shape != qs[0].shape:
            raise ValueError("every layer's q has the same shape")
    if idx.dtype != torch.int32 or not idx.is_contiguous() or idx.dim() != 2 \
            or idx.shape[0] != qs[0].shape[0]:
        raise ValueError("idx must be contiguous int32 [b][k]")
    qa = (ctypes.c_void_p * n_layers)(*[q.data_ptr() for q in qs])
    oa = (ctypes.c_void_p * n_layers)(*[o.data_ptr() for o in os])
    la = (ctypes.c_void_p * n_layers)(*[t.data_ptr() for t in lses])
    ka = (DustinKV * n_layers)(*kvs)
    return qa, ka, oa, la


def dustin_sparse_verify_attn_layers(qs: Sequence[torch.Tensor],
                                     kvs: Sequence[DustinKV], h_kv: int, n: int,
                                     idx: torch.Tensor, scale: float,
                                     os: Sequence[torch.Tensor],
                                     lses: Sequence[torch.Tensor], stream=None,
                                     flags: int = 0) -> None:
    """The sparse call for several layers in one persistent launch (one
    index set for all layers)."""
    qa, ka, oa, la = _layers_args(qs, kvs, idx, os, lses)
    b, h_q, w, d = qs[0].shape
    _check(load().dustin_sparse_verify_attn_layers(
        len(qs), b, h_q, h_kv, d, w, n, idx.shape[1], ctypes.addressof(qa),
        ctypes.addressof(ka), idx.data_ptr(), float(scale), ctypes.addressof(oa),
        ctypes.addressof(la), int(flags), _stream(stream, qs[0].device)))


def prepare_sparse_verify_attn_layers(qs, kvs, h_kv, n, idx, scale, os, lses,
                                      stream=None, flags=0):
    qa, ka, oa, la = _layers_args(qs, kvs, idx, os, lses)
    b, h_q, w, d = qs[0].shape
    fn = load().dustin_sparse_verify_attn_layers
    args = (len(qs), b, h_q, h_kv, d, w, n, idx.shape[1], ctypes.addressof(qa),
            ctypes.addressof(ka), idx.data_ptr(), float(scale), ctypes.addressof(oa),
            ctypes.addressof(la), int(flags), _stream(stream, qs[0].device))

    def call():
        _check(fn(*args))
    call.keep = (qa, ka, oa, la)
    return call


# ------------------------------------------------ Quest page scoring baseline

def dustin_quest_page_stats(kv: DustinKV, b: int, h_kv: int, d: int, n: int,
                            page: int, stats: Optional[torch.Tensor] = None,
                            device=None, stream=None) -> torch.Tensor:
    """Per-page channel min/max of the keys: bf16 [b][h_kv][P][2][d]."""
    n_pages = (n + page - 1) // page
    if stats is None:
        stats = torch.empty((b, h_kv, n_pages, 2, d), dtype=torch.bfloat16,
                            device=device)
    _need_cuda(stats)
    _check(load().dustin_quest_page_stats(b, h_kv, d, n, page, ctypes.byref(kv),
                                          stats.data_ptr(),
                                          _stream(stream, stats.device)))
    return stats


def dustin_quest_page_scores(q: torch.Tensor, stats: torch.Tensor, n: int,
                             page: int, scores: Optional[torch.Tensor] = None,
                             stream=None) -> torch.Tensor:
    """q bf16 [b][h_q][d] (one row per head) -> fp32 [b][h_q][P]."""
    _need_cuda(q, stats)
    b, h_q, d = q.shape
    h_kv, n_pages = stats.shape[1], stats.shape[2]
    if q.dtype != torch.bfloat16 or not q.is_contiguous() or not stats.is_contiguous():
        raise ValueError("q bf16 contiguous [b][h_q][d]; stats contiguous")
    if scores is None:
        scores = torch.empty((b, h_q, n_pages), device=q.device)
    _check(load().dustin_quest_page_scores(b, h_q, h_kv, d, n, page, q.data_ptr(),
                                           stats.data_ptr(), scores.data_ptr(),
                                           _stream(stream, q.device)))
    return scores


# ------------------------------------------------------------------ misc

def dustin_wait_selftest(limit_cycles: int, stream=None) -> None:
    """Launches the bounded-wait self-test (one wait that nothing ends)."""
    _check(load().dustin_wait_selftest(int(limit_cycles),
                                       _stream(stream, torch.device("cuda"))))


def dustin_device_status() -> int:
    """Synchronises the device, returns and clears the device-side flags."""
    flags = ctypes.c_uint32(0)
    status = load().dustin_device_status(ctypes.byref(flags))
    if status not in (DUSTIN_OK, 7):          # 7: DUSTIN_ERR_DEVICE
        _check(status)
    return int(flags.value)


def dustin_launch_count() -> int:
    return int(load().dustin_launch_count())


# ------------------------------------------------------------------ prepared
# Pre-marshalled calls for timing loops: every argument (device pointers,
# descriptors, workspace, stream) is fixed once, so a call is one ctypes
# dispatch.  The tensors passed in must outlive the returned callable.

def prepare_score_heads(q, kvs, kv_heads, scale, s_out, ws, n, stream=None):
    _need_cuda(q, s_out, ws)
    n_pairs, b, rows, d = q.shape
    arr = (DustinKV * n_pairs)(*kvs)
    heads = (ctypes.c_int32 * n_pairs)(*[int(h) for h in kv_heads])
    fn = load().dustin_score_heads
    args = (b, n, d, n_pairs, rows, q.data_ptr(), ctypes.addressof(arr),
            ctypes.addressof(heads), float(scale), s_out.data_ptr(),
            ws.data_ptr(), ws.numel(), _stream(stream, q.device))

    def call():
        _check(fn(*args))
    call.keep = (arr, heads)
    return call


def prepare_hybrid_topk(s_draft, s_target, k, n_sink, n_recent, alpha, m,
                        norm, idx, stream=None):
    ref = s_draft if s_draft is not None else s_target
    b, n = ref.shape
    fn = load().dustin_hybrid_topk
    args = (b, n, k, n_sink, n_recent, float(alpha), m, norm, _ptr(s_draft),
            _ptr(s_target), idx.data_ptr(), _stream(stream, ref.device))

    def call():
        _check(fn(*args))
    return call


def prepare_sparse_verify_attn(q, kv, h_kv, n, idx, scale, o, lse, ws,
                               stream=None, flags=0):
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    fn = load().dustin_sparse_verify_attn
    kvc = DustinKV.from_buffer_copy(kv)
    args = (b, h_q, h_kv, d, w, n, idx.shape[1], q.data_ptr(),
            ctypes.addressof(kvc), idx.data_ptr(), float(scale), o.data_ptr(),
            lse.data_ptr(), _ptr(ws), 0 if ws is None else ws.numel(),
            int(flags), _stream(stream, q.device))

    def call():
        _check(fn(*args))
    call.keep = kvc
    return call


def prepare_sparse_verify_attn_window(q, kv, h_kv, n, idx, win, scale, o, lse,
                                      ws, stream=None, flags=0):
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    fn = load().dustin_sparse_verify_attn_window
    kvc, winc = DustinKV.from_buffer_copy(kv), DustinKV.from_buffer_copy(win)
    args = (b, h_q, h_kv, d, w, n, idx.shape[1], q.data_ptr(),
            ctypes.addressof(kvc), idx.data_ptr(), ctypes.addressof(winc),
            float(scale), o.data_ptr(), lse.data_ptr(), _ptr(ws),
            0 if ws is None else ws.numel(), int(flags), _stream(stream, q.device))

    def call():
        _check(fn(*args))
    call.keep = (kvc, winc)
    return call


def prepare_full_verify_attn_window(q, kv, h_kv, n, win, scale, o, lse, ws,
                                    stream=None, flags=0):
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    fn = load().dustin_full_verify_attn_window
    kvc, winc = DustinKV.from_buffer_copy(kv), DustinKV.from_buffer_copy(win)
    args = (b, h_q, h_kv, d, w, n, q.data_ptr(), ctypes.addressof(kvc),
            ctypes.addressof(winc), float(scale), o.data_ptr(), lse.data_ptr(),
            _ptr(ws), 0 if ws is None else ws.numel(), int(flags),
            _stream(stream, q.device))

    def call():
        _check(fn(*args))
    call.keep = (kvc, winc)
    return call


def prepare_full_verify_attn(q, kv, h_kv, n, scale, o, lse, ws, stream=None,
                             flags=0):
    _attn_checks(q, o, lse)
    b, h_q, w, d = q.shape
    fn = load().dustin_full_verify_attn
    kvc = DustinKV.from_buffer_copy(kv)
    args = (b, h_q, h_kv, d, w, n, q.data_ptr(), ctypes.addressof(kvc),
            float(scale), o.data_ptr(), lse.data_ptr(), _ptr(ws),
            0 if ws is None else ws.numel(), int(flags), _stream(stream, q.device))

    def call():
        _check(fn(*args))
    call.keep = kvc
    return call
