"""Helpers for the GPU parity tests: run the CUDA path through the C-ABI
binding and convert inputs for the CPU oracle.  Nothing here computes any
part of the method."""
import numpy as np
import torch

from sparse_kv_verification_gb300 import native as N

O_TOL = 2e-2      # max abs error on bf16 attention outputs
LSE_TOL = 1e-3    # max abs error on the fp32 log-sum-exp
ARR_TOL = 1e-5    # windowed ARR, indices from GPU scores vs oracle scores


def f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def sync():
    torch.cuda.synchronize()


def sparse_attn(q, k, v, idx, scale, n=None, page_table=None):
    b, hq, w, d = q.shape
    hkv = k.shape[1]
    n = k.shape[2] if n is None else n
    desc = N.kv_desc(k, v, page_table)
    kk = idx.shape[1]
    ws = N.workspace(N.dustin_sparse_verify_attn_workspace_size(
        b, hq, hkv, d, w, kk), q.device)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((b, hq, w), float("nan"), device=q.device)
    N.dustin_sparse_verify_attn(q, desc, hkv, n, idx, scale, o, lse, ws)
    sync()
    return o, lse


def full_attn(q, k, v, scale, n=None, page_table=None):
    b, hq, w, d = q.shape
    hkv = k.shape[1]
    n = k.shape[2] if n is None else n
    desc = N.kv_desc(k, v, page_table)
    ws = N.workspace(N.dustin_full_verify_attn_workspace_size(
        b, hq, hkv, d, w, n), q.device)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((b, hq, w), float("nan"), device=q.device)
    N.dustin_full_verify_attn(q, desc, hkv, n, scale, o, lse, ws)
    sync()
    return o, lse


def sparse_attn_window(q, k, v, idx, kw, vw, scale, n=None, page_table=None,
                       flags=0):
    b, hq, w, d = q.shape
    hkv = k.shape[1]
    n = k.shape[2] if n is None else n
    ws = N.workspace(N.dustin_sparse_verify_attn_workspace_size(
        b, hq, hkv, d, w, idx.shape[1]), q.device)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((b, hq, w), float("nan"), device=q.device)
    N.dustin_sparse_verify_attn_window(q, N.kv_desc(k, v, page_table), hkv, n,
                                       idx, N.kv_desc(kw, vw), scale, o, lse, ws,
                                       flags=flags)
    sync()
    return o, lse


def full_attn_window(q, k, v, kw, vw, scale, n=None, page_table=None, flags=0):
    b, hq, w, d = q.shape
    hkv = k.shape[1]
    n = k.shape[2] if n is None else n
    ws = N.workspace(N.dustin_full_verify_attn_workspace_size(
        b, hq, hkv, d, w, n), q.device)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((b, hq, w), float("nan"), device=q.device)
    N.dustin_full_verify_attn_window(q, N.kv_desc(k, v, page_table), hkv, n,
                                     N.kv_desc(kw, vw), scale, o, lse, ws,
                                     flags=flags)
    sync()
    return o, lse


def score(q, keys, kv_heads, scale, n, page_tables=None, out=None):
    """q [P][b][rows][d]; keys: list of K tensors (one per pair); out: an
    optional [b][n] fp32 output (any 4-byte alignment)."""
    p, b, rows, d = q.shape
    pts = page_tables or [None] * p
    descs = [N.kv_desc(k, None, pt) for k, pt in zip(keys, pts)]
    ws = N.workspace(N.dustin_score_heads_workspace_size(b, n, p, rows),
                     q.device)
    s = torch.full((b, n), float("nan"), device=q.device) if out is None else out
    N.dustin_score_heads(q, descs, kv_heads, scale, s, ws, n)
    sync()
    return s


def select(sd, st, k, ns, nr, alpha, m, norm):
    ref = sd if sd is not None else st
    b, n = ref.shape
    idx = torch.full((b, min(k, n)), -7, dtype=torch.int32, device=ref.device)
    N.dustin_hybrid_topk(sd, st, k, ns, nr, alpha, m, norm, idx)
    sync()
    return idx


def assert_attn_close(o, lse, o_ref, lse_ref):
    og = f64(o)
    lg = f64(lse)
    assert np.all(np.isfinite(og)), "non-finite output"
    err_o = np.max(np.abs(og - o_ref)) if og.size else 0.0
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lg), fin), "LSE finiteness differs"
    err_l = np.max(np.abs(lg[fin] - lse_ref[fin])) if fin.any() else 0.0
    assert err_o <= O_TOL, f"O max abs error {err_o}"
    assert err_l <= LSE_TOL, f"LSE max abs error {err_l}"
    return err_o, err_l
