"""dustin_score_heads_noalloc: scoring for callers that cannot allocate
device memory (a serving loop that has given all of HBM to the KV cache, a
plugin whose framework owns the allocator).  Its scratch is a fixed array
inside the library, so the call takes no workspace.  These tests call it
through the C-ABI and compare it with dustin_score_heads (which takes a
caller workspace) on two calls in a row with different shapes, so the second
call runs over the first one's leftovers in the shared array.  The file is
named to be collected last."""
import ctypes

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


def _case(p, b, rows, d, n, hkv, seed):
    g = I.generator(seed)
    q = torch.randn((p, b, rows, d), generator=g).to(torch.bfloat16).to(DEV)
    keys = [(2.0 * torch.randn((b, hkv, n, d), generator=g)).to(torch.bfloat16)
            .to(DEV) for _ in range(p)]
    heads = [i % hkv for i in range(p)]
    return q, keys, heads


def test_noalloc_matches_workspace_call_twice():
    cases = [(3, 2, 4, 64, 3000, 2, 11),      # draft-like: rows = gamma
             (2, 4, 1, 128, 5000, 4, 12)]     # target-like: one row
    for p, b, rows, d, n, hkv, seed in cases:
        q, keys, heads = _case(p, b, rows, d, n, hkv, seed)
        scale = d ** -0.5
        ref = H.score(q, keys, heads, scale, n)          # caller workspace
        got = torch.full((b, n), float("nan"), device=DEV)
        N.dustin_score_heads_noalloc(q, [N.kv_desc(k) for k in keys], heads,
                                     scale, got, n)
        torch.cuda.synchronize()
        np.testing.assert_allclose(H.f64(got), H.f64(ref), rtol=2e-4,
                                   atol=1e-7)
        np.testing.assert_allclose(H.f64(got).sum(axis=1), p * rows,
                                   rtol=1e-4)
        # and against the oracle directly, at the scoring parity tolerance
        want = O.score_heads([H.f64(q[i].cpu()) for i in range(p)],
                             [H.f64(keys[i][:, heads[i]].cpu()) for i in range(p)],
                             scale)
        np.testing.assert_allclose(H.f64(got), want, rtol=2e-4, atol=1e-7)


def test_noalloc_rejects_sizes_beyond_the_array():
    """A valid call whose scratch would overflow the built-in array is
    refused with DUSTIN_ERR_WORKSPACE before anything runs (the pointers
    below are never dereferenced)."""
    lib = N.load()
    b, n, pairs, rows, d = 16, 65536, 64, 1, 128  # 256 MiB of logits
    heads = (ctypes.c_int32 * pairs)(*([0] * pairs))
    desc = N.DustinKV()
    desc.k = desc.v = 0x10000
    desc.stride_n, desc.stride_h, desc.stride_b = d, n * d, 8 * n * d
    arr = (N.DustinKV * pairs)(*([desc] * pairs))
    need = N.dustin_score_heads_workspace_size(b, n, pairs, rows)
    cap = N.noalloc_scratch_bytes()
    assert need > cap
    status = lib.dustin_score_heads_noalloc(
        b, n, d, pairs, rows, 0x10000, ctypes.addressof(arr),
        ctypes.addressof(heads), 0.1, 0x10000, None)
    assert status == 4                            # DUSTIN_ERR_WORKSPACE
    msg = lib.dustin_last_error().decode()
    assert str(cap) in msg and str(need) in msg
