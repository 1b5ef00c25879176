"""Seeded synthetic inputs for the Dustin sparse-verification hot path.

This module is the only code shared by the CUDA path's callers (tests, bench)
and the CPU oracle's callers.  It draws random tensors and lays them out; it
holds none of the method's arithmetic (no attention, scoring, mixing or
selection).

Recipe (stands in for the PG-19 / LongBench long-context inputs the paper
evaluates on, which are not available here):

* Q, K, V ~ N(0, 1), rounded to bf16 (round-to-nearest-even, torch ``.to``).
* Heavy hitters: a fraction ``hh_frac`` of history positions per sequence
  (the same positions in every layer, kv-head and in the draft cache, since
  draft and target share a tokenizer) get ``K_j += hh_scale * u``, where ``u``
  is the unit mean of that kv-head's query rows (verification rows for the
  target, lookahead rows for the draft).  This makes attention peaked, as in
  the paper's Fig. 2-4 ARR curves.
* Sink bias: positions ``j < n_sink_bias`` get ``K_j += sink_scale * u``.
* Drift (saliency shift): the historical scoring queries are built to look at
  heavy hitters displaced by a uniform integer in ``[-drift, drift]`` from the
  positions the verification window looks at.
* Scored (layer, head) pairs: a seeded uniform choice without replacement.
* Paged KV: page size 16 and a seeded random permutation page table.

Seeds: ``1234 + config id``; layer ``l`` of a config folds ``l`` into the seed.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Dict, List, Optional, Tuple

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload shaped like a Qwen2.5 target plus a 0.5B draft."""

    name: str
    config_id: int
    b: int                 # batch (sequences)
    n: int                 # history length (KV positions)
    hq: int                # target query heads
    hkv: int               # target kv heads
    d: int                 # target head dim
    layers: int            # target layers
    w: int                 # verification rows per sequence (= gamma + 1)
    k: int                 # KV budget per sequence
    n_sink: int            # always-kept leading positions
    n_recent: int          # always-kept trailing positions
    alpha: float           # hybrid weight on the draft signal
    p_t: int               # scored target (layer, head) pairs
    p_d: int               # scored draft (layer, head) pairs
    draft_hq: int = 14
    draft_hkv: int = 2
    draft_d: int = 64
    draft_layers: int = 24
    m: int = -1            # draft share of the budget (-1: alpha mode)
    hh_frac: float = 0.01
    hh_scale: float = 3.0
    sink_scale: float = 6.0
    n_sink_bias: int = 4
    drift: int = 0

    @property
    def gamma(self) -> int:
        return self.w - 1

    @property
    def group(self) -> int:
        return self.hq // self.hkv

    @property
    def draft_group(self) -> int:
        return self.draft_hq // self.draft_hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def draft_scale(self) -> float:
        return 1.0 / math.sqrt(self.draft_d)

    @property
    def seed(self) -> int:
        return 1234 + self.config_id

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


WORKLOADS: Dict[str, Workload] = {
    # 1 layer, batch 1, n=256, target 4/2 heads d=64, draft 2/1 heads d=64,
    # gamma=3 (w=4), k=32, 2 sinks + 8 recent, alpha=0.5, 2% heavy hitters.
    "tiny": Workload("tiny", 0, b=1, n=256, hq=4, hkv=2, d=64, layers=1, w=4,
                     k=32, n_sink=2, n_recent=8, alpha=0.5, p_t=2, p_d=2,
                     draft_hq=2, draft_hkv=1, draft_d=64, draft_layers=1,
                     hh_frac=0.02, n_sink_bias=0),
    # Qwen2.5-7B-shaped target, 0.5B draft, b4 n8192 w4 k512, 4+4 pairs.
    "7b": Workload("7b", 1, b=4, n=8192, hq=28, hkv=4, d=128, layers=28, w=4,
                   k=512, n_sink=4, n_recent=64, alpha=0.5, p_t=4, p_d=4),
    # Qwen2.5-32B-shaped target, b16 n16384 w5 k1024, 8 pairs, drift 64.
    "32b": Workload("32b", 2, b=16, n=16384, hq=40, hkv=8, d=128, layers=64,
                    w=5, k=1024, n_sink=4, n_recent=64, alpha=0.5, p_t=4,
                    p_d=4, drift=64),
    # Qwen2.5-72B-shaped target, b16 n32768 w5 k2048, 4+4 pairs, alpha 0.5,
    # 4 sinks + 64 recent: the headline workload.
    "72b": Workload("72b", 3, b=16, n=32768, hq=64, hkv=8, d=128, layers=80,
                    w=5, k=2048, n_sink=4, n_recent=64, alpha=0.5, p_t=4,
                    p_d=4),
}


def sweep_workload(n: int, b: int, w: int, k: int, pairs: int) -> Workload:
    """A point of the 72B-shape sweep (pairs split evenly target/draft)."""
    p_t = max(1, pairs // 2) if pairs > 1 else 1
    p_d = pairs - p_t
    return WORKLOADS["72b"].replace(name=f"sweep_n{n}_b{b}_w{w}_k{k}_p{pairs}",
                                    config_id=4, n=n, b=b, w=w, k=k,
                                    p_t=p_t, p_d=p_d)


# ---------------------------------------------------------------- generators

def generator(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _randn(shape, gen, device) -> torch.Tensor:
    return torch.randn(shape, generator=gen, device=device, dtype=torch.float32)


def heavy_hitter_positions(wl: Workload, device="cpu") -> torch.Tensor:
    """[b][n_hh] int64 heavy-hitter positions per sequence (sorted)."""
    g = generator(wl.seed * 7 + 1, "cpu")
    n_hh = max(1, int(round(wl.hh_frac * wl.n))) if wl.n > 0 else 0
    lo = wl.n_sink_bias
    rows = []
    for _ in range(wl.b):
        span = max(wl.n - lo, 1)
        perm = torch.randperm(span, generator=g)[:min(n_hh, span)] + lo
        rows.append(torch.sort(perm).values)
    if not rows or n_hh == 0:
        return torch.zeros((wl.b, 0), dtype=torch.int64, device=device)
    return torch.stack(rows).to(device)


def _plant(keys32: torch.Tensor, queries32: torch.Tensor, rows_per_kv: int,
           positions: torch.Tensor, scale: float, sink_n: int,
           sink_scale: float) -> None:
    """In place: shift heavy-hitter and sink keys along the kv-head's mean
    query direction.  keys32 [b][hkv][n][d]; queries32 [b][hkv*rows][d]."""
    b, hkv, n, d = keys32.shape
    mean = queries32.reshape(b, hkv, rows_per_kv, d).mean(dim=2)
    unit = mean / mean.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    if positions.numel() > 0 and scale != 0.0:
        pos = positions.clamp(max=max(n - 1, 0))
        bi = torch.arange(b, device=keys32.device)[:, None, None]
        hi = torch.arange(hkv, device=keys32.device)[None, :, None]
        pi = pos[:, None, :]
        keys32[bi, hi, pi] += scale * unit[:, :, None, :]
    if sink_n > 0 and sink_scale != 0.0 and n > 0:
        s = min(sink_n, n)
        keys32[:, :, :s] += sink_scale * unit[:, :, None, :]


def target_layer(wl: Workload, layer: int, device="cpu",
                 hh: Optional[torch.Tensor] = None
                 ) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Q [b][hq][w][d], K and V [b][hkv][n][d], all bf16, for one layer."""
    gen = generator(wl.seed * 1000 + 17 * layer + 3, device)
    q = _randn((wl.b, wl.hq, wl.w, wl.d), gen, device)
    k = _randn((wl.b, wl.hkv, wl.n, wl.d), gen, device)
    v = _randn((wl.b, wl.hkv, wl.n, wl.d), gen, device)
    if hh is None:
        hh = heavy_hitter_positions(wl, device)
    q = q.to(torch.bfloat16)
    _plant(k, q.float().reshape(wl.b, wl.hq * wl.w, wl.d), wl.group * wl.w,
           hh.to(device), wl.hh_scale, wl.n_sink_bias, wl.sink_scale)
    return q, k.to(torch.bfloat16), v.to(torch.bfloat16)


def draft_layer(wl: Workload, layer: int, device="cpu",
                hh: Optional[torch.Tensor] = None
                ) -> Tuple[torch.Tensor, torch.Tensor]:
    """Draft lookahead queries [b][draft_hq][gamma][dd] and draft K
    [b][draft_hkv][n][dd], bf16, for one draft layer."""
    gen = generator(wl.seed * 1000 + 17 * layer + 500_001, device)
    g = max(wl.gamma, 1)
    q = _randn((wl.b, wl.draft_hq, g, wl.draft_d), gen, device)
    k = _randn((wl.b, wl.draft_hkv, wl.n, wl.draft_d), gen, device)
    if hh is None:
        hh = heavy_hitter_positions(wl, device)
    q = q.to(torch.bfloat16)
    _plant(k, q.float().reshape(wl.b, wl.draft_hq * g, wl.draft_d),
           wl.draft_group * g, hh.to(device), wl.hh_scale, wl.n_sink_bias,
           wl.sink_scale)
    return q, k.to(torch.bfloat16)


def scored_pairs(wl: Workload) -> Tuple[List[Tuple[int, int]],
                                         List[Tuple[int, int]]]:
    """Seeded (layer, q_head) pairs for the target and the draft."""
    g = generator(wl.seed * 31 + 5, "cpu")

    def pick(layers: int, heads: int, count: int) -> List[Tuple[int, int]]:
        total = layers * heads
        count = min(count, total)
        flat = torch.randperm(total, generator=g)[:count].tolist()
        return sorted((f // heads, f % heads) for f in flat)

    return pick(wl.layers, wl.hq, wl.p_t), pick(wl.draft_layers, wl.draft_hq,
                                                 wl.p_d)


def historical_query(wl: Workload, q_layer: torch.Tensor, head: int,
                     device="cpu") -> torch.Tensor:
    """The target's latest-token query for one scored head, [b][1][d] bf16.

    It is the first verification row of that head (the last accepted token),
    or, with drift, a fresh draw, since the historical signal then looks at
    displaced positions."""
    if wl.drift == 0:
        return q_layer[:, head, 0:1, :].contiguous()
    gen = generator(wl.seed * 977 + head, device)
    return _randn((wl.b, 1, wl.d), gen, device).to(torch.bfloat16)


def drifted_positions(wl: Workload, hh: torch.Tensor) -> torch.Tensor:
    """Heavy-hitter positions moved by a seeded uniform integer in
    [-drift, drift], clamped to the history (saliency shift)."""
    if wl.drift == 0 or hh.numel() == 0:
        return hh
    g = generator(wl.seed * 13 + 11, "cpu")
    delta = torch.randint(-wl.drift, wl.drift + 1, tuple(hh.shape),
                          generator=g).to(hh.device)
    return (hh + delta).clamp(wl.n_sink_bias, max(wl.n - 1, 0))


def plant_historical(wl: Workload, keys: torch.Tensor, q_hist: torch.Tensor,
                     kv_head: int, positions: torch.Tensor) -> torch.Tensor:
    """With drift, make the historical query prefer the drifted positions:
    K[b, kv_head, pos] += hh_scale * unit(q_hist[b]).  Returns new bf16 K."""
    if wl.drift == 0 or positions.numel() == 0:
        return keys
    k32 = keys.float()
    qh = q_hist.float().reshape(wl.b, 1, -1)
    unit = qh / qh.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    bi = torch.arange(wl.b, device=keys.device)[:, None]
    k32[bi, kv_head, positions.to(keys.device)] += wl.hh_scale * unit
    return k32.to(torch.bfloat16)


def random_sorted_indices(b: int, n: int, k: int, seed: int,
                          device="cpu") -> torch.Tensor:
    """[b][min(k, n)] int32, strictly ascending, each row a seeded random
    subset of [0, n)."""
    g = generator(seed, "cpu")
    kk = min(k, n)
    rows = [torch.sort(torch.randperm(n, generator=g)[:kk]).values
            for _ in range(b)]
    if kk == 0:
        return torch.zeros((b, 0), dtype=torch.int32, device=device)
    return torch.stack(rows).to(torch.int32).to(device)


def synthetic_scores(b: int, n: int, seed: int, ties: bool = True,
                     specials: bool = False) -> torch.Tensor:
    """[b][n] fp32 score vectors shaped like summed softmax rows: a
    log-normal body, a few large entries, and (optionally) planted exact
    ties and special values (+0/-0, NaN, +/-inf)."""
    g = generator(seed, "cpu")
    s = torch.exp(2.0 * torch.randn((b, n), generator=g)) / max(n, 1)
    if n > 0:
        spikes = torch.randint(0, n, (b, max(1, n // 50)), generator=g)
        s.scatter_(1, spikes, 0.05)
    if ties and n > 1:
        # Quantise a third of the entries onto a coarse grid: many exact ties.
        sel = torch.rand((b, n), generator=g) < 0.33
        q = torch.round(s * n * 4.0) / (n * 4.0)
        s = torch.where(sel, q, s)
    s = s.to(torch.float32)
    if specials and n >= 8:
        for r in range(b):
            cols = torch.randperm(n, generator=g)[:6]
            s[r, cols[0]] = 0.0
            s[r, cols[1]] = -0.0
            s[r, cols[2]] = float("nan")
            s[r, cols[3]] = float("inf")
            s[r, cols[4]] = float("-inf")
            s[r, cols[5]] = -0.0
    return s


def to_paged(keys: torch.Tensor, values: Optional[torch.Tensor],
             page_size: int, seed: int
             ) -> Tuple[torch.Tensor, Optional[torch.Tensor], torch.Tensor]:
    """Scatter contiguous [b][hkv][n][d] caches into a page pool
    [P][hkv][page_size][d] with a seeded random page table [b][n/page_size]
    (int32).  The pool holds one spare page so page ids are not a plain
    identity."""
    b, hkv, n, d = keys.shape
    pages = (n + page_size - 1) // page_size
    total = b * pages + 1
    g = generator(seed, "cpu")
    perm = torch.randperm(total, generator=g)[: b * pages]
    table = perm.reshape(b, pages).to(torch.int32)

    def scatter(x: torch.Tensor) -> torch.Tensor:
        pool = torch.zeros((total, hkv, page_size, d), dtype=x.dtype,
                           device=x.device)
        pad = pages * page_size - n
        xp = torch.nn.functional.pad(x, (0, 0, 0, pad)) if pad else x
        xp = xp.reshape(b, hkv, pages, page_size, d).permute(0, 2, 1, 3, 4)
        pool[table.reshape(-1).long().to(x.device)] = xp.reshape(
            b * pages, hkv, page_size, d)
        return pool

    return scatter(keys), (scatter(values) if values is not None else None), \
        table.to(keys.device)


# ------------------------------------------------------------ one decode step

@dataclasses.dataclass
class StepInputs:
    """Every tensor one pass of the hot path reads, for one workload.

    q[i], k[i], v[i]: target layer ``layer_ids[i]``'s verification queries
    [b][hq][w][d] and KV [b][hkv][n][d].  q_t [p_t][b][1][d] are the scored
    target heads' latest-token queries, k_t[p] the key cache their pair reads
    at kv head kvh_t[p].  q_d [p_d][b][gamma][dd] and k_d / kvh_d likewise for
    the draft's lookahead queries."""
    wl: Workload
    layer_ids: List[int]
    q: List[torch.Tensor]
    k: List[torch.Tensor]
    v: List[torch.Tensor]
    pairs_t: List[Tuple[int, int]]
    pairs_d: List[Tuple[int, int]]
    q_t: torch.Tensor
    k_t: List[torch.Tensor]
    kvh_t: List[int]
    q_d: torch.Tensor
    k_d: List[torch.Tensor]
    kvh_d: List[int]
    hh: torch.Tensor


def step_inputs(wl: Workload, device="cpu", n_layers: Optional[int] = None
                ) -> StepInputs:
    """Materialises ``n_layers`` target layers (default: all) and the draft
    layers the scored pairs use.  With fewer layers than the model has, a
    scored pair at layer l reads layer l % n_layers."""
    n_layers = wl.layers if n_layers is None else max(1, min(n_layers,
                                                             wl.layers))
    hh = heavy_hitter_positions(wl, device)
    layer_ids = list(range(n_layers))
    qs, ks, vs = [], [], []
    for l in layer_ids:
        q, k, v = target_layer(wl, l, device, hh)
        qs.append(q)
        ks.append(k)
        vs.append(v)
    pairs_t, pairs_d = scored_pairs(wl)
    pairs_t = [(l % n_layers, h) for l, h in pairs_t]
    q_t_list, kvh_t = [], []
    hh_hist = drifted_positions(wl, hh)
    for l, h in pairs_t:
        qh = historical_query(wl, qs[l], h, device)
        ks[l] = plant_historical(wl, ks[l], qh, h // wl.group, hh_hist)
        q_t_list.append(qh)
        kvh_t.append(h // wl.group)
    k_t = [ks[l] for l, _ in pairs_t]
    draft = {}
    for l, _ in pairs_d:
        if l not in draft:
            draft[l] = draft_layer(wl, l, device, hh)
    q_d = torch.stack([draft[l][0][:, h] for l, h in pairs_d]) if pairs_d \
        else torch.zeros((0, wl.b, max(wl.gamma, 1), wl.draft_d),
                         dtype=torch.bfloat16, device=device)
    k_d = [draft[l][1] for l, _ in pairs_d]
    kvh_d = [h // wl.draft_group for _, h in pairs_d]
    q_t = torch.stack(q_t_list) if q_t_list else torch.zeros(
        (0, wl.b, 1, wl.d), dtype=torch.bfloat16, device=device)
    return StepInputs(wl, layer_ids, qs, ks, vs, pairs_t, pairs_d,
                      q_t.contiguous(), k_t, kvh_t, q_d.contiguous(), k_d,
                      kvh_d, hh)
