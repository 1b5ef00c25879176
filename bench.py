#!/usr/bin/env python3
"""Benchmark of the Dustin sparse-verification hot path on GB300.

One step is one pass of the whole hot path over one batch: score the
target's scored heads (S_Target), score the draft's (S_Draft), the hybrid
Top-K, then the sparse verification attention of every target layer over the
selected KV.  The metric is verified tokens per second per layer,
b * w * layers / step time, on the Qwen2.5-72B-shaped workload (b16, n32768,
w5, k2048, 80 layers, 4 + 4 scored pairs).  The KV cache (172 GB) is resident
in HBM: each step's queries are the per-step inputs.  Inputs are larger than
L2 (80 distinct 2.1 GB layers per step), so no flush is needed.

Also reported: the dense full-cache verification (the in-run baseline),
per-kernel times, the roofline of the sparse attention kernel, an end-to-end
number with the queries copied from pinned host memory and the outputs read
back every step, SM clocks during the timed region, and the CPU oracle timed
on a bounded sample of the same workload.

  python bench.py [--gpus N --steps K --warmup W] [--impl reference]
Under torchrun each rank runs an independent replica (weak scaling).
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = ("verified tokens/s per layer, 72B-shape 32k×b16 k=2048; "
          "HBM GB/s vs peak")
UNIT = "tokens/s/layer"
FALLBACK_HBM_GBS = 6800.0
ATTN_SOURCES = ("attn.cuh", "attn_host.cuh", "device_common.cuh",
                "attn_sparse.cu")
# Machine-readable record of the sparse attention capture (the markdown
# beside it is the human summary of the same capture).
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "sparse_verify_attn_72b.json")


def parse_args(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--config", default="72b")
    p.add_argument("--layers", type=int, default=None,
                   help="target layers to materialise (default: all)")
    p.add_argument("--batch", type=int, default=None,
                   help="override the batch (sequences per GPU)")
    p.add_argument("--dense-steps", type=int, default=3)
    p.add_argument("--no-dense", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu", action="store_true")
    p.add_argument("--sweep", action="store_true",
                   help="time the 72B-shape sweep (n, b, k) and report crossovers")
    p.add_argument("--no-extras", action="store_true",
                   help="skip the window-merge and naive-estimator numbers")
    p.add_argument("--cpu-rows", type=int, default=1)
    p.add_argument("--cpu-layers", type=int, default=2)
    p.add_argument("--cpu-reps", type=int, default=2)
    p.add_argument("--cpu-seconds", type=float, default=12.0,
                   help="approximate CPU work of the oracle leg")
    p.add_argument("--cpu-threads", type=int, default=0,
                   help="oracle threads (0: every core of the affinity mask)")
    p.add_argument("--profile-once", action="store_true",
                   help="launch every kernel of the library once on the workload "
                        "(one target layer), for a profiler's capture")
    p.add_argument("--oracle-worker", action="store_true",
                   help=argparse.SUPPRESS)
    return p.parse_args(argv)


# ----------------------------------------------------------------- helpers

def measured_peak_gbs():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def attn_source_hash() -> str:
    h = hashlib.sha256()
    for name in ATTN_SOURCES:
        with open(os.path.join(ROOT, "sparse_kv_verification_gb300", "csrc",
                               name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def committed_traffic():
    """DRAM bytes per launch of the sparse attention kernel from the
    committed ncu record, if it was taken on the current kernel source."""
    try:
        with open(TRAFFIC_FILE) as f:
            rec = json.load(f)
    except (OSError, ValueError):
        return None
    if rec.get("source_sha") != attn_source_hash():
        return None
    try:
        return float(rec["dram_bytes_per_launch"])
    except (KeyError, TypeError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,"
             "clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
             "clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,"
             "clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.file = None

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv",
                                                    delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index),
                 f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "note": "nvidia-smi unavailable"}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        rows = [r.split(",") for r in self.file.read().splitlines() if r.strip()]
        os.unlink(self.file.name)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for i, name in enumerate(names):
                if len(r) > 5 + i and r[5 + i].strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- replica

class Replica:
    """One GPU's copy of the workload with pre-marshalled library calls."""

    def __init__(self, wl, device, n_layers):
        import torch
        from sparse_kv_verification_gb300 import inputs as I
        from sparse_kv_verification_gb300 import native as N
        self.wl, self.dev = wl, device
        inp = I.step_inputs(wl, device, n_layers)
        self.inp = inp
        self.L = len(inp.layer_ids)
        b, n = wl.b, wl.n
        self.s_t = torch.empty((b, n), device=device)
        self.s_d = torch.empty((b, n), device=device)
        self.idx = torch.empty((b, min(wl.k, n)), dtype=torch.int32,
                               device=device)
        # All layers' queries and outputs live in one contiguous buffer each,
        # so the end-to-end leg moves them with one copy per direction.
        self.q_all = torch.stack(inp.q)
        inp.q = [self.q_all[l] for l in range(self.L)]
        self.o_all = torch.empty_like(self.q_all)
        self.lse_all = torch.empty(self.q_all.shape[:4], device=device)
        self.o = [self.o_all[l] for l in range(self.L)]
        self.lse = [self.lse_all[l] for l in range(self.L)]
        self.ws_t = N.workspace(N.dustin_score_heads_workspace_size(
            b, n, wl.p_t, 1), device)
        self.ws_d = N.workspace(N.dustin_score_heads_workspace_size(
            b, n, wl.p_d, wl.gamma), device)
        self.ws_a = N.workspace(N.dustin_sparse_verify_attn_workspace_size(
            b, wl.hq, wl.hkv, wl.d, wl.w, wl.k), device)
        self.ws_f = N.workspace(N.dustin_full_verify_attn_workspace_size(
            b, wl.hq, wl.hkv, wl.d, wl.w, n), device)
        kv = [N.kv_desc(k, v) for k, v in zip(inp.k, inp.v)]
        self.score_t = N.prepare_score_heads(
            inp.q_t, [N.kv_desc(k) for k in inp.k_t], inp.kvh_t, wl.scale,
            self.s_t, self.ws_t, n)
        self.score_d = N.prepare_score_heads(
            inp.q_d, [N.kv_desc(k) for k in inp.k_d], inp.kvh_d,
            wl.draft_scale, self.s_d, self.ws_d, n)
        self.select = N.prepare_hybrid_topk(
            self.s_d, self.s_t, wl.k, wl.n_sink, wl.n_recent, wl.alpha, wl.m,
            N.DUSTIN_NORM_L1, self.idx)
        # Layer 0 follows the select kernel, which writes idx; every later
        # layer follows the previous layer's attention, which writes only its
        # own outputs, so its K/V gather may start before that one finishes.
        ready = lambda l: N.DUSTIN_ATTN_KV_READY if l > 0 else 0
        self.attn = [N.prepare_sparse_verify_attn(
            inp.q[l], kv[l], wl.hkv, n, self.idx, wl.scale, self.o[l],
            self.lse[l], self.ws_a, flags=ready(l)) for l in range(self.L)]
        self.full = [N.prepare_full_verify_attn(
            inp.q[l], kv[l], wl.hkv, n, wl.scale, self.o[l], self.lse[l],
            self.ws_f, flags=ready(l)) for l in range(self.L)]

    def step(self, ev=None):
        """One pass of the hot path; ev (optional) records events at the
        phase boundaries only (score target | score draft | select | all
        layers' attention), so consecutive kernels keep their programmatic
        dependent launch."""
        if ev is not None:
            ev[0].record()
        self.score_t()
        if ev is not None:
            ev[1].record()
        self.score_d()
        if ev is not None:
            ev[2].record()
        self.select()
        if ev is not None:
            ev[3].record()
        for a in self.attn:
            a()
        if ev is not None:
            ev[4].record()

    # Algorithmic bytes (what the method must move), per launch / per step.
    def bytes_sparse_launch(self):
        wl = self.wl
        kk = min(wl.k, wl.n)
        return (wl.b * wl.hkv * kk * wl.d * 2 * 2 +          # K, V rows
                2 * wl.b * wl.hq * wl.w * wl.d * 2 +           # Q in, O out
                wl.b * wl.hq * wl.w * 4 + wl.b * kk * 4)       # LSE, idx

    def bytes_dense_launch(self):
        wl = self.wl
        return (wl.b * wl.hkv * wl.n * wl.d * 2 * 2 +
                2 * wl.b * wl.hq * wl.w * wl.d * 2 + wl.b * wl.hq * wl.w * 4)

    def bytes_score_t(self):
        wl = self.wl
        return (wl.p_t * wl.b * wl.n * wl.d * 2 + wl.p_t * wl.b * wl.d * 2 +
                wl.b * wl.n * 4)

    def bytes_score_d(self):
        wl = self.wl
        return (wl.p_d * wl.b * wl.n * wl.draft_d * 2 +
                wl.p_d * wl.b * wl.gamma * wl.draft_d * 2 + wl.b * wl.n * 4)

    def bytes_select(self):
        wl = self.wl
        return 2 * wl.b * wl.n * 4 + wl.b * min(wl.k, wl.n) * 4


# ----------------------------------------------------------------- extras

def run_extras(rep, wl, dev, stream, L, args, t_attn, t_dense):
    """Per-layer times of the window-merge entry points (the w x w causal
    block as one more tile of the same launch), the multi-layer launch, one
    step of the naive estimator (every target head of every layer and every
    draft head of every draft layer scored) and of Quest-16."""
    import torch
    from sparse_kv_verification_gb300 import native as N
    inp = rep.inp
    g = torch.Generator(device=dev)
    g.manual_seed(4321)
    shape = (wl.b, wl.hkv, wl.w, wl.d)
    wins = [(torch.randn(shape, generator=g, device=dev).to(torch.bfloat16),
             torch.randn(shape, generator=g, device=dev).to(torch.bfloat16))
            for _ in range(L)]
    kv = [N.kv_desc(k, v) for k, v in zip(inp.k, inp.v)]
    ready = lambda l: N.DUSTIN_ATTN_KV_READY if l > 0 else 0
    sw = [N.prepare_sparse_verify_attn_window(
        inp.q[l], kv[l], wl.hkv, wl.n, rep.idx, N.kv_desc(*wins[l]), wl.scale,
        rep.o[l], rep.lse[l], rep.ws_a, flags=ready(l)) for l in range(L)]
    fw = [N.prepare_full_verify_attn_window(
        inp.q[l], kv[l], wl.hkv, wl.n, N.kv_desc(*wins[l]), wl.scale, rep.o[l],
        rep.lse[l], rep.ws_f, flags=ready(l)) for l in range(L)]

    def time_pass(calls, reps):
        for c in calls:
            c()
        torch.cuda.synchronize(dev)
        e0, e1 = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
        e0.record(stream)
        for _ in range(reps):
            for c in calls:
                c()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / (reps * len(calls))

    t_sw = time_pass(sw, 5)
    # All layers' sparse attention in one persistent launch.
    ml = N.prepare_sparse_verify_attn_layers(
        inp.q, kv, wl.hkv, wl.n, rep.idx, wl.scale, rep.o, rep.lse)
    t_ml = time_pass([ml], 5) / L
    t_fw = time_pass(fw, 1) if not args.no_dense else None
    # Naive estimator: all h_q heads of each layer as that layer's scored
    # pairs (latest-token query, one row), one scoring call per layer.
    hq = wl.hq
    q_all = torch.randn((hq, wl.b, 1, wl.d), generator=g, device=dev).to(torch.bfloat16)
    s_out = torch.empty((wl.b, wl.n), device=dev)
    ws = N.workspace(N.dustin_score_heads_workspace_size(wl.b, wl.n, hq, 1), dev)
    heads = [h // wl.group for h in range(hq)]
    naive = [N.prepare_score_heads(q_all, [N.kv_desc(inp.k[l])] * hq, heads,
                                   wl.scale, s_out, ws, wl.n) for l in range(L)]
    t_naive_layer = time_pass(naive, 1)
    # ... and the draft side: all draft query heads of each draft layer with
    # their Gamma lookahead rows (distinct draft key buffers cycled).
    nbuf_d = min(wl.draft_layers, 6)
    k_draft = [torch.randn((wl.b, wl.draft_hkv, wl.n, wl.draft_d), generator=g,
                           device=dev).to(torch.bfloat16) for _ in range(nbuf_d)]
    q_dall = torch.randn((wl.draft_hq, wl.b, wl.gamma, wl.draft_d), generator=g,
                         device=dev).to(torch.bfloat16)
    ws_nd = N.workspace(N.dustin_score_heads_workspace_size(wl.b, wl.n, wl.draft_hq,
                                                            wl.gamma), dev)
    heads_d = [h // wl.draft_group for h in range(wl.draft_hq)]
    naive_d = [N.prepare_score_heads(q_dall, [N.kv_desc(k_draft[l % nbuf_d])] * wl.draft_hq,
                                     heads_d, wl.draft_scale, s_out, ws_nd, wl.n)
               for l in range(wl.draft_layers)]
    t_naive_draft_layer = time_pass(naive_d, 1)
    del k_draft
    # Quest-16: page statistics (kept up to date at append time in Quest, so
    # timed apart) and, per step and layer, page scores for every query head
    # (latest-token query) plus the top k/16 pages per (sequence, head).
    page = 16
    n_pages = (wl.n + page - 1) // page
    nbuf = min(8, L)
    stats = [N.dustin_quest_page_stats(kv[l], wl.b, wl.hkv, wl.d, wl.n, page,
                                       device=dev) for l in range(nbuf)]
    t_stats = time_pass([lambda l=l: N.dustin_quest_page_stats(
        kv[l], wl.b, wl.hkv, wl.d, wl.n, page, stats=stats[l]) for l in range(nbuf)], 2)
    q_row = torch.randn((wl.b, hq, wl.d), generator=g, device=dev).to(torch.bfloat16)
    scores = torch.empty((wl.b, hq, n_pages), device=dev)
    keep = max(1, wl.k // page)
    pidx = torch.empty((wl.b * hq, keep), dtype=torch.int32, device=dev)
    sel = N.prepare_hybrid_topk(scores.view(wl.b * hq, n_pages), None, keep, 0, 0,
                                1.0, -1, N.DUSTIN_NORM_NONE, pidx)
    quest = []
    for l in range(L):
        quest.append(lambda l=l: N.dustin_quest_page_scores(q_row, stats[l % nbuf],
                                                            wl.n, page, scores=scores))
        quest.append(sel)
    t_quest_layer = time_pass(quest, 1) * 2
    t_qscore = time_pass(quest[0::2], 1)
    t_qsel = time_pass([sel] * 8, 2)
    return {
        "multi_layer_sparse_us_per_layer": t_ml,
        "multi_layer_sparse_gbs": rep.bytes_sparse_launch() / (t_ml * 1e-6) / 1e9,
        "multi_layer_note": (f"all {L} layers in one launch: only for callers that "
                             "hold every layer's queries at once; the headline "
                             "calls one launch per layer"),
        "window_sparse_us_per_layer": t_sw,
        "window_sparse_overhead_us": t_sw - t_attn,
        "window_dense_us_per_layer": t_fw,
        "window_dense_overhead_us": (t_fw - t_dense) if (t_fw and t_dense) else None,
        "quest16_estimator": {
            "what": (f"page scores of all {hq} query heads (latest-token query) "
                     f"over 16-position page min/max statistics, then the top "
                     f"{keep} pages per (sequence, head), for each of {L} layers"),
            "ms_per_step": t_quest_layer * L / 1e3,
            "page_scores_ms_per_step": t_qscore * L / 1e3,
            "page_select_ms_per_step": t_qsel * L / 1e3,
            "ratio_to_dense": (t_quest_layer / t_dense) if t_dense else None,
            "stats_build_us_per_layer": t_stats,
        },
        "naive_estimator": {
            "what": (f"all {hq} target query heads of each of {L} layers (latest-"
                     f"token query) and all {wl.draft_hq} draft heads of each of "
                     f"{wl.draft_layers} draft layers ({wl.gamma} lookahead rows) "
                     "scored, one scoring call per layer"),
            "ms_per_step": (t_naive_layer * L + t_naive_draft_layer * wl.draft_layers) / 1e3,
            "target_ms_per_step": t_naive_layer * L / 1e3,
            "draft_ms_per_step": t_naive_draft_layer * wl.draft_layers / 1e3,
            "dense_attention_ms_per_step": (t_dense * L / 1e3) if t_dense else None,
            "ratio_to_dense": ((t_naive_layer * L + t_naive_draft_layer * wl.draft_layers)
                               / (t_dense * L)) if t_dense else None,
        },
    }


# ----------------------------------------------------------------- sweep

def run_sweep(args):
    """The 72B-shape sweep on paged caches (page 16, seeded random page
    tables): for n in 4K..64K and b in {1, 4, 16, 32} (w = 4, 8 scored
    pairs), the step's scoring (target + draft) and select, and per layer
    the sparse attention for each budget k and the dense attention; then
    w in {2, 4, 8} and scored pairs in {1, 4, 8, 16} at n = 32K, b = 16,
    k = 2048, and the contiguous cache at that point.  Layer buffers are
    cycled so that each pass reads well past L2.  Crossover (amortised over
    80 layers): the smallest tested k/n at which scoring + select + 80
    sparse layers take at least as long as 80 dense layers.  One JSON line
    per point, then a summary line."""
    import torch
    from sparse_kv_verification_gb300 import build, inputs as I, native as N
    build.build()
    N.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    layers_model, page = 80, 16
    ks_all = [256, 512, 1024, 2048, 4096, 8192]

    def timed(calls, reps):
        for c in calls:
            c()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        for _ in range(reps):
            for c in calls:
                c()
        e1.record()
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) * 1e3 / (reps * len(calls))

    def point(n, b, w, pairs, ks, paged=True):
        wl = I.sweep_workload(n, b, w, max(ks), pairs)
        layer_bytes = b * wl.hkv * n * wl.d * 2 * 2
        n_buf = int(min(layers_model, max(3, -(-400_000_000 // layer_bytes))))
        inp = I.step_inputs(wl, dev, n_buf)
        if paged:
            kt = [I.to_paged(k, None, page, seed=100 + i) for i, k in enumerate(inp.k_t)]
            kd = [I.to_paged(k, None, page, seed=200 + i) for i, k in enumerate(inp.k_d)]
            desc_t = [N.kv_desc(pk, None, t) for pk, _, t in kt]
            desc_d = [N.kv_desc(pk, None, t) for pk, _, t in kd]
            kvp = []
            for l in range(n_buf):
                kvp.append(I.to_paged(inp.k[l], inp.v[l], page, seed=300 + l))
                inp.k[l] = inp.v[l] = None   # keep only the paged copy
            kvs = [N.kv_desc(pk, pv, t) for pk, pv, t in kvp]
        else:
            kt = kd = kvp = None
            desc_t = [N.kv_desc(k) for k in inp.k_t]
            desc_d = [N.kv_desc(k) for k in inp.k_d]
            kvs = [N.kv_desc(k, v) for k, v in zip(inp.k, inp.v)]
        s_t = torch.empty((b, n), device=dev)
        s_d = torch.empty((b, n), device=dev)
        ws_t = N.workspace(N.dustin_score_heads_workspace_size(b, n, wl.p_t, 1), dev)
        ws_d = N.workspace(N.dustin_score_heads_workspace_size(b, n, max(1, wl.p_d),
                                                                wl.gamma), dev)
        sc_t = N.prepare_score_heads(inp.q_t, desc_t, inp.kvh_t, wl.scale, s_t, ws_t, n)
        t_score = timed([sc_t], 5)
        alpha = wl.alpha
        if wl.p_d > 0:
            sc_d = N.prepare_score_heads(inp.q_d, desc_d, inp.kvh_d, wl.draft_scale, s_d,
                                         ws_d, n)
            t_score += timed([sc_d], 5)
        else:   # a single scored pair: the target's, selected on its own
            s_d, alpha = None, 0.0
        o = [torch.empty_like(q) for q in inp.q]
        lse = [torch.empty(q.shape[:3], device=dev) for q in inp.q]
        ws_f = N.workspace(N.dustin_full_verify_attn_workspace_size(
            b, wl.hq, wl.hkv, wl.d, w, n), dev)
        ready = lambda l: N.DUSTIN_ATTN_KV_READY if l > 0 else 0
        dense = [N.prepare_full_verify_attn(inp.q[l], kvs[l], wl.hkv, n, wl.scale, o[l],
                                            lse[l], ws_f, flags=ready(l))
                 for l in range(n_buf)]
        t_dense = timed(dense, max(1, 6 // n_buf + 1))
        points = []
        for k in ks:
            idx = torch.empty((b, k), dtype=torch.int32, device=dev)
            sel = N.prepare_hybrid_topk(s_d, s_t, k, wl.n_sink, wl.n_recent, alpha,
                                        wl.m, N.DUSTIN_NORM_L1, idx)
            t_sel = timed([sel], 5)
            ws_a = N.workspace(N.dustin_sparse_verify_attn_workspace_size(
                b, wl.hq, wl.hkv, wl.d, w, k), dev)
            sparse = [N.prepare_sparse_verify_attn(inp.q[l], kvs[l], wl.hkv, n, idx,
                                                   wl.scale, o[l], lse[l], ws_a,
                                                   flags=ready(l))
                      for l in range(n_buf)]
            t_sp = timed(sparse, max(1, 30 // n_buf + 1))
            est = t_score + t_sel
            points.append({
                "k": k, "k_over_n": k / n, "select_us": t_sel, "sparse_us_per_layer": t_sp,
                "speedup_attention_per_layer": t_dense / t_sp,
                "speedup_amortised_80": layers_model * t_dense /
                                        (est + layers_model * t_sp),
                "speedup_estimation_charged_to_one_layer": t_dense / (est + t_sp),
            })
        cross = next((p["k_over_n"] for p in points if p["speedup_amortised_80"] <= 1.0),
                     None)
        cross1 = next((p["k_over_n"] for p in points
                       if p["speedup_estimation_charged_to_one_layer"] <= 1.0), None)
        line = {"sweep": True, "n": n, "b": b, "w": w, "pairs": pairs,
                "kv": f"paged{page}" if paged else "contiguous",
                "layer_buffers": n_buf, "score_us": t_score,
                "dense_us_per_layer": t_dense, "points": points,
                "crossover_k_over_n_amortised": cross,
                "crossover_k_over_n_charged_to_one_layer": cross1}
        print(json.dumps(line), flush=True)
        del inp, kvs, o, lse, dense, sparse, kt, kd, kvp, desc_t, desc_d
        torch.cuda.empty_cache()
        return line

    grid = []
    for n in (4096, 8192, 16384, 32768, 65536):
        for b in (1, 4, 16, 32):
            grid.append(point(n, b, 4, 8, [k for k in ks_all if k < n]))
    by_w = [point(32768, 16, w, 8, [2048]) for w in (2, 4, 8)]
    by_pairs = [point(32768, 16, 4, p, [2048]) for p in (1, 4, 8, 16)]
    contiguous = point(32768, 16, 4, 8, [2048], paged=False)
    key = lambda l: f"n{l['n']}_b{l['b']}"
    summary = {"sweep_summary": True,
               "crossovers_amortised_80": {key(l): l["crossover_k_over_n_amortised"]
                                           for l in grid},
               "crossovers_charged_to_one_layer": {
                   key(l): l["crossover_k_over_n_charged_to_one_layer"] for l in grid},
               "sparse_us_by_w": {l["w"]: l["points"][0]["sparse_us_per_layer"]
                                  for l in by_w},
               "score_us_by_pairs": {l["pairs"]: l["score_us"] for l in by_pairs},
               "paged16_vs_contiguous_sparse_us": {
                   "paged": by_w[1]["points"][0]["sparse_us_per_layer"],
                   "contiguous": contiguous["points"][0]["sparse_us_per_layer"]},
               "paged16_vs_contiguous_dense_us": {
                   "paged": by_w[1]["dense_us_per_layer"],
                   "contiguous": contiguous["dense_us_per_layer"]}}
    print(json.dumps(summary), flush=True)
    return 0


def host_cores() -> int:
    """Cores this process may run on (the affinity mask, not the machine)."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


# Oracle leg state shared with forked children (copy-on-write, read-only).
_ORACLE = {}


def _oracle_estimate(_):
    O, c = _ORACLE["O"], _ORACLE
    s_t = O.score_heads(c["q_t"], c["k_t"], c["scale"])
    s_d = O.score_heads(c["q_d"], c["k_d"], c["draft_scale"])
    sp = c["sample"]
    return O.hybrid_select(s_d, s_t, sp.k, sp.n_sink, sp.n_recent, sp.alpha, sp.m,
                           O.NORM_L1)


def _oracle_attend(_):
    O, c = _ORACLE["O"], _ORACLE
    for q, k, v in c["layers"]:
        O.verify_attention(q, k, v, c["idx"], c["scale"])
    return 0


def oracle_worker(args):
    """Runs inside a fresh process that never touches a GPU: the CPU oracle,
    as it stands, on a bounded sample of the workload, on every host core.
    The inputs are generated once, then one process per core (forked after
    the inputs exist and before any GPU use, sharing them copy-on-write)
    runs one sequence's scoring, selection and attention per repetition;
    the oracle code stays one plain path and only this driver loop is
    parallel.  BLAS and torch are single-threaded in every process."""
    import multiprocessing
    import torch
    torch.set_num_threads(1)
    from oracle import dustin_oracle as O
    from sparse_kv_verification_gb300 import inputs as I
    wl = I.WORKLOADS[args.config]
    if args.batch:
        wl = wl.replace(b=args.batch)
    full_layers = wl.layers
    cores = max(1, min(host_cores(), args.cpu_threads or host_cores()))
    # One seeded sequence of the workload; every process works through its
    # own copy's worth of work over these arrays.
    sample = wl.replace(b=args.cpu_rows)
    inp = I.step_inputs(sample, "cpu", args.cpu_layers)
    f = lambda t: t.to(torch.float64).numpy()
    _ORACLE.update(
        O=O, sample=sample, scale=sample.scale, draft_scale=sample.draft_scale,
        q_t=[f(inp.q_t[i]) for i in range(sample.p_t)],
        k_t=[f(k[:, h]) for k, h in zip(inp.k_t, inp.kvh_t)],
        q_d=[f(inp.q_d[i]) for i in range(sample.p_d)],
        k_d=[f(k[:, h]) for k, h in zip(inp.k_d, inp.kvh_d)],
        layers=[(f(q), f(k), f(v)) for q, k, v in zip(inp.q, inp.k, inp.v)])
    del inp
    _ORACLE["idx"] = _oracle_estimate(0)
    n_layers = len(_ORACLE["layers"])

    times = []
    t_begin = time.perf_counter()
    reps = 0
    with multiprocessing.get_context("fork").Pool(cores) as pool:
        # Time-bounded: at least cpu_reps repetitions and about cpu_seconds
        # of oracle work (capped at 200 repetitions).
        while reps < args.warmup + args.cpu_reps or (
                time.perf_counter() - t_begin < args.cpu_seconds and reps < 200):
            reps += 1
            t0 = time.perf_counter()
            pool.map(_oracle_estimate, range(cores), chunksize=1)
            t1 = time.perf_counter()
            pool.map(_oracle_attend, range(cores), chunksize=1)
            t2 = time.perf_counter()
            times.append((t1 - t0, (t2 - t1) / n_layers))
    times = times[min(args.warmup, len(times) - 1):]
    t_est = statistics.median(t[0] for t in times)
    t_attn = statistics.median(t[1] for t in times)
    t_step = t_est + full_layers * t_attn
    seqs = cores * sample.b
    value = seqs * sample.w * full_layers / t_step
    print(json.dumps({
        "value": value, "t_step_s": t_step, "t_estimate_s": t_est,
        "t_attn_layer_s": t_attn, "cores": cores,
        "wall_s": sum(t[0] + t[1] * n_layers for t in times),
        "sample": (f"{seqs} sequences ({cores} processes, one per host core, each "
                   f"running the oracle on the same seeded sequence) x {n_layers} of "
                   f"{full_layers} layers timed ({len(times)} reps, median); scoring "
                   f"and selection once per step, attention extrapolated to "
                   f"{full_layers} layers; numpy fp64")}))


def run_oracle_leg(args, reps, warmup):
    env = dict(os.environ, OPENBLAS_NUM_THREADS="1", OMP_NUM_THREADS="1",
               MKL_NUM_THREADS="1", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, os.path.abspath(__file__), "--oracle-worker",
           "--config", args.config, "--cpu-rows", str(args.cpu_rows),
           "--cpu-layers", str(args.cpu_layers), "--cpu-reps", str(reps),
           "--warmup", str(warmup), "--cpu-seconds", str(args.cpu_seconds),
           "--cpu-threads", str(args.cpu_threads)]
    if args.batch:
        cmd += ["--batch", str(args.batch)]
    r = subprocess.run(cmd, capture_output=True, text=True, env=env)
    if r.returncode != 0:
        raise RuntimeError("oracle leg failed:\n" + r.stderr[-2000:])
    return json.loads(r.stdout.strip().splitlines()[-1])


# ----------------------------------------------------------------- arms

def e2e_chunk_bounds(L):
    """Layer boundaries of the end-to-end copy chunks: chunks of up to 8
    layers, shrinking to 4, 2, 1, 1 layers at the end, so that little output
    is left to copy after the last kernel."""
    tail = []
    for size in (1, 1, 2, 4):
        if sum(tail) + size <= L // 2:
            tail.insert(0, size)
    head = L - sum(tail)
    n_head = -(-head // 8) if head else 0
    sizes = [head * (c + 1) // n_head - head * c // n_head
             for c in range(n_head)] + tail
    bounds = [0]
    for size in sizes:
        bounds.append(bounds[-1] + size)
    return bounds


def l2_note(wl, n_layers):
    """How the timed steps avoid reading from a warm L2 (129 MB)."""
    layer_gb = wl.b * wl.hkv * wl.n * wl.d * 2 * 2 / 1e9
    if n_layers * layer_gb * 1e9 > 129e6:
        return (f"inputs larger than L2: every step reads {n_layers} distinct "
                f"layers of {layer_gb:.3g} GB KV")
    return (f"inputs within L2 ({n_layers} layers of {layer_gb * 1e3:.3g} MB KV): "
            "a small case, not a bandwidth measurement")


def workload_config(wl, n_layers):
    return {"workload": (f"{wl.name}: Qwen2.5-shaped target h_q{wl.hq}/h_kv"
                         f"{wl.hkv} d{wl.d}, 0.5B-shaped draft h_q{wl.draft_hq}"
                         f"/h_kv{wl.draft_hkv} d{wl.draft_d}; b{wl.b} n{wl.n} "
                         f"w{wl.w} k{wl.k}; {n_layers} layers; {wl.p_t}+"
                         f"{wl.p_d} scored pairs; alpha {wl.alpha}; "
                         f"{wl.n_sink} sinks + {wl.n_recent} recent"),
            "b": wl.b, "n": wl.n, "w": wl.w, "k": wl.k, "layers": n_layers,
            "h_q": wl.hq, "h_kv": wl.hkv, "d": wl.d,
            "l2": l2_note(wl, n_layers),
            "parallelism": "replicas: each GPU runs its own batch, no "
                           "data-path collective"}


def run_reference(args):
    from sparse_kv_verification_gb300 import inputs as I
    from sparse_kv_verification_gb300 import replicas as R
    rank, _, world = R.env_rank()
    if rank != 0:
        return 0
    wl = I.WORKLOADS[args.config]
    if args.batch:
        wl = wl.replace(b=args.batch)
    res = run_oracle_leg(args, max(1, args.steps), max(0, args.warmup))
    line = {"impl": "reference", "metric": METRIC, "value": res["value"],
            "unit": UNIT, "n_gpus": args.gpus, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": res["t_step_s"] * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64", "data": "synthetic",
            "config": workload_config(wl, wl.layers),
            "cpu_baseline": {"value": res["value"], "unit": UNIT,
                             "cores": res["cores"], "kind": "oracle",
                             "sample": res["sample"]},
            "e2e": {"value": res["value"], "unit": UNIT,
                    "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    from sparse_kv_verification_gb300 import build
    from sparse_kv_verification_gb300 import inputs as I
    from sparse_kv_verification_gb300 import native as N
    from sparse_kv_verification_gb300 import replicas as R

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    build.build()
    N.load()
    rank, local, world = R.env_rank()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    R.init("nccl")

    wl = I.WORKLOADS[args.config]
    if args.batch:
        wl = wl.replace(b=args.batch)
    n_layers = args.layers or wl.layers
    rep = Replica(wl, dev, n_layers)
    L = rep.L
    K, W = args.steps, max(3, args.warmup)
    stream = torch.cuda.current_stream(dev)

    for _ in range(W):
        rep.step()
    torch.cuda.synchronize(dev)

    # ---- timed region: K steps, per-phase events on the launch stream.
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(5)]
           for _ in range(K)]
    start, end = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    R.barrier(dev)
    torch.cuda.synchronize(dev)
    launches0 = N.dustin_launch_count()
    start.record(stream)
    for i in range(K):
        rep.step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    launches = N.dustin_launch_count() - launches0
    R.barrier(dev)
    clock_info = clocks.stop()
    t_ms = R.reduce_max(start.elapsed_time(end) / K, dev)

    def med(a, b):
        """Median over the K timed steps of one phase, in microseconds."""
        return statistics.median(evs[i][a].elapsed_time(evs[i][b])
                                 for i in range(K)) * 1e3
    t_score_t = med(0, 1)
    t_score_d = med(1, 2)
    t_select = med(2, 3)
    # Launch duration of the sparse attention: the attention phase of each
    # step divided by its launches (back-to-back launches; the gaps between
    # them are included, so this is conservative), median over the steps.
    t_attn = med(3, 4) / L
    t_step_median = med(0, 4) / 1e3   # ms

    tokens = wl.b * wl.w * L
    value = R.reduce_sum(tokens, dev) / (t_ms * 1e-3)
    peak, peak_kind = measured_peak_gbs()
    b_attn = rep.bytes_sparse_launch()
    achieved = b_attn / (t_attn * 1e-6) / 1e9

    # ---- dense in-run baseline: every layer over the full cache.
    dense = None
    if not args.no_dense:
        for full in rep.full[:2]:
            full()
        torch.cuda.synchronize(dev)
        ds = [(torch.cuda.Event(enable_timing=True),
               torch.cuda.Event(enable_timing=True))
              for _ in range(args.dense_steps)]
        for i in range(args.dense_steps):
            ds[i][0].record()
            for full in rep.full:
                full()
            ds[i][1].record()
        torch.cuda.synchronize(dev)
        t_dense = statistics.median(a.elapsed_time(b) * 1e3 / L for a, b in ds)
        b_dense = rep.bytes_dense_launch()
        t_est = t_score_t + t_score_d + t_select
        dense = {"us_per_layer": t_dense,
                 "hbm_gbs": b_dense / (t_dense * 1e-6) / 1e9,
                 "frac_of_peak": b_dense / (t_dense * 1e-6) / 1e9 / peak,
                 f"ms_per_step_{L}_layers": t_dense * L / 1e3,
                 # the three speedups of the hot-path table's measurement row
                 "speedup_attention_per_layer": t_dense / t_attn,
                 "speedup_step": t_dense * L / 1e3 / t_ms,
                 "estimation_us": t_est,
                 "speedup_estimation_charged_to_one_layer":
                     t_dense / (t_est + t_attn)}

    # ---- end to end: queries from pinned host memory in, outputs out.
    # Copies run on two copy streams beside the compute stream, in chunks
    # of layers: the scoring queries and the first layers' queries go in
    # first, each chunk's attention waits only for its own queries, and
    # each chunk's outputs go out as soon as they are written.  A step waits
    # for the previous step's copies on both sides, so nothing crosses step
    # boundaries and every byte is inside the step's timed region.
    e2e = None
    if not args.no_e2e:
        inp = rep.inp
        L = rep.L
        bounds = e2e_chunk_bounds(L)
        n_chunks = len(bounds) - 1
        h_qt, h_qd = inp.q_t.cpu().pin_memory(), inp.q_d.cpu().pin_memory()
        h_q = rep.q_all.cpu().pin_memory()
        h_o = torch.empty(rep.o_all.shape, dtype=rep.o_all.dtype, pin_memory=True)
        h_lse = torch.empty(rep.lse_all.shape, dtype=rep.lse_all.dtype,
                            pin_memory=True)
        h_idx = torch.empty(rep.idx.shape, dtype=rep.idx.dtype, pin_memory=True)
        h2d = sum(t.numel() * t.element_size() for t in (h_qt, h_qd, h_q))
        d2h = sum(t.numel() * t.element_size() for t in (h_o, h_lse, h_idx))
        s_in = torch.cuda.Stream(dev)
        s_out = torch.cuda.Stream(dev)
        ev = lambda: torch.cuda.Event()

        def e2e_step():
            s_in.wait_stream(stream)      # this step's inputs replace the last
            stream.wait_stream(s_out)     # the last step's outputs are out
            with torch.cuda.stream(s_in):
                inp.q_t.copy_(h_qt, non_blocking=True)
                inp.q_d.copy_(h_qd, non_blocking=True)
                in_ev = [ev()]
                in_ev[0].record(s_in)
                for c in range(n_chunks):
                    a, b = bounds[c], bounds[c + 1]
                    rep.q_all[a:b].copy_(h_q[a:b], non_blocking=True)
                    in_ev.append(ev())
                    in_ev[-1].record(s_in)
            stream.wait_event(in_ev[0])
            rep.score_t()
            rep.score_d()
            rep.select()
            sel_ev = ev()
            sel_ev.record(stream)
            out_ev = []
            for c in range(n_chunks):
                stream.wait_event(in_ev[c + 1])
                for l in range(bounds[c], bounds[c + 1]):
                    rep.attn[l]()
                out_ev.append(ev())
                out_ev[-1].record(stream)
            with torch.cuda.stream(s_out):
                s_out.wait_event(sel_ev)
                h_idx.copy_(rep.idx, non_blocking=True)
                for c in range(n_chunks):
                    a, b = bounds[c], bounds[c + 1]
                    s_out.wait_event(out_ev[c])
                    h_o[a:b].copy_(rep.o_all[a:b], non_blocking=True)
                    h_lse[a:b].copy_(rep.lse_all[a:b], non_blocking=True)
            stream.wait_stream(s_out)     # the step ends when its outputs are out
        for _ in range(W):
            e2e_step()
        torch.cuda.synchronize(dev)
        R.barrier(dev)
        e0, e1 = (torch.cuda.Event(enable_timing=True),
                  torch.cuda.Event(enable_timing=True))
        e0.record(stream)
        for _ in range(K):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        # The copies of the last step landed: host outputs equal the device's.
        assert torch.equal(h_o, rep.o_all.cpu()) and torch.equal(h_idx, rep.idx.cpu())
        t_e2e = R.reduce_max(e0.elapsed_time(e1) / K, dev)
        e2e = {"value": R.reduce_sum(tokens, dev) / (t_e2e * 1e-3),
               "unit": UNIT, "ms_per_step": t_e2e,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    # ---- extras: the window's causal block merged in (sparse and dense),
    # and the naive estimator (every target head of every layer scored).
    extras = None
    if not args.no_extras:
        extras = run_extras(rep, wl, dev, stream, L, args, t_attn,
                            dense["us_per_layer"] if dense else None)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu:
        res = run_oracle_leg(args, args.cpu_reps, 1)
        cpu = {"value": res["value"], "unit": UNIT, "cores": res["cores"],
               "kind": "oracle", "sample": res["sample"],
               "wall_s": res["wall_s"]}

    kernels = {
        "score_target_us": t_score_t,
        "score_draft_us": t_score_d,
        "select_us": t_select,
        "sparse_attn_us_per_layer": t_attn,
        "score_target_gbs": rep.bytes_score_t() / (t_score_t * 1e-6) / 1e9,
        "score_draft_gbs": rep.bytes_score_d() / (t_score_d * 1e-6) / 1e9,
        "sparse_attn_gbs": achieved,
    }
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": W, "ms_per_step": t_ms,
        "ms_per_step_median": t_step_median,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic",
        "config": workload_config(wl, L),
        "roofline": {"bound": "hbm", "kernel": "verify_attn_kernel (sparse)",
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak,
                     "peak_kind": f"{peak_kind} hbm_gbs",
                     "algorithmic_bytes_per_launch": b_attn,
                     "traffic": committed_traffic()},
        "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": launches,
        "clocks": clock_info, "kernels": kernels, "dense": dense,
        "extras": extras,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    R.barrier(dev)
    R.shutdown()
    return 0


def run_profile_once(args):
    """One launch of every kernel of the library on the workload's shapes
    (one materialised target layer, so that a capture holds a few GB): target
    and draft scoring (TMA logits pass + reduce), the selection (clusters),
    sparse and dense attention of the layer, the sparse call of one sequence
    (positions split over CTAs: the combine kernel), the multi-layer launch
    over the layer twice, Quest page statistics and page scores with their
    page selection (the 256-thread select instance), and the cp.async
    logits pass (a paged cache with 48-position pages, four sequences)."""
    import torch
    from sparse_kv_verification_gb300 import build
    from sparse_kv_verification_gb300 import inputs as I
    from sparse_kv_verification_gb300 import native as N
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    build.build()
    N.load()
    dev = torch.device("cuda", 0)
    wl = I.WORKLOADS[args.config]
    if args.batch:
        wl = wl.replace(b=args.batch)
    rep = Replica(wl, dev, 1)
    inp = rep.inp
    sync = torch.cuda.synchronize
    ran = []

    def once(name, fn):
        fn()
        sync()
        ran.append(name)

    once("score target", rep.score_t)
    once("score draft", rep.score_d)
    once("select", rep.select)
    once("sparse attention", rep.attn[0])
    once("dense attention", rep.full[0])
    # One sequence: 8 units on 152 SMs, so the positions are split.
    q1 = inp.q[0][:1].contiguous()
    k1, v1 = inp.k[0][:1].contiguous(), inp.v[0][:1].contiguous()
    o1, l1 = torch.empty_like(q1), torch.empty(q1.shape[:3], device=dev)
    ws1 = N.workspace(N.dustin_sparse_verify_attn_workspace_size(
        1, wl.hq, wl.hkv, wl.d, wl.w, wl.k), dev)
    once("sparse attention, one sequence (split + combine)",
         lambda: N.dustin_sparse_verify_attn(q1, N.kv_desc(k1, v1), wl.hkv, wl.n,
                                             rep.idx[:1].contiguous(), wl.scale, o1, l1, ws1))
    kv0 = N.kv_desc(inp.k[0], inp.v[0])
    o2 = [torch.empty_like(inp.q[0]) for _ in range(2)]
    l2 = [torch.empty(inp.q[0].shape[:3], device=dev) for _ in range(2)]
    once("multi-layer sparse attention (the layer twice)",
         lambda: N.dustin_sparse_verify_attn_layers([inp.q[0], inp.q[0]], [kv0, kv0],
                                                    wl.hkv, wl.n, rep.idx, wl.scale, o2, l2))
    page = 16
    n_pages = (wl.n + page - 1) // page
    stats = torch.empty((wl.b, wl.hkv, n_pages, 2, wl.d), dtype=torch.bfloat16, device=dev)
    once("quest page statistics",
         lambda: N.dustin_quest_page_stats(kv0, wl.b, wl.hkv, wl.d, wl.n, page, stats=stats))
    q_row = inp.q[0][:, :, 0, :].contiguous()
    scores = torch.empty((wl.b, wl.hq, n_pages), device=dev)
    once("quest page scores",
         lambda: N.dustin_quest_page_scores(q_row, stats, wl.n, page, scores=scores))
    keep = max(1, wl.k // page)
    pidx = torch.empty((wl.b * wl.hq, keep), dtype=torch.int32, device=dev)
    once("quest page selection (short rows)",
         N.prepare_hybrid_topk(scores.view(wl.b * wl.hq, n_pages), None, keep, 0, 0, 1.0,
                               -1, N.DUSTIN_NORM_NONE, pidx))
    bp = min(4, wl.b)
    pool, _, table = I.to_paged(inp.k_t[0][:bp].contiguous(), None, 48, seed=7)
    q_p = inp.q_t[:1, :bp].contiguous()
    s_p = torch.empty((bp, wl.n), device=dev)
    ws_p = N.workspace(N.dustin_score_heads_workspace_size(bp, wl.n, 1, 1), dev)
    once("scoring, paged cache of 48-position pages (cp.async logits pass)",
         lambda: N.dustin_score_heads(q_p, [N.kv_desc(pool, None, table)], inp.kvh_t[:1],
                                      wl.scale, s_p, ws_p, wl.n))
    print(json.dumps({"profile_once": ran, "config": workload_config(wl, 1),
                      "target_pairs_share_kv_heads": len(set(inp.kvh_t)) < len(inp.kvh_t),
                      "device_status": N.dustin_device_status()}), flush=True)
    return 0


def main(argv=None):
    args = parse_args(argv)
    if args.oracle_worker:
        oracle_worker(args)
        return 0
    if args.profile_once:
        return run_profile_once(args)
    if args.impl == "reference":
        return run_reference(args)
    if args.sweep:
        return run_sweep(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
