"""The benchmark's JSON line, checked on CPU through its reference arm (the
oracle, timed): one line with the keys the measurement contract names."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(*args):
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                         cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, out.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--config", "tiny", "--steps", "2", "--warmup", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 2 and d["warmup"] == 1
    assert d["value"] > 0 and d["ms_per_step"] > 0
    assert d["higher_is_better"] is True and d["scaling"] == "weak"
    assert d["data"] == "synthetic" and "workload" in d["config"]
    cpu = d["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["sample"]
    assert cpu["value"] == d["value"] and cpu["unit"] == d["unit"]
    e2e = d["e2e"]
    assert e2e["value"] == d["value"] and e2e["unit"] == d["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    # the tiny workload fits in L2 and says so
    assert "within L2" in d["config"]["l2"]


def test_e2e_chunk_bounds():
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    assert bench.e2e_chunk_bounds(80) == [0, 8, 16, 24, 32, 40, 48, 56, 64, 72, 76, 78, 79, 80]
    for L in range(1, 130):
        b = bench.e2e_chunk_bounds(L)
        sizes = [y - x for x, y in zip(b, b[1:])]
        assert b[0] == 0 and b[-1] == L and all(s >= 1 for s in sizes)
        assert max(sizes) <= 8 and sizes[-1] == 1


def test_committed_sparse_profile_fields():
    """The ncu record the bench reads its traffic figure from names the
    kernel source it was taken on and a per-launch DRAM traffic close to
    the algorithmic bytes."""
    with open(os.path.join(ROOT, "profiles", "sparse_verify_attn_72b.json")) as f:
        rec = json.load(f)
    assert len(rec["source_sha"]) == 16
    traffic = float(rec["dram_bytes_per_launch"])
    algorithmic = float(rec["algorithmic_bytes_per_launch"])
    assert algorithmic <= traffic <= 1.1 * algorithmic
