"""The reference arm of bench.py (the oracle timed on the host cores) keeps
the JSON-line contract: one line with the metric, unit and direction of the
GPU arm, impl = reference, a cpu_baseline that describes the run, and an
e2e object with no device copies.  Runs on the CPU with a tiny row sample."""
import json
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_reference_arm_prints_one_contract_line():
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "h16-s8192", "--steps", "1", "--warmup", "1", "--ref-rows", "4"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference"
    assert d["n_gpus"] == 1 and d["steps"] == 1 and d["warmup"] == 1
    assert d["higher_is_better"] is True and d["unit"] == "TFLOP/s" and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1
    assert cb["sample"] and cb["affinity"]
    assert d["e2e"] == {"value": d["value"], "unit": d["unit"], "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}
    assert d["config"]["workload"].startswith("h16-s8192")


def test_reference_arm_other_ranks_exit_without_output():
    env = dict(os.environ, RANK="1", LOCAL_RANK="1", WORLD_SIZE="2")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "1", "--ref-rows", "4"],
                       capture_output=True, text=True, timeout=600, cwd=ROOT, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""


def test_oracle_sample_rows():
    # the oracle legs' row samples: the video-DiT key length's work in rows,
    # never more rows than exist, within as few heads from the first on as
    # hold them (a head's rows share its keys)
    import importlib.util
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(bench)
    for name, w in bench.WORKLOADS.items():
        S, total, Sk = w["S"], w["B"] * w["H"] * w["S"], bench.keys(w)
        for n_rows in (1, 96, 1024, 12288):
            rows = bench.sample_rows(w, n_rows)
            want = min(total, max(1, round(n_rows * 75600 / Sk)))
            assert len(rows) == want, (name, n_rows, len(rows), want)
            assert rows[0] == 0 and rows[-1] < total
            assert all(rows[1:] > rows[:-1])
            heads_needed = -(-want // S)
            assert rows[-1] < heads_needed * S, (name, n_rows)
    assert bench.sample_rows(bench.WORKLOADS["video-dit"], 12288)[-1] < 75600
