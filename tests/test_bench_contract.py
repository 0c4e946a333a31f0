"""The benchmark's reference arm on the host (no GPU): the fp64 oracle timed on a
bounded sample, printed as one JSON line with the keys the benchmark line carries;
ranks other than 0 print nothing and succeed."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench(*extra, env=None):
    e = dict(os.environ)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", *extra],
                          cwd=ROOT, env=e, capture_output=True, text=True, timeout=300)


@pytest.mark.parametrize("workload", ["tiny_fp32", "linear_chunk64"])
def test_reference_arm_prints_one_complete_line(workload):
    r = _bench("--workload", workload, "--steps", "2", "--warmup", "3", "--cpu-budget", "0.5")
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference"
    assert line["unit"] == "tokens/s" and line["higher_is_better"] is True
    assert (line["steps"], line["warmup"], line["n_gpus"]) == (2, 3, 1)
    assert line["value"] > 0 and line["vs_baseline"] is None
    assert line["config"]["workload"] == workload
    # the per-step time is the whole workload at the sampled rate, and says so
    cfg = line["config"]
    assert line["ms_per_step"] == pytest.approx(cfg["B"] * cfg["T"] / line["value"] * 1e3, rel=1e-9)
    assert line["ms_per_step_kind"].startswith("extrapolated")
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "tokens/s",
                           "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_reference_arm_runs_on_rank_zero_only():
    r = _bench("--workload", "tiny_fp32", "--steps", "1", "--warmup", "3", "--cpu-budget", "0.1",
               env={"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
