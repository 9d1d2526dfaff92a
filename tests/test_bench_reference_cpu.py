"""The benchmark's reference arm (the fp64 CPU oracle on a bounded sample of the 50k x 50k,
d = 512 workload) runs without a GPU: its one JSON line carries the fields the benchmark
contract asks of that arm, and ranks other than 0 print nothing and exit 0."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(env_extra):
    env = dict(os.environ, **env_extra)
    return subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1",
                           "--warmup", "3"], cwd=ROOT, env=env, capture_output=True, text=True,
                          timeout=300)


def test_reference_arm_prints_one_contract_line():
    t0 = time.perf_counter()
    r = _run({"RANK": "0", "WORLD_SIZE": "1"})
    wall = time.perf_counter() - t0
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference"
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config"):
        assert key in line, key
    assert line["value"] > 0 and line["higher_is_better"] is True
    cpu = line["cpu_baseline"]
    assert cpu["kind"] == "oracle" and cpu["cores"] >= 1 and cpu["value"] == line["value"]
    assert "rows" in cpu["sample"]
    # The line says what it executed: each timed step is one bounded row sample, so the
    # steps' time fits inside the run; the full-problem figure is marked extrapolated.
    assert line["extrapolated"] is True and line["sampled_rows_per_step"] >= 1
    assert line["ms_per_step"] * line["steps"] / 1e3 < wall
    assert line["extrapolated_ms_per_full_step"] > line["ms_per_step"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_exit_quietly():
    r = _run({"RANK": "1", "WORLD_SIZE": "2"})
    assert r.returncode == 0, r.stderr[-2000:]
    assert not [ln for ln in r.stdout.splitlines() if ln.startswith("{")]


if __name__ == "__main__":
    sys.exit(pytest.main([__file__, "-q"]))
