"""bench.py's output contract, checked on the arm that needs no GPU (the CPU
oracle timed as the reference arm): one JSON line with the required keys,
e2e with zero copy bytes, cpu_baseline of kind "oracle"; ranks other than 0
print nothing and exit 0.  Plus the launch count the GPU arm reports."""

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(args, env_extra=None, timeout=600):
    env = dict(os.environ)
    env.update(env_extra or {})
    p = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py")] + args, cwd=ROOT,
                       env=env, capture_output=True, text=True, timeout=timeout)
    assert p.returncode == 0, p.stderr[-2000:]
    return [l for l in p.stdout.splitlines() if l.strip()]


@pytest.mark.parametrize("config,tokens", [("tiny", 32), ("moe30b_logits", 32)])
def test_reference_arm_json_line(config, tokens):
    lines = _run(["--impl", "reference", "--config", config, "--steps", "2", "--warmup", "1",
                  "--cpu-tokens", str(tokens)])
    assert len(lines) == 1
    r = json.loads(lines[0])
    for k in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
              "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
              "cpu_baseline", "e2e"):
        assert k in r, k
    assert r["impl"] == "reference" and r["steps"] == 2 and r["warmup"] == 1
    assert r["value"] > 0 and r["unit"] == "tokens/s" and r["higher_is_better"] is True
    assert r["config"]["workload"] == config and r["config"]["tokens_per_step"] == tokens
    # value and ms_per_step describe the same run
    assert r["value"] == pytest.approx(tokens / (r["ms_per_step"] / 1e3), rel=1e-9)
    cb = r["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == r["value"] and cb["cores"] >= 1
    assert cb["sample"]
    e2e = r["e2e"]
    assert e2e["value"] == r["value"] and e2e["unit"] == r["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0


def test_reference_arm_other_ranks_are_silent():
    lines = _run(["--impl", "reference", "--config", "tiny", "--steps", "1", "--warmup", "0"],
                 env_extra={"RANK": "1", "WORLD_SIZE": "2"})
    assert lines == []


def test_launch_count_formula():
    sys.path.insert(0, ROOT)
    import bench
    # advantage + response factors + two loss kernels, five launches per
    # 38,912-row chunk
    assert bench.launches_per_step(1, 151936) == 4 + 5
    assert bench.launches_per_step(38912, 151936) == 4 + 5
    assert bench.launches_per_step(38913, 151936) == 4 + 10
    assert bench.launches_per_step(1_083_112, 151936) == 144
