"""bench.py on the CPU: argument checks, the workload description both arms
print, and a short run of the reference arm (the oracle on the host cores)."""
import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _run(args, env=None):
    e = dict(os.environ)
    for k in ("RANK", "LOCAL_RANK", "WORLD_SIZE"):
        e.pop(k, None)
    e.update(env or {})
    return subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                          capture_output=True, text=True, env=e, timeout=600)


def test_gpus_must_match_world_size():
    r = _run(["--gpus", "2"])
    assert r.returncode != 0
    assert "WORLD_SIZE is 1" in r.stderr


def test_warmup_below_three_rejected():
    r = _run(["--warmup", "2"])
    assert r.returncode != 0 and "--warmup" in r.stderr


def test_unknown_also_workload_rejected():
    r = _run(["--also", "mla_decode,no_such_workload"])
    assert r.returncode != 0 and "no_such_workload" in r.stderr


@pytest.mark.parametrize("name", ["mla_decode", "mla_prefill_fp8", "knorm64"])
def test_both_arms_describe_the_workload_alike(name):
    w = bench.WORKLOADS[name][0](bench.DEFAULT_SEED)
    a = bench.config_of(name, w, 1)
    b = bench.config_of(name, w, 1)
    assert a == b
    assert set(a) == {"workload", "tokens_per_gpu", "l2", "io", "parallelism"}
    assert a["tokens_per_gpu"] == w.T
    big = bench.algorithmic_bytes(w, name) >= 2 * bench.L2_BYTES
    assert ("larger than L2" in a["l2"]) == big


def test_default_line_is_the_fp8_prefill():
    assert bench.DEFAULT_WORKLOAD == "mla_prefill_fp8"
    assert "mla_decode" in bench.DEFAULT_ALSO
    assert bench.metric_of("mla_prefill_fp8", "tokens/s") == bench.METRIC


def test_reference_arm_prints_one_line():
    r = _run(["--impl", "reference", "--workload", "mla_decode", "--steps", "1", "--warmup", "3",
              "--ref-step-s", "0.05"])
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference"
    assert line["metric"] == bench.METRIC and line["unit"] == "tokens/s"
    assert line["value"] > 0 and line["higher_is_better"] is True
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0
    w = bench.WORKLOADS["mla_decode"][0](bench.DEFAULT_SEED)
    assert line["config"] == bench.config_of("mla_decode", w, 1)
