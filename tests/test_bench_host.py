"""Host-side logic of bench.py on CPU: the traffic figures' source guard, the
reference arm and the CPU baseline (both the oracle on the host cores, on the
same bounded sample), and the single-GPU refusal of --gpus N > 1."""
import json
import os
import subprocess
import sys
import time

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_profiled_traffic_is_dropped_when_the_kernel_source_changes(monkeypatch):
    sys.path.insert(0, ROOT)
    import bench
    for name, e in bench.NCU_TRAFFIC.items():
        assert os.path.exists(os.path.join(ROOT, e["profile"])), name
        got = bench.profiled_traffic(name)
        assert got in (None, e["bytes"])
        assert (got is not None) == (bench.source_digest(e["files"]) == e["digest"])
    e = dict(bench.NCU_TRAFFIC["glance_tree_attention"], digest="0" * 16)
    monkeypatch.setitem(bench.NCU_TRAFFIC, "glance_tree_attention", e)
    assert bench.profiled_traffic("glance_tree_attention") is None
    assert bench.profiled_traffic("no_such_kernel") is None


def test_reference_arm_prints_one_bounded_line():
    """The reference arm (the oracle on the host cores) runs on the small
    workload without a GPU and prints the contract's line."""
    t0 = time.perf_counter()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "small", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "rounds/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert time.perf_counter() - t0 < 120
    assert line["n_gpus"] == 1 and 0 < line["rounds_per_step"] < 1
    # value = the round fraction a step covers / the step's wall time
    assert line["value"] == pytest.approx(line["rounds_per_step"] / (line["ms_per_step"] / 1e3), rel=0.05)


def test_cpu_baseline_uses_the_reference_arms_sample():
    sys.path.insert(0, ROOT)
    import bench
    cb = bench.cpu_baseline(bench.SMALL, seconds=0.0)
    assert cb["kind"] == "oracle" and cb["steps_timed"] >= 3 and cb["cores"] >= 1
    assert cb["sample"] == bench.oracle_sample_text(bench.SMALL)
    assert set(cb["stage_seconds_full_round"]) == {"tree", "attention", "lmhead", "commit"}


def test_more_than_one_gpu_is_refused_with_a_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--gpus", "2", "--steps", "1"],
                         capture_output=True, text=True, timeout=120, cwd=ROOT,
                         env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    assert line["n_gpus"] == 2 and "unavailable" in line
