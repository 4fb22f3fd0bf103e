"""Host-side logic of bench.py on CPU: the N>1 replica path's max-over-ranks
timing and whole-job aggregation, run as two gloo ranks."""
import os
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _rank(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 100.0 + 50.0 * rank          # rank 1 is slower
    m = bench.max_over_ranks(ms, dist, "cpu")
    q.put((rank, m, bench.job_value(world, 10, m)))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29500 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, m, v in out:
        assert m == 150.0
        assert v == pytest.approx(2 * 10 / 0.150)


def test_single_process_value():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(12.5, None, "cpu") == 12.5
    assert bench.job_value(1, 50, 1000.0) == pytest.approx(50.0)


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
    import json
    import subprocess
    import sys
    import time
    t0 = time.perf_counter()
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                          "small", "--steps", "3", "--warmup", "3"], capture_output=True, text=True, timeout=300,
                         cwd=ROOT, env=dict(os.environ, CUDA_VISIBLE_DEVICES=""))
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["value"] > 0 and line["unit"] == "rounds/s"
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
    assert time.perf_counter() - t0 < 120
