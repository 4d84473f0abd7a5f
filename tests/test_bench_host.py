"""bench.py's multi-rank host logic on CPU: two gloo ranks (spawned processes)
take the slowest rank's time and report the whole-job aggregate; the
reference arm prints only on rank 0.  No GPU is touched."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist = bench.init_dist(world, "gloo")
    seconds = [0.5, 2.0][rank]          # rank 1 is the slow one
    t_max = bench.reduce_max(dist, seconds)
    bench.barrier(dist)
    out.put((rank, t_max, bench.aggregate(1000.0, world, t_max)))
    dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, t_max, agg in res:
        assert t_max == 2.0
        assert agg == pytest.approx(1000.0 * 2 / 2.0)   # both ranks' units over the slowest time


@pytest.mark.parametrize("rank,prints", [(0, True), (1, False)])
def test_reference_arm_prints_on_rank_zero_only(rank, prints):
    env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload", "tiny",
                        "--steps", "2", "--warmup", "1", "--cpu-seconds", "0.2"],
                       env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.strip()]
    if not prints:
        assert lines == []
        return
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["unit"] == "GB/s" and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_times_the_exact_codes_oracle_for_the_exact_workload():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--workload",
                        "gate_up_exact", "--steps", "1", "--warmup", "1", "--cpu-seconds", "0.2"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr
    d = json.loads([ln for ln in r.stdout.splitlines() if ln.strip()][0])
    assert d["impl"] == "reference" and d["value"] > 0 and d["config"]["workload"] == "gate_up_exact"
    assert "exact-codes oracle" in d["cpu_baseline"]["sample"] and d["cpu_baseline"]["cores"] == 1
