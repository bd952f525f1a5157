"""The benchmark's multi-rank host logic on CPU: replicas over gloo at world size 2
(rendezvous on 127.0.0.1, barrier, max over ranks of the step time, the whole-job
throughput, the reference arm printing on rank 0 only).  The path has no data exchange
between ranks (replicas only), so no collective is on the data path."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    r, w, _ = bench.dist_setup(None)
    bench.barrier(w)
    own = 1.0 + rank                       # this rank's timed seconds
    slowest = bench.allreduce_max(own, w)  # what rank 0 reports
    value = bench.step_throughput(32, 10, w, slowest, 20)
    q.put((r, w, own, slowest, value))
    bench.barrier(w)
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank_and_the_whole_job():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[:2] for g in got] == [(0, 2), (1, 2)]
    for _, _, own, slowest, value in got:
        assert slowest == 2.0                       # max over ranks, on every rank
        assert value == 32 * 10 * 2 * 20 / 2.0      # both ranks' queries over the slowest time


def test_reference_arm_prints_on_rank_zero_only():
    lines = {}
    for rank in (0, 1):
        env = dict(os.environ, RANK=str(rank), WORLD_SIZE="2", LOCAL_RANK=str(rank),
                   MASTER_ADDR="127.0.0.1")
        r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                            "--workload", "tiny_full_1q_ctx4k", "--steps", "1", "--warmup", "0"],
                           cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
        assert r.returncode == 0, r.stderr[-2000:]
        lines[rank] = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert lines[1] == []
    assert len(lines[0]) == 1
    d = json.loads(lines[0][0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1


def test_step_quantiles_are_nearest_rank():
    sys.path.insert(0, ROOT)
    import bench
    q = bench.step_quantiles(list(range(20, 0, -1)))   # 1..20 ms in any order
    assert q == {"p10": 2.0, "p50": 10.0, "p90": 18.0}
    assert bench.step_quantiles([0.25]) == {"p10": 0.25, "p50": 0.25, "p90": 0.25}
    assert bench.step_quantiles([]) == {}
