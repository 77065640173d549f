"""bench.py's multi-rank host logic on the CPU: world-size-2 gloo ranks.

The drafter does not shard (one replica a GPU), so the only multi-rank steps
are the benchmark's: a barrier around the timed region, the slowest rank's
time taken as the job's, and the whole job's throughput from it.  The same
helpers run under NCCL on GPUs.
"""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        sys.path.insert(0, ROOT)
        import bench
        local = 0.25 * (rank + 1)  # rank 1 is the slow one
        t = bench.max_over_ranks(local, dist, "cpu")
        dist.barrier()
        q.put((rank, local, t, bench.job_throughput(world, 15, t)))
    finally:
        dist.destroy_process_group()


def test_two_ranks_report_the_slowest_time_and_the_whole_job():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    try:
        res = sorted(q.get(timeout=120) for _ in range(2))
    finally:
        for p in ps:
            p.join(timeout=60)
    assert all(p.exitcode == 0 for p in ps)
    assert [r[2] for r in res] == [0.5, 0.5]  # every rank sees the slowest rank's time
    assert res[0][3] == 2 * 15 / 0.5  # the units of both ranks over that time


def test_one_rank_without_a_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(0.125) == 0.125
    assert bench.job_throughput(1, 15, 0.125) == 120.0


def test_reference_arm_under_two_ranks_prints_one_line():
    """Launched as the multi-GPU runs are (torchrun, two ranks): rank 0 alone
    times the oracle and prints the line; rank 1 exits 0 without work."""
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), "bench.py", "--impl", "reference",
           "--gpus", "2", "--steps", "1", "--warmup", "0", "--workload", "tiny_f32"]
    out = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    lines = [l for l in out.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
