"""The N > 1 path of bench.py on CPU: replicas only, so the only
cross-rank operations are the timing barrier and the maximum of the per-rank
times; world_size 2 over gloo, rendezvous on 127.0.0.1.  Also: under torchrun
the reference arm runs on rank 0 alone and the other ranks exit 0."""
import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = [3.25, 4.5][rank]
        slowest = bench.max_over_ranks(ms, world)
        rate = bench.whole_job_rate(world, 1000, 10, slowest / 1e3)
        q.put((rank, slowest, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_on_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, rate in got:
        assert slowest == 4.5                    # the slowest replica sets the time
        assert abs(rate - 2 * 1000 * 10 / 4.5e-3 / 1e6) < 1e-9   # both replicas' cells


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(7.0, 1) == 7.0
    assert bench.whole_job_rate(1, 100, 3, 0.5) == 100 * 3 / 0.5 / 1e6


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1",
               MASTER_ADDR="127.0.0.1", MASTER_PORT=str(free_port()))
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "dam128", "--steps", "2", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=300, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_reference_arm_line_on_rank_zero():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--workload", "dam128", "--steps", "2", "--warmup", "3"],
                       env=env, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
