"""The bench's multi-rank host logic on CPU with world_size-2 gloo groups: the timed values
are reduced to the slowest rank's, the whole-job rate counts every rank's units over that time,
and the reference arm runs on rank 0 alone (other ranks exit at once, printing nothing)."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [1.0 + rank, 5.0 - rank, 2.5]             # rank 1 is slower on the first value only
    out = bench.ranks_max(times, "cpu", world)
    q.put((rank, out, bench.job_rate(world, 1e9, out[0])))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_report_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, out, rate in results:
        assert out == [2.0, 5.0, 2.5]                  # the same maxima on every rank
        assert rate == 2 * 1e9 / 2e-3                  # both ranks' units over the slowest time


def test_single_rank_needs_no_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.ranks_max([3.0, 1.0], "cpu", 1) == [3.0, 1.0]
    assert bench.job_rate(1, 5e8, 0.5) == 1e12


def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    for extra in ([], ["--workload", "v3_prefill_b2_s4096"]):
        r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "0"] + extra,
                           cwd=ROOT, env=env, capture_output=True, timeout=300)
        assert r.returncode == 0 and r.stdout.strip() == b""
