"""The N > 1 path on the CPU (gloo, world size 2): every rank times its own
layer, the job's time is the slowest rank's (a MAX all-reduce after a
barrier), throughput is every rank's FLOP over that time, and rank 0 alone
prints; the reference arm runs on rank 0 only."""

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


def _rank_main(rank, world, port, out):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        elapsed = 1.0 + 0.5 * rank  # the last rank is the slowest
        t_max = bench.max_over_ranks(elapsed, world, "cpu")
        out.put((rank, t_max, bench.whole_job_tflops(world, 1e12, 3, t_max)))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_slowest_rank_sets_the_job_time_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    # both ranks see 1.5 s; 2 ranks x 1e12 FLOP x 3 steps / 1.5 s = 4 TFLOP/s
    assert got == [(0, 1.5, 4.0), (1, 1.5, 4.0)]


def test_reference_arm_runs_on_rank_zero_only():
    base = [sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1", "--warmup", "0"]
    env = dict(os.environ, WORLD_SIZE="2", MASTER_ADDR="127.0.0.1")
    r1 = subprocess.run(base, env=dict(env, RANK="1", LOCAL_RANK="1"), capture_output=True, text=True, timeout=300)
    assert r1.returncode == 0 and r1.stdout.strip() == ""
    r0 = subprocess.run(base, env=dict(env, RANK="0", LOCAL_RANK="0"), capture_output=True, text=True, timeout=300)
    assert r0.returncode == 0, r0.stderr
    line = json.loads(r0.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["value"] > 0
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["cpu_baseline"]["kind"] == "oracle"
