"""Multi-rank host logic of bench.py on CPU: two gloo ranks, each running its
own replica (independent problems, no collective on the data path), then the
max-over-ranks time and the whole-job rate.  Also: the reference arm prints
from rank 0 only."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, out):
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import synthetic
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=ws)
    try:
        # each rank solves its own seeded problem with the oracle (a stand-in for its GPU replica)
        inp = synthetic.taylor_inputs(1, 2, 40, dtype=torch.float32, seed=7 + bench.rank_seed_offset(rank))
        y = oracle.taylor(*(synthetic.to_oracle(inp[n]) for n in ("q", "k", "v")), nthreads=1)["y"]
        ms = 10.0 + 5.0 * rank
        mx = bench.max_over_ranks(ms, ws)
        rate = bench.whole_job_rate(1000.0, ws, mx * 1e-3)
        bench.barrier(ws)
        out.put((rank, mx, rate, float(np.abs(y).sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, mx0, rate0, y0), (r1, mx1, rate1, y1) = res
    assert (r0, r1) == (0, 1)
    assert mx0 == mx1 == 15.0                      # the slowest rank's time on both ranks
    assert rate0 == rate1 == 2 * 1000.0 / 15e-3    # units of all ranks / slowest time
    assert y0 != y1                                 # independent replicas: different seeded inputs


def test_reference_arm_prints_on_rank_zero_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip() == ""
    env.update(RANK="0", LOCAL_RANK="0")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "tokens/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["e2e"]["h2d_bytes_per_step"] == 0
