"""Multi-rank host logic of the replica path, on CPU with the gloo backend.

The path runs as independent replicas (one layer batch per rank, no data
collective).  These tests run two ranks as processes on 127.0.0.1 and check
the job-wide totals (retained pairs summed, time of the slowest rank), that
replicas draw distinct batches with rank 0 drawing the single-GPU one, that
per-rank oracle results add up to the serial computation, and that the
reference arm leaves every rank but 0 idle.
"""

import os
import socket
import subprocess
import sys
from fractions import Fraction

import numpy as np
import pytest

import oracle as O
from backward_token_expert_gb300.replicas import job_throughput, job_totals, replica_seed
from workloads import generate, get_workload

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TINY = "tiny_T256_E8_k2_h64_I32"


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, task, q):
    import torch.distributed as dist

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        if task == "totals":
            out = (job_totals(100 + rank, 1.0 + 0.5 * rank),
                   job_throughput(10 + rank, 3, 2.0 - rank * 0.25))
        elif task == "oracle":
            w = get_workload(TINY, seed=replica_seed(rank))
            inp = generate(w)
            st = O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)
            out = (int(st["retained"]), job_totals(int(st["retained"]), 1.0)[0])
        else:
            raise ValueError(task)
        q.put((rank, out))
    finally:
        dist.destroy_process_group()


def _run_ranks(task, world=2):
    import multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, task, q)) for r in range(world)]
    for p in procs:
        p.start()
    results = {}
    for _ in range(world):
        rank, out = q.get(timeout=120)
        results[rank] = out
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return results


def test_job_totals_sum_pairs_and_take_slowest_rank():
    res = _run_ranks("totals")
    for rank in (0, 1):
        (pairs, slowest), thr = res[rank]
        assert pairs == 100 + 101
        assert slowest == 1.5
        # (10 * 3 + 11 * 3) pairs over the slowest rank's 2.0 s
        assert thr == pytest.approx((30 + 33) / 2.0)


def test_per_rank_oracle_retained_adds_up_to_the_serial_sum():
    res = _run_ranks("oracle")
    serial = 0
    for rank in (0, 1):
        w = get_workload(TINY, seed=replica_seed(rank))
        inp = generate(w)
        serial += int(O.route_stats(inp.logits, inp.expert_idx, w.E, w.cf, w.rho)["retained"])
    assert res[0][0] + res[1][0] == serial
    assert res[0][1] == res[1][1] == serial


def test_single_process_totals_are_identity():
    assert job_totals(7, 0.25) == (7, 0.25)
    assert job_throughput(5, 4, 2.0) == 10.0
    with pytest.raises(ValueError):
        job_throughput(5, 0, 1.0)


def test_replicas_draw_distinct_batches_and_rank0_is_the_default():
    assert replica_seed(0) == 0 and replica_seed(3) == 3
    base = generate(get_workload(TINY))
    r0 = generate(get_workload(TINY, seed=replica_seed(0)))
    r1 = generate(get_workload(TINY, seed=replica_seed(1)))
    assert np.array_equal(base.logits, r0.logits) and np.array_equal(base.g, r0.g)
    assert not np.array_equal(r0.logits, r1.logits)
    assert not np.array_equal(r0.g, r1.g)
    assert r1.workload.rho == Fraction(3, 4)


def test_reference_arm_leaves_other_ranks_idle():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                          "--warmup", "3"], env=env, capture_output=True, text=True, timeout=120)
    assert out.returncode == 0
    assert out.stdout.strip() == ""
