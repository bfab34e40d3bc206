"""Multi-rank host logic of the benchmark on CPU: two gloo processes stand in
for two GPUs (one process per GPU, weak scaling).  Checks that every rank
times its own seeded batch of the same shapes, that the step time reported is
the slowest rank's (a MAX all-reduce), that the whole-job rate counts every
rank's tokens, and that the reference arm runs on rank 0 only."""
import importlib.util
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_mod", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    bench = load_bench()
    from long_context_sparse_moba_gb300 import workloads
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w_env, r_env, l_env = bench.dist_env()
        base = workloads.custom((512,), H=2, D=64, block_size=128, topk=3, seed=7)
        wr = bench.rank_workload(base, r_env)
        inp = workloads.make_inputs(wr, device="cpu")
        # each rank's own step time; the reported one is the slowest
        my_ms = 1.0 + 0.5 * r_env
        slowest = bench.max_over_ranks(my_ms, w_env)
        dist.barrier()
        out[rank] = (w_env, r_env, l_env, wr.seed, float(inp.q.float().sum()), slowest,
                     bench.whole_job_rate(wr.total, w_env, slowest))
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling_and_max_time():
    world = 2
    manager = mp.get_context("spawn").Manager()  # no fork of a threaded process
    out = manager.dict()
    mp.spawn(_worker, args=(world, free_port(), out), nprocs=world, join=True)
    r0, r1 = out[0], out[1]
    assert (r0[0], r0[1], r0[2]) == (2, 0, 0) and (r1[0], r1[1], r1[2]) == (2, 1, 1)
    assert r0[3] != r1[3]                 # every rank draws its own batch
    assert r0[4] != r1[4]
    assert r0[5] == r1[5] == 1.5          # the slowest rank's time everywhere
    assert r0[6] == pytest.approx(512 * 2 / 1.5e-3)


def test_one_rank_needs_no_process_group():
    bench = load_bench()
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_rate(32768, 1, 2.0) == pytest.approx(32768 / 2e-3)


def test_reference_arm_prints_on_rank_0_only():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--steps", "1", "--warmup", "0"],
                       env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
