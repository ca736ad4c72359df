"""The multi-GPU path's host logic on CPU: two gloo ranks run the benchmark's cross-rank reduction.

Rows are independent, so `bench.py --gpus N` runs one replica per GPU with no data-path collective
(weak scaling). Each rank draws its own seeded batch; the job's step time is the slowest rank's,
and the job's value counts every rank's verified positions. Ragged draft lengths give the ranks
different counts.
"""
import importlib.util
import multiprocessing as mp
import os
import socket
import sys
from argparse import Namespace
from pathlib import Path

import numpy as np
import pytest

torch = pytest.importorskip("torch")

ROOT = Path(__file__).resolve().parent.parent


def load_bench():
    spec = importlib.util.spec_from_file_location("bench_under_test", ROOT / "bench.py")
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, ms, units, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, str(ROOT))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench = load_bench()
        got = bench.job_totals(ms[rank], units[rank], "cpu")
        # the ranks' own view of the environment the benchmark reads
        q.put((rank, got, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def run_ranks(ms, units):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = free_port()
    world = len(ms)
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, ms, units, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = {}
    for _ in procs:
        rank, got, env = q.get(timeout=120)
        out[rank] = (got, env)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    return out


def test_job_totals_two_gloo_ranks():
    """Slowest rank's time, sum of the ranks' units, the same on every rank."""
    ms, units = [1.25, 1.5], [5541, 5602]
    out = run_ranks(ms, units)
    for rank in (0, 1):
        (t, n), env = out[rank]
        assert t == pytest.approx(1.5)
        assert n == 5541 + 5602
        assert env == (2, rank, rank)


def test_job_totals_single_process_passthrough():
    bench = load_bench()
    assert bench.job_totals(2.5, 77) == (2.5, 77.0)


def test_rank_batches_are_independent_shards():
    """Each rank's seed draws a different batch; ragged lengths give different position counts, and
    the job total is their sum (what job_totals adds up)."""
    bench = load_bench()
    from workloads import get_config, make_workload
    import dataclasses
    cfg = dataclasses.replace(get_config(5), B=64, V=256)
    seeds = [bench.rank_seed(cfg.seed, r) for r in range(2)]
    assert seeds[0] != seeds[1]
    w = [make_workload(cfg, seed=s, backend="numpy") for s in seeds]
    assert not np.array_equal(w[0].draft_len, w[1].draft_len)
    assert not np.array_equal(w[0].target_logits, w[1].target_logits)
    pos = [x.positions() for x in w]
    assert pos[0] != pos[1]                 # so world x (rank 0's count) would misstate the job
    assert sum(pos) != 2 * pos[0]


def test_reference_arm_runs_on_rank_zero_only(capsys, monkeypatch):
    """Under torchrun the reference arm is timed by rank 0 alone; the other ranks exit 0 without
    work or output."""
    bench = load_bench()
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = Namespace(tree=False, workload=1, onehot=False, filter=False, steps=1, warmup=0)
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
