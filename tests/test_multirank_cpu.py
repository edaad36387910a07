"""The multi-rank host logic on CPU with two gloo ranks: each rank owns an
independent slice of heads (no collective on the data path), and the only
cross-rank step is the max over ranks of the timings.  The second test runs
bench.py's own multi-rank path (rank environment, barriers around the timed
region, max over ranks, whole-job value) with a CPU stand-in for the kernel
calls."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import workloads as wl
    w = wl.Workload("t", "fwd", 2, 3, 40, 8, "bf16", True)
    # rank-local slice of the global job: its own seeded batch
    mine = bench.rank_workload(w, rank)
    inp = wl.make_inputs(mine)
    O, L = oracle.attention(*(inp[n].to(torch.float64).numpy() for n in ("q", "k", "v")),
                            True, w.scale)
    np.save(os.path.join(out_dir, f"o{rank}.npy"), O)
    # the only collective: max over ranks of per-rank timings
    got = bench.max_over_ranks([1.0 + rank, 10.0 - rank])
    np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array(got))
    # head partition helper covers every head exactly once
    parts = [list(wl.head_range(r, world, 7)) for r in range(world)]
    assert sorted(sum(parts, [])) == list(range(7))
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world, port = 2, _free_port()
    mp.start_processes(_worker, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    import oracle
    import workloads as wl
    import bench
    w = wl.Workload("t", "fwd", 2, 3, 40, 8, "bf16", True)
    for r in range(world):
        np.testing.assert_array_equal(np.load(tmp_path / f"t{r}.npy"), [2.0, 10.0])
        inp = wl.make_inputs(bench.rank_workload(w, r))
        O, _ = oracle.attention(*(inp[n].to(torch.float64).numpy() for n in ("q", "k", "v")),
                                True, w.scale)
        np.testing.assert_array_equal(np.load(tmp_path / f"o{r}.npy"), O)
    # different ranks really hold different slices of the global batch
    assert not np.array_equal(np.load(tmp_path / "o0.npy"), np.load(tmp_path / "o1.npy"))


class _CpuTimer:
    """Host stand-in for bench.CudaTimer (wall clock, nothing to sync)."""

    def sync(self):
        pass

    def mark(self):
        import time
        return time.perf_counter()

    def elapsed_ms(self, a, b):
        return (b - a) * 1e3


def _host_path_worker(rank, world, port, out_dir):
    """One rank of bench.py's multi-rank host path with a CPU stand-in for the
    kernel calls: the rank environment check, the barriers around the timed
    region, the max over ranks of the per-step times and the whole-job value."""
    import json
    import sys
    import time
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), WORLD_SIZE=str(world),
                      RANK=str(rank), LOCAL_RANK=str(rank))
    import bench
    got_rank, got_world, local = bench.rank_env(world)
    assert (got_rank, got_world, local) == (rank, world, rank)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    steps = 4
    calls = []

    def step():  # rank 1 is deliberately slower: the job time is its time
        calls.append(1)
        time.sleep(0.01 * (1 + 2 * rank))

    ms_total = bench.timed_region(steps, step, world, _CpuTimer())
    ms_step, e2e_ms = bench.job_times(ms_total / steps, 1.0 + rank, world)
    value = bench.job_value(1e12, ms_step, world)
    with open(os.path.join(out_dir, f"r{rank}.json"), "w") as f:
        json.dump({"calls": len(calls), "mine": ms_total / steps, "ms_step": ms_step,
                   "e2e_ms": e2e_ms, "value": value}, f)
    dist.destroy_process_group()


def test_bench_host_path_two_gloo_ranks(tmp_path):
    import json
    world, port = 2, _free_port()
    mp.start_processes(_host_path_worker, args=(world, port, str(tmp_path)), nprocs=world,
                       start_method="spawn")
    recs = [json.load(open(tmp_path / f"r{r}.json")) for r in range(world)]
    slowest = max(r["mine"] for r in recs)
    for r in recs:
        assert r["calls"] == 4                      # exactly `steps` timed calls
        assert r["ms_step"] == slowest              # both ranks report the slowest rank
        assert r["e2e_ms"] == 2.0                   # max over ranks of (1 + rank)
        # whole job: world x the per-rank FLOPs in the slowest rank's time
        np.testing.assert_allclose(r["value"], world * 1e12 / (slowest * 1e-3) / 1e12)
    assert recs[1]["mine"] > recs[0]["mine"]


def test_rank_env_rejects_a_mismatched_world(monkeypatch):
    import sys
    import pytest
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    with pytest.raises(SystemExit):
        bench.rank_env(4)
    monkeypatch.delenv("WORLD_SIZE")
    assert bench.rank_env(1) == (0, 1, 0)
    with pytest.raises(SystemExit):
        bench.rank_env(2)
