"""The multi-rank host logic on CPU with two gloo ranks: each rank owns an
independent slice of heads (no collective on the data path), and the only
cross-rank step is the max over ranks of the timings."""
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
