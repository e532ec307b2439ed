"""The N > 1 host logic of bench.py on CPU with world_size-2 gloo ranks:
rows of one seeded global batch are split between ranks with no overlap or
gap, and the job throughput is the bytes of all ranks over the slowest rank's
time (max all-reduce)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import sys

    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from residual_add_rmsnorm_vec_gb300 import synth

    T, H = 96, 128
    rows = bench.rank_rows(rank, world, T)
    wl_global = synth.prefill_workload(T * world, H)
    mine = synth.make_inputs(wl_global, rows=rows)
    np.save(os.path.join(out_dir, f"x{rank}.npy"), mine["x"].float().numpy())
    # rank r pretends its timed region took (r + 1) * 10 ms for 1e9 bytes
    max_ms, total, gbs = bench.aggregate(dist, (rank + 1) * 10.0, 1e9, torch.device("cpu"))
    np.save(os.path.join(out_dir, f"agg{rank}.npy"), np.array([max_ms, total, gbs]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_rows_and_aggregate(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       start_method="spawn", join=True)
    from residual_add_rmsnorm_vec_gb300 import synth

    full = synth.make_inputs(synth.prefill_workload(96 * world, 128))["x"].float().numpy()
    parts = [np.load(tmp_path / f"x{r}.npy") for r in range(world)]
    assert np.array_equal(np.concatenate(parts), full)
    for r in range(world):
        max_ms, total, gbs = np.load(tmp_path / f"agg{r}.npy")
        assert max_ms == pytest.approx(20.0)
        assert total == pytest.approx(2e9)
        assert gbs == pytest.approx(2e9 / 0.020 / 1e9)
