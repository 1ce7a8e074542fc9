"""The multi-GPU layout on the CPU with gloo, world size 2: ranks shard the
independent (batch, channel) scans with no data-path exchange, and the
benchmark's timing reduction takes the slowest rank. The per-rank compute here
is the oracle (no GPU in this test)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    from workloads import gen

    # shard the channels of one problem across ranks: no exchange is needed
    x = gen.random_scan_inputs(2, 48, 10, 16, in_dtype="bf16", seed=5, with_h0=True)
    chans = np.array([[b, d] for b in range(2) for d in range(10)])
    mine = chans[rank::world]
    y, h = oracle.scan(x, channels=mine, nthreads=1)
    np.save(os.path.join(out_dir, f"y{rank}.npy"), y)
    np.save(os.path.join(out_dir, f"h{rank}.npy"), h)
    np.save(os.path.join(out_dir, f"c{rank}.npy"), mine)
    # the benchmark's timing reduction: every rank sees the slowest rank's time
    t = bench.max_over_ranks(world, 1.5 + rank)
    np.save(os.path.join(out_dir, f"t{rank}.npy"), np.array([t]))
    # weak scaling: each rank's own batch is seeded differently
    from workloads import configs
    np.save(os.path.join(out_dir, f"s{rank}.npy"), np.array([bench.rank_seed(configs.MAMBA2P8B_LAYER, rank)]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, start_method="spawn",
                       join=True)
    import oracle
    from workloads import gen

    x = gen.random_scan_inputs(2, 48, 10, 16, in_dtype="bf16", seed=5, with_h0=True)
    yf, hf = oracle.scan(x)
    for r in range(world):
        ch = np.load(tmp_path / f"c{r}.npy")
        y = np.load(tmp_path / f"y{r}.npy")
        h = np.load(tmp_path / f"h{r}.npy")
        for i, (b, d) in enumerate(ch):
            assert np.array_equal(y[i], yf[b, :, d]) and np.array_equal(h[i], hf[b, d])
        assert float(np.load(tmp_path / f"t{r}.npy")[0]) == 2.5
    assert np.load(tmp_path / "s0.npy")[0] != np.load(tmp_path / "s1.npy")[0]
