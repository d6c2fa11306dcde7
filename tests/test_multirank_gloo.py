"""The multi-rank path on CPU with two gloo ranks: decode shards by sequence
with no exchange, so ranks run independent replicas; the only cross-rank
operations are the timing barrier and the max-reduction of the elapsed time.
Each rank also runs the oracle on its own shard of a batch and the shards
together reproduce the whole batch's result (sequence sharding needs no
collective)."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, result_dir):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    from oracle.attention import paged_decode
    from workloads import make_decode_case
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slow one
        t_max = bench.reduce_max_ms(local_ms, dist)
        value = bench.whole_job_gbps(1_000_000, 4, world, t_max)
        # shard a batch by sequence: rank r takes sequences r, r + world, ...
        wl = make_decode_case(77, [5, 40, 17, 90, 33, 64], 8, 2, 64)
        mine = np.arange(rank, len(wl.dec_ctx), world)
        out = paged_decode(wl.q[mine], wl.k_pool, wl.v_pool, wl.dec_tables[mine], wl.dec_ctx[mine], wl.scale)
        np.save(os.path.join(result_dir, f"shard{rank}.npy"), out)
        np.save(os.path.join(result_dir, f"timing{rank}.npy"), np.array([t_max, value]))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_timing_and_sequence_shards(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    t0 = np.load(tmp_path / "timing0.npy")
    t1 = np.load(tmp_path / "timing1.npy")
    assert t0[0] == t1[0] == 15.0               # both ranks see the slowest rank's time
    assert np.isclose(t0[1], 2 * 1_000_000 * 4 / 0.015 / 1e9)
    from oracle.attention import paged_decode
    from workloads import make_decode_case
    wl = make_decode_case(77, [5, 40, 17, 90, 33, 64], 8, 2, 64)
    whole = paged_decode(wl.q, wl.k_pool, wl.v_pool, wl.dec_tables, wl.dec_ctx, wl.scale)
    s0, s1 = np.load(tmp_path / "shard0.npy"), np.load(tmp_path / "shard1.npy")
    assert np.array_equal(whole[0::2], s0) and np.array_equal(whole[1::2], s1)


def test_single_rank_reduction_is_identity():
    import bench
    assert bench.reduce_max_ms(12.5, None) == 12.5
    assert np.isclose(bench.whole_job_gbps(586_436_608, 10, 1, 1.0), 5864.36608)
