"""The N > 1 path of bench.py on CPU ranks (gloo, world size 2).

The hot path shards by sequence with no exchange step: each rank times its own
batch (a different seeded workload), the ranks meet at a barrier, and the job
time is the maximum over ranks.  This checks that host logic without a GPU.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    import bench
    d, r, w = bench._dist()
    assert (r, w) == (rank, world)
    bench._barrier(d)
    # each rank reports its own elapsed time; every rank must see the maximum
    mx = bench._max_over_ranks(d, 10.0 + 5.0 * rank, torch.device("cpu"))
    # ranks draw different batches (weak scaling): seeds differ by the rank
    import zp_inputs
    B, h_q, h_kv, d_, b, N_max, lr, dtype, seed = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    c = zp_inputs.make_paged_case(seed + rank, 4, 4, 2, 16, 16, len_range=(16, 64), dtype="f32")
    out[rank] = (mx, int(c.seq_lens.sum()))
    dist.destroy_process_group()


def test_two_gloo_ranks_time_is_max_over_ranks():
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 15.0
    assert out[0][1] != out[1][1]  # different batches per rank
