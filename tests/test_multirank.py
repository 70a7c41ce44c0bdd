"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

With --shard sequences each rank runs its own independent sequence; with
--shard pairs (tests/test_sharded.py covers the split itself) the ranks share
one layer's head pairs.  Either way only the step time is reduced (max over
ranks) to form the whole-job throughput.  This runs that reduction and the
rank -> sequence assignment in two real gloo processes.
"""
import os
import socket

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import gdn_synth
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ms = 10.0 + 5.0 * rank                       # rank 1 is the slow one
    step = bench.reduce_step_ms(ms, world, "cpu")
    x = gdn_synth.make_inputs(1, 128, 1, 2, dtype="f32", seed=gdn_synth.seed_for(2, 0, bench.rank_batch_index(rank)))
    out[rank] = (step, bench.job_throughput(128, world, step), float(x.v.sum()))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_reduction_and_sharding():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 15.0        # max over ranks
    assert res[0][1] == res[1][1] == pytest.approx(2 * 128 / 0.015)
    assert res[0][2] != res[1][2]                # each rank draws its own sequence
