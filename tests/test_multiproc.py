"""Multi-rank host logic of bench.py on CPU: two gloo ranks, weak scaling.

Every rank verifies its own batch; the job's verified tokens are summed over the ranks and the
step time is the slowest rank's. No GPU and no data-path collective are involved.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    from speculative_decoding_verification_33_gb300 import workloads as W
    w = W.small_variant(W.WORKLOADS[5], B=6, V=64)
    d = W.make_inputs(w, offset=rank, threads=1)  # each rank its own replica of the workload
    toks = float(d["draft_lens"].sum())
    total, ms = bench.aggregate(toks, 10.0 * (rank + 1))
    out[rank] = (toks, total, ms, bench.dist_env())
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
    toks = [out[r][0] for r in range(world)]
    for r in range(world):
        _, total, ms, env = out[r]
        assert total == sum(toks)           # units all ranks processed
        assert ms == 10.0 * world           # the slowest rank's time
        assert env == (r, world, r)


def test_single_rank_aggregation_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.aggregate(7.0, 3.5) == (7.0, 3.5)
