"""The N>1 benchmark path on CPU: two gloo ranks, independent replicas, max-over-ranks timing.

Decode attention has no exchange step, so multi-GPU runs are independent
replicas; the only cross-rank traffic is the barrier and the max of the
ranks' timings. This exercises exactly that code (bench.aggregate_throughput)
with world_size 2 over gloo.
"""

import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, ws, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=ws)
    import bench
    import workloads
    ws_, rank_, local_ = bench.dist_env()
    assert (ws_, rank_, local_) == (ws, rank, rank)
    # each replica draws its own batch (seed + rank) of the same shape
    cfg = workloads.CONFIGS[workloads.SMALL].with_(num_seqs=2, ctx=64)
    b = workloads.make_batch(cfg, seed=cfg.seed + rank)
    per_rank_bytes = workloads.algorithmic_bytes(cfg, b.seq_lens_host)
    elapsed = [10.0, 25.0][rank]
    dist.barrier()
    value, ms = bench.aggregate_throughput(per_rank_bytes, 4, elapsed, ws, torch.device("cpu"))
    q.put((rank, value, ms, per_rank_bytes, float(b.q.float().sum())))
    dist.destroy_process_group()


def test_two_replicas_max_timing():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in ps]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    (_, v0, ms0, b0, qs0), (_, v1, ms1, b1, qs1) = res
    assert ms0 == ms1 == 25.0, "every rank must report the slowest rank's time"
    assert v0 == v1 == pytest.approx(2 * b0 * 4 / 25e-3 / 1e9)
    assert b0 == b1
    assert qs0 != qs1, "replicas must draw different inputs"
