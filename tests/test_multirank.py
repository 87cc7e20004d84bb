"""World-size-2 host logic of the multi-GPU benchmark path, on CPU with gloo.

Documents are independent, so N ranks each score their own documents (weak
scaling) with no data-path collective; the only cross-rank step is the max
of the per-rank elapsed times. These tests run that logic in two gloo ranks.
"""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads
    local_ms = 10.0 + 5.0 * rank
    mx = bench.max_over_ranks(local_ms, world, "cpu")
    rate = bench.whole_job_rate(1000, 4, world, mx)
    # each rank's documents differ (own seed), so the job covers world x B distinct documents
    D = workloads.normalized_tokens((4, 8, 64), seed=bench.rank_seed(rank) + 1, dtype="fp32")
    gathered = [torch.zeros_like(D) for _ in range(world)]
    dist.all_gather(gathered, D)
    distinct = not torch.equal(gathered[0], gathered[1])
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, mx, rate, distinct))


def test_two_rank_timing_aggregation_and_sharding():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, rate, distinct in res:
        assert mx == 15.0                       # max over ranks, seen by every rank
        assert rate == pytest.approx(1000 * 4 * 2 / 0.015)
        assert distinct


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(3.5, 1, "cpu") == 3.5


def _dq_worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import numpy as np
    import oracle
    import workloads
    import maxsim_scoring_02_gb300 as m
    # shared query; each rank owns different documents and their dS
    Q = workloads.normalized_tokens((2, 6, 16), seed=5, dtype="fp32").double().numpy()
    D = workloads.normalized_tokens((3, 7, 16), seed=100 + rank, dtype="fp32").double().numpy()
    dS = workloads.normal((2, 3), seed=200 + rank).double().numpy()
    _, am, _ = oracle.maxsim(Q, D)
    dQ_local, _ = oracle.backward(Q, D, am, dS)
    dQ = torch.tensor(dQ_local)
    m.allreduce_dq(dQ)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, dQ.numpy()))


def test_sharded_backward_dq_allreduce_equals_full_gradient():
    """Two ranks with disjoint documents: the all-reduced dQ equals the
    oracle's dQ over the union of both ranks' documents."""
    import numpy as np
    import oracle
    import workloads
    ctx = mp.get_context("spawn")
    qu = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_dq_worker, args=(r, 2, port, qu)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(qu.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    Q = workloads.normalized_tokens((2, 6, 16), seed=5, dtype="fp32").double().numpy()
    D = np.concatenate([workloads.normalized_tokens((3, 7, 16), seed=100 + r, dtype="fp32").double().numpy()
                        for r in range(2)])
    dS = np.concatenate([workloads.normal((2, 3), seed=200 + r).double().numpy() for r in range(2)], axis=1)
    _, am, _ = oracle.maxsim(Q, D)
    dQ_full, _ = oracle.backward(Q, D, am, dS)
    for r in range(2):
        np.testing.assert_allclose(res[r], dQ_full, rtol=1e-12, atol=1e-12)
