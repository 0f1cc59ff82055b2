"""The multi-rank host logic of the benchmark on CPU, world size 2 (gloo).

The hot path shards by units: every rank builds and decodes its own batch
(disjoint sequences, no exchange of data), and the only collective is the
max of the ranks' timings, from which the whole-job rate is computed.
"""
import os
import socket

import pytest


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads

    w = bench.rank_workload("llama31_8b_16k", rank)
    slowest = bench.max_over_ranks(10.0 + rank, world, "cpu")
    rate = bench.whole_job_rate(w.units * w.n_tokens, 3, world, slowest)
    K, _ = workloads.unit_kv(w.scaled(n_tokens=64), 0, 0, 0)
    q.put((rank, w.seed, slowest, rate, float(K.astype("float64").sum())))
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_weak_scaling_host_logic():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (_, s0, m0, v0, k0), (_, s1, m1, v1, k1) = res
    assert s0 != s1 and k0 != k1  # each rank owns different sequences
    assert m0 == m1 == 11.0  # both ranks see the slowest rank's time
    expect = 2 * 8 * 16384 * 3 / 11.0e-3
    assert v0 == pytest.approx(expect) and v1 == pytest.approx(expect)
