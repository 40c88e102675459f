"""The multi-replica bench path on CPU: two gloo ranks, barrier and max-over-ranks timing, and the
per-rank inputs.

Requests are independent (no collective on the data path); each replica serves its own batch of
requests and the replicas only agree on the timed region (barrier) and report the slowest rank's
time.  Each gloo rank builds its bench workload on the CPU, exactly as it would on its GPU, and the
ranks compare what they built."""
import os
import socket

import numpy as np
import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench

    class A:
        impl = "reference"

    w, r, _ = bench.dist_setup(A())
    bench.barrier(w)
    got = bench.reduce_max(1.5 + r, w)
    # this rank's workload, built on the CPU the way run_ours builds it on the rank's GPU
    wl = bench.Workload(dict(bench.WORKLOADS["tiny"], R=3), 4, "cpu", seed=bench.replica_seed(r))
    trace = torch.from_numpy(wl.trace_host.copy())          # [steps][L][R][k]
    qsum = wl.q.float().sum().reshape(1)
    traces = [torch.empty_like(trace) for _ in range(world)]
    qsums = [torch.empty_like(qsum) for _ in range(world)]
    dist.all_gather(traces, trace)
    dist.all_gather(qsums, qsum)
    q.put((r, w, got, bench.replica_seed(r), [t.numpy() for t in traces], [float(x) for x in qsums]))
    dist.destroy_process_group()


def test_two_rank_max_over_ranks_and_own_requests():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=300) for _ in range(2)), key=lambda x: x[0])
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert [x[:3] for x in res] == [(0, 2, 2.5), (1, 2, 2.5)]
    # distinct seeds, so each replica serves a batch of its own
    assert res[0][3] != res[1][3]
    traces, qsums = res[0][4], res[0][5]
    assert all(np.array_equal(a, b) for a, b in zip(traces, res[1][4]))  # both ranks saw the same gather
    t0, t1 = traces
    assert t0.shape == t1.shape == (4, 1, 3, 256)
    for r in range(3):
        # request r of rank 0 and request r of rank 1 select different positions at every step
        for t in range(4):
            assert not np.array_equal(np.sort(t0[t, 0, r]), np.sort(t1[t, 0, r])), (r, t)
    assert qsums[0] != qsums[1]
