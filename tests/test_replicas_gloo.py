"""The N>1 path of bench.py on CPU: two gloo ranks, each an independent
replica, agree on the barrier and take the maximum of their timings."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import bench
    r = bench.Ranks(world)
    r.barrier()
    m = r.max(10.0 + rank)
    out.put((rank, r.world, m))
    r.close()


def test_two_rank_max_and_barrier():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(i, 2, port, q)) for i in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == [(0, 2, 11.0), (1, 2, 11.0)]


def _split_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    import torch as t

    import bench
    r = bench.Ranks(world, split=True, device_backend="gloo")
    counts = t.tensor([10 + rank, 1], dtype=t.int32)
    dW = t.full((3, 4), float(rank + 1))
    loss = t.tensor([0.25 * (rank + 1)])
    r.sum_(counts)
    r.sum_(dW, loss)
    out.put((rank, counts.tolist(), dW.tolist(), float(loss.item())))
    r.close()


def test_split_sums_counts_loss_and_dW_over_the_ranks():
    # the exchange of bench.py --split, on CPU tensors through a gloo device group
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_split_worker, args=(i, 2, port, q)) for i in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, counts, dW, loss in res:
        assert counts == [21, 2]
        assert dW == [[3.0] * 4] * 3
        assert loss == 0.75
