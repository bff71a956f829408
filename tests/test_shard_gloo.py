"""The data-parallel split of the loss on CPU ranks, through the fp64 oracle.

Two gloo ranks each hold half of a batch's prompt groups (whole groups, so
the advantages need no exchange) and the shared W.  Each rank counts its
masked-in rows and active completions, the ranks sum the counts, each rank
takes the oracle's loss share, dH and dW with the batch's divisors, and the
ranks sum the loss shares and dW.  The sums must equal the one-rank oracle
on the whole batch, and every rank's dH rows the whole batch's rows, under
both means.  This pins the shard weights of the oracle to its own whole-batch
definition and checks the exchange protocol the library's shard entry points
are made for.
"""
import os
import socket

import numpy as np
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


def _config():
    import synth
    # four prompt groups; one completion fully masked; ragged V and d
    return synth.make_config("tiny", n_groups=4, G=3, L=40, d=96, V=301, len_lo=1, len_hi=40, n_zero_seq=1,
                             sigma_ref=0.3)


def _shard_result(wl, counts_batch, loss_mode):
    import oracle
    cfg = wl.cfg
    adv = oracle.group_advantages(wl.rewards, cfg.n_groups, cfg.G, cfg.eps, True)
    mask = oracle.build_mask(wl.lengths, cfg.L)
    rows = oracle.valid_rows(mask)
    terms = oracle.row_terms(wl.h_pol, wl.h_ref, wl.W, cfg.dtype, wl.tokens, adv, cfg.L, rows, cfg.beta)
    w = oracle.row_weights_shard(rows, cfg.L, counts_batch[0], counts_batch[1], loss_mode)
    share = oracle.weighted_sum(terms["ell"], w)
    dH, dW = oracle.grad(wl.h_pol, wl.W, cfg.dtype, wl.tokens, rows, terms["lse_pol"], terms["g"], w)
    return share, rows, dH, dW


def _worker(rank, world, port, loss_mode, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    import torch.distributed as dist

    import oracle
    import synth
    oracle.set_threads(1)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        wl = synth.split_groups(synth.generate(_config(), seed=5), world)[rank]
        cfg = wl.cfg
        mask = oracle.build_mask(wl.lengths, cfg.L)
        counts = torch.tensor(oracle.shard_counts(mask, cfg.n_seq, cfg.L), dtype=torch.int64)
        dist.all_reduce(counts)
        share, rows, dH, dW = _shard_result(wl, counts.tolist(), loss_mode)
        loss = torch.tensor([share], dtype=torch.float64)
        dW_t = torch.from_numpy(dW)
        dist.all_reduce(loss)
        dist.all_reduce(dW_t)
        q.put((rank, counts.tolist(), float(loss.item()), dW_t.numpy(), rows + rank * cfg.N, dH))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("loss_mode", [0, 1])
def test_two_shards_sum_to_the_whole_batch(loss_mode):
    import oracle
    import synth
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(i, 2, port, loss_mode, q)) for i in range(2)]
    for p in procs:
        p.start()
    res = sorted((q.get(timeout=180) for _ in procs), key=lambda r: r[0])
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0

    wl = synth.generate(_config(), seed=5)
    exp = oracle.expected(wl, loss_mode=loss_mode)
    n_act = int(np.sum(wl.lengths > 0))
    for rank, counts, loss, dW, rows, dH in res:
        assert counts == [exp["n_valid"], n_act]
        assert abs(loss - exp["loss"]) <= 1e-12 * max(1.0, abs(exp["loss"]))
        assert np.abs(dW - exp["dW"]).max() <= 1e-12 * np.abs(exp["dW"]).max()
        idx = np.searchsorted(exp["rows"], rows)
        assert np.array_equal(exp["rows"][idx], rows)
        assert np.abs(dH - exp["dH"][idx]).max() <= 1e-12 * np.abs(exp["dH"]).max()
    # the shards hold every masked-in row once
    assert np.array_equal(np.concatenate([r[4] for r in res]), exp["rows"])


def test_one_shard_holding_the_batch_is_the_batch_mean():
    import oracle
    import synth
    wl = synth.generate(_config(), seed=6)
    cfg = wl.cfg
    mask = oracle.build_mask(wl.lengths, cfg.L)
    nv, nact = oracle.shard_counts(mask, cfg.n_seq, cfg.L)
    rows = oracle.valid_rows(mask)
    assert nv == rows.size and nact == int(np.sum(wl.lengths > 0))
    for mode in (0, 1):
        np.testing.assert_allclose(oracle.row_weights_shard(rows, cfg.L, nv, nact, mode),
                                   oracle.row_weights(rows, cfg.L, mode), rtol=0, atol=0)
        ell = np.linspace(-1.0, 2.0, rows.size)
        assert abs(oracle.weighted_sum(ell, oracle.row_weights(rows, cfg.L, mode)) -
                   oracle.reduce_loss(ell, rows, cfg.L, mode)) <= 1e-14
