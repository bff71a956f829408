"""Data-parallel shards on one GPU, through the C ABI.

A batch of prompt groups is cut into two shards of whole groups.  Each shard
is run with grpo_loss_fwd_bwd_shard and the batch's counts (the sums of
grpo_shard_counts over the shards).  The shards' loss shares and dW must add
up to one grpo_loss_fwd_bwd call on the whole batch, every shard's dH rows
and per-row terms must equal the whole batch's bit for bit, and the sums must
match the fp64 oracle.  A shard whose rows are all masked contributes zero;
global counts below a shard's own are reported in its status word.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import rl_fine_tuning_gb300 as rg  # noqa: E402
from gpu_harness import DeviceWorkload, host_f64  # noqa: E402


def _counts(dw):
    c = torch.zeros(2, dtype=torch.int32, device="cuda")
    rg.grpo_shard_counts(dw.mask, dw.shape, c)
    return c


def _run_shard(dw, global_counts, scale=1.0):
    rg.grpo_loss_fwd_bwd_shard(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, global_counts, scale,
                               dw.ws, dw.loss, dw.dH, dw.dW, dw.found_inf, dw.row_stats, dw.status)
    torch.cuda.synchronize()


def _split_run(wl, n_shards, loss_mode=0, chunk_rows=0, masks=None):
    shards = synth.split_groups(wl, n_shards)
    dws = [DeviceWorkload(s, mask=None if masks is None else masks[i], chunk_rows=chunk_rows, loss_mode=loss_mode)
           for i, s in enumerate(shards)]
    cnts = [_counts(d) for d in dws]
    total = cnts[0].clone()
    for c in cnts[1:]:
        total += c                     # what an all-reduce of the counts gives
    for d in dws:
        _run_shard(d, total)
    return dws, cnts, total


CASES = [
    # name, overrides, seed, chunk rows
    ("tiny", dict(n_groups=4, G=4, L=96, d=128, V=1024, len_lo=1, len_hi=96, n_zero_seq=2, sigma_ref=0.3), 3, 0),
    ("tiny", dict(n_groups=2, G=4, L=300, d=320, V=777, len_lo=40, len_hi=300, sigma_ref=0.1), 4, 256),
]


@pytest.mark.parametrize("loss_mode", [0, 1])
@pytest.mark.parametrize("name,over,seed,chunk_rows", CASES)
def test_shards_add_up_to_the_whole_batch(name, over, seed, chunk_rows, loss_mode):
    cfg = synth.make_config(name, **over)
    wl = synth.generate(cfg, seed=seed)
    whole = DeviceWorkload(wl, chunk_rows=chunk_rows, loss_mode=loss_mode).fwd_bwd()
    assert int(whole.status.item()) == 0
    dws, cnts, total = _split_run(wl, 2, loss_mode=loss_mode, chunk_rows=chunk_rows)
    mask = oracle.build_mask(wl.lengths, cfg.L)
    assert total.tolist() == [int(mask.sum()), int(np.sum(wl.lengths > 0))]
    for d, c in zip(dws, cnts):
        assert int(d.status.item()) == 0
        m = d.mask.cpu().numpy()
        assert c.tolist() == list(oracle.shard_counts(m, d.cfg.n_seq, d.cfg.L))
    # losses and dW add up; dH rows and per-row terms are the whole batch's, bit for bit
    loss_sum = sum(float(d.loss.item()) for d in dws)
    loss_whole = float(whole.loss.item())
    assert abs(loss_sum - loss_whole) <= 1e-6 * max(abs(loss_whole), 1e-6), (loss_sum, loss_whole)
    dW_sum = sum(d.dW.double() for d in dws)
    err = float((dW_sum - whole.dW.double()).abs().max().item())
    assert err <= 1e-5 * float(whole.dW.abs().max().item()), err
    n = dws[0].cfg.N
    for r, d in enumerate(dws):
        assert torch.equal(d.dH.view(torch.int16), whole.dH[r * n:(r + 1) * n].view(torch.int16)), r
        assert torch.equal(d.row_stats, whole.row_stats[r * n:(r + 1) * n]), r
    # and the sums match the fp64 oracle on the whole batch
    exp = oracle.expected(wl, loss_mode=loss_mode)
    assert abs(loss_sum - exp["loss"]) <= 1e-3 * abs(exp["loss"])
    dW = dW_sum.cpu().numpy()
    assert np.abs(dW - exp["dW"]).max() <= 2e-2 * np.abs(exp["dW"]).max()
    dH = np.concatenate([host_f64(d.dH, cfg.dtype) for d in dws])[exp["rows"]]
    assert np.abs(dH - exp["dH"]).max() <= 2e-2 * np.abs(exp["dH"]).max()


def test_fully_masked_shard_contributes_nothing():
    cfg = synth.make_config("tiny", n_groups=2, G=4, L=128, d=128, V=1000, len_lo=1, len_hi=128)
    wl = synth.generate(cfg, seed=8)
    full = oracle.build_mask(wl.lengths, cfg.L)
    half = cfg.N // 2
    masks = [full[:half].copy(), np.zeros(half, np.uint8)]
    dws, cnts, total = _split_run(wl, 2, masks=masks)
    assert cnts[1].tolist() == [0, 0]
    assert int(dws[1].status.item()) == 0
    assert float(dws[1].loss.item()) == 0.0
    assert bool((dws[1].dW == 0).all().item()) and bool((dws[1].dH == 0).all().item())
    # the other shard alone then carries the batch: equal to a plain call on its rows
    plain = DeviceWorkload(synth.split_groups(wl, 2)[0], mask=masks[0]).fwd_bwd()
    assert abs(float(dws[0].loss.item()) - float(plain.loss.item())) <= 1e-6 * abs(float(plain.loss.item()))
    assert torch.equal(dws[0].dH.view(torch.int16), plain.dH.view(torch.int16))
    assert torch.equal(dws[0].dW, plain.dW)


def test_global_counts_below_the_shards_own_are_reported():
    cfg = synth.make_config("tiny", n_groups=2, G=4, L=64, d=128, V=512, len_lo=8, len_hi=64)
    d = DeviceWorkload(synth.split_groups(synth.generate(cfg, seed=9), 2)[0])
    c = _counts(d)
    too_small = c - torch.tensor([1, 0], dtype=torch.int32, device="cuda")
    _run_shard(d, too_small)
    assert int(d.status.item()) == 2                 # GRPO_ERR_SHAPE
    _run_shard(d, c)
    assert int(d.status.item()) == 0


def test_forward_only_shards_add_up_to_the_whole_batch():
    cfg = synth.make_config("tiny", n_groups=4, G=4, L=96, d=128, V=1024, len_lo=1, len_hi=96, n_zero_seq=2,
                            sigma_ref=0.3)
    wl = synth.generate(cfg, seed=3)
    for loss_mode in (0, 1):
        whole = DeviceWorkload(wl, loss_mode=loss_mode).fwd()
        dws = [DeviceWorkload(s, loss_mode=loss_mode) for s in synth.split_groups(wl, 2)]
        total = sum(_counts(d) for d in dws)
        for d in dws:
            rg.grpo_loss_fwd_shard(d.h_pol, d.h_ref, d.W, d.tokens, d.mask, d.adv, d.shape, total, d.ws, d.loss,
                                   d.row_stats, d.status)
        torch.cuda.synchronize()
        assert all(int(d.status.item()) == 0 for d in dws)
        loss = sum(float(d.loss.item()) for d in dws)
        assert abs(loss - float(whole.loss.item())) <= 1e-6 * abs(float(whole.loss.item())), loss_mode
        n = dws[0].cfg.N
        for r, d in enumerate(dws):
            assert torch.equal(d.row_stats, whole.row_stats[r * n:(r + 1) * n])
