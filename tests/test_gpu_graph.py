"""A whole step (advantages, mask, fused loss forward+backward) captured into
one CUDA graph and replayed gives the eager result bit for bit, also after the
inputs change in place between replays: nothing in the captured launches
depends on host-side knowledge of the data (the chunk count is the bound for
all rows masked in; empty chunks exit on the device)."""
import numpy as np
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import rl_fine_tuning_gb300 as rg  # noqa: E402
from gpu_harness import DeviceWorkload, dev_bits  # noqa: E402


def _call(dw):
    cfg = dw.cfg
    rg.grpo_group_advantages(dw.rewards, cfg.n_groups, cfg.G, cfg.eps, True, dw.adv)
    rg.grpo_build_mask(dw.lengths, dw.shape, dw.mask)
    rg.grpo_loss_fwd_bwd(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, 1.0, dw.ws, dw.loss,
                         dw.dH, dw.dW, dw.found_inf, dw.row_stats, dw.status)


def _outputs(dw):
    return [t.clone() for t in (dw.loss, dw.dH, dw.dW, dw.row_stats, dw.adv, dw.mask, dw.status)]


def _poison(dw):
    for t in (dw.loss, dw.dW, dw.row_stats):
        t.fill_(7.0)
    dw.dH.fill_(7.0)


def _same(a, b):
    return all(torch.equal(x.view(torch.uint8), y.view(torch.uint8)) for x, y in zip(a, b))


def test_graph_replay_is_bitwise_equal_to_eager():
    cfg = synth.make_config("tiny", G=3, L=333, d=320, V=1000, len_lo=1, len_hi=333)
    wl = synth.generate(cfg, seed=3)
    dw = DeviceWorkload(wl, chunk_rows=256)

    _call(dw)
    torch.cuda.synchronize()
    eager = _outputs(dw)
    assert int(dw.status.item()) == 0

    # warm up on a side stream, then capture on it
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _call(dw)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(dw)

    for _ in range(2):
        _poison(dw)
        g.replay()
        torch.cuda.synchronize()
        assert _same(_outputs(dw), eager)

    # new hidden states, tokens, lengths and rewards written into the same buffers
    wl2 = synth.generate(cfg, seed=4)
    dw.h_pol.copy_(dev_bits(wl2.h_pol, cfg.dtype))
    dw.h_ref.copy_(dev_bits(wl2.h_ref, cfg.dtype))
    dw.tokens.copy_(torch.from_numpy(wl2.tokens))
    dw.lengths.copy_(torch.from_numpy(wl2.lengths))
    dw.rewards.copy_(torch.from_numpy(wl2.rewards))
    _poison(dw)
    g.replay()
    torch.cuda.synchronize()
    replayed = _outputs(dw)
    _poison(dw)
    _call(dw)
    torch.cuda.synchronize()
    assert _same(replayed, _outputs(dw))
    assert not np.array_equal(replayed[1].cpu().view(torch.int16).numpy(), eager[1].cpu().view(torch.int16).numpy())
