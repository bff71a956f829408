"""Two independent loss calls in flight at once on two streams, each with its
own workspace and outputs, give the same bits as the same calls one after the
other: the path keeps no state outside the caller's buffers."""
import pytest

import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import rl_fine_tuning_gb300 as rg  # noqa: E402
from gpu_harness import DeviceWorkload  # noqa: E402


def _call(dw, stream):
    cfg = dw.cfg
    with torch.cuda.stream(stream):
        rg.grpo_group_advantages(dw.rewards, cfg.n_groups, cfg.G, cfg.eps, True, dw.adv)
        rg.grpo_build_mask(dw.lengths, dw.shape, dw.mask)
        rg.grpo_loss_fwd_bwd(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, 1.0, dw.ws, dw.loss,
                             dw.dH, dw.dW, dw.found_inf, dw.row_stats, dw.status)


def _snapshot(dw):
    return [t.clone() for t in (dw.loss, dw.dH, dw.dW, dw.row_stats, dw.status)]


def _same(a, b):
    return all(torch.equal(x.view(torch.uint8), y.view(torch.uint8)) for x, y in zip(a, b))


def test_concurrent_calls_on_two_streams_match_sequential():
    cfg_a = synth.make_config("tiny", G=3, L=333, d=320, V=1000, len_lo=1, len_hi=333)
    cfg_b = synth.make_config("tiny", G=4, L=200, d=256, V=777, sigma_ref=0.3)
    a = DeviceWorkload(synth.generate(cfg_a, seed=31), chunk_rows=256)
    b = DeviceWorkload(synth.generate(cfg_b, seed=32), chunk_rows=128)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())

    _call(a, s1)
    s1.synchronize()
    _call(b, s1)
    s1.synchronize()
    seq_a, seq_b = _snapshot(a), _snapshot(b)
    assert int(seq_a[-1].item()) == 0 and int(seq_b[-1].item()) == 0

    for _ in range(3):
        for dw in (a, b):
            dw.dH.fill_(7.0)
            dw.dW.fill_(7.0)
            dw.loss.fill_(7.0)
        torch.cuda.synchronize()
        _call(a, s1)
        _call(b, s2)
        torch.cuda.synchronize()
        assert _same(_snapshot(a), seq_a)
        assert _same(_snapshot(b), seq_b)
