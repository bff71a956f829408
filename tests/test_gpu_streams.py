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


def test_calls_from_two_host_threads_match_sequential():
    """Two host threads call the library at once (ctypes releases the GIL for
    the call), with per-kernel profiling on: the same bits as sequential
    calls, and the profiler counts every launch of both threads once."""
    import threading

    cfg_a = synth.make_config("tiny", G=2, L=300, d=192, V=900, len_lo=1, len_hi=300)
    cfg_b = synth.make_config("tiny", G=4, L=128, d=128, V=1300, sigma_ref=0.2)
    a = DeviceWorkload(synth.generate(cfg_a, seed=41), chunk_rows=128)
    b = DeviceWorkload(synth.generate(cfg_b, seed=42), chunk_rows=256)
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    s1.wait_stream(torch.cuda.current_stream())
    s2.wait_stream(torch.cuda.current_stream())
    reps = 4

    rg.grpo_profile_enable(True)
    try:
        rg.grpo_profile_collect()
        _call(a, s1)
        _call(b, s1)
        s1.synchronize()
        once = rg.grpo_profile_collect()
        seq_a, seq_b = _snapshot(a), _snapshot(b)
        assert int(seq_a[-1].item()) == 0 and int(seq_b[-1].item()) == 0

        errors = []
        start = threading.Barrier(2)

        def worker(dw, stream):
            try:
                torch.cuda.set_device(0)
                start.wait(timeout=60)
                for _ in range(reps):
                    _call(dw, stream)
            except Exception as e:   # re-raised in the main thread
                errors.append(e)

        threads = [threading.Thread(target=worker, args=(a, s1)), threading.Thread(target=worker, args=(b, s2))]
        for t in threads:
            t.start()
        for t in threads:
            t.join()
        torch.cuda.synchronize()
        assert not errors, errors
        prof = rg.grpo_profile_collect()
    finally:
        rg.grpo_profile_enable(False)
        rg.grpo_profile_collect()
    assert _same(_snapshot(a), seq_a)
    assert _same(_snapshot(b), seq_b)
    for kind, (_, n) in once.items():
        assert prof[kind][1] == reps * n, (kind, prof[kind][1], n)
