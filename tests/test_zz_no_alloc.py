"""The forward loss entry point that allocates nothing (grpo_loss_fwd_noalloc).

It exists for callers that cannot allocate device memory at the point where
they need the loss -- e.g. a step sharing the GPU with an inference engine
that has reserved all free memory -- and uses a fixed 8 MiB array inside the
library instead of a caller workspace.  These tests call it through the C ABI
twice in a row (the array keeps the previous call's contents) and compare it
with grpo_loss_fwd, the entry point that takes a workspace; and they compare
it with the fp64 oracle for every objective variant under both means, and for
fp16 inputs with a scattered mask.  The file sorts last so that a run
stopping at the first failure has run everything else.
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
from gpu_harness import DeviceWorkload  # noqa: E402
from test_gpu_parity import assert_fwd_parity  # noqa: E402

LOSS_RTOL = 1e-3
STAT_TOL = 1e-3


def _noalloc(dw, loss, stats, status):
    rg.grpo_loss_fwd_noalloc(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, loss, stats, status)
    torch.cuda.synchronize()


@pytest.mark.parametrize("name,over,seed", [
    ("tiny", {}, 0),
    ("tiny", dict(G=8, L=4096, d=256, V=5000, len_lo=1, len_hi=4096), 1),   # 32768 rows: the stated limit
])
def test_noalloc_matches_workspace_forward_twice(name, over, seed):
    cfg = synth.make_config(name, **over)
    wl = synth.generate(cfg, seed=seed)
    dw = DeviceWorkload(wl)
    dw.fwd()
    assert int(dw.status.item()) == 0
    ref_loss = float(dw.loss.item())
    ref_stats = dw.row_stats.cpu().numpy()
    for call in range(2):
        loss = torch.full((1,), float("nan"), dtype=torch.float32, device="cuda")
        stats = torch.full((cfg.N, 5), float("nan"), dtype=torch.float32, device="cuda")
        status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
        _noalloc(dw, loss, stats, status)
        assert int(status.item()) == 0, call
        got = float(loss.item())
        assert abs(got - ref_loss) <= LOSS_RTOL * max(abs(ref_loss), 1e-30), (call, got, ref_loss)
        s = stats.cpu().numpy()
        assert np.all(np.abs(s - ref_stats) <= STAT_TOL * np.maximum(1.0, np.abs(ref_stats))), call


def _noalloc_against_oracle(cfg, seed, mask=None, objective=0, loss_mode=0):
    wl = synth.generate(cfg, seed=seed)
    dw = DeviceWorkload(wl, mask=mask, objective=objective, loss_mode=loss_mode)
    dw.loss.fill_(float("nan"))
    dw.status.fill_(-1)
    _noalloc(dw, dw.loss, dw.row_stats, dw.status)
    res = dw.results()
    exp = oracle.expected(wl, mask=res["mask"], want_dH=False, want_dW=False, objective=objective,
                          loss_mode=loss_mode)
    assert_fwd_parity(res, exp)


@pytest.mark.parametrize("objective", ["grpo", "no_detach", "reverse_kl_q", "forward_kl"])
@pytest.mark.parametrize("loss_mode", [0, 1])
def test_noalloc_objectives_and_means_against_oracle(objective, loss_mode):
    # three prompt groups, one completion fully masked, a KL large enough to matter
    cfg = synth.make_config("tiny", n_groups=3, G=4, L=150, d=192, V=1000, len_lo=1, len_hi=150,
                            n_zero_seq=1, sigma_ref=0.3)
    _noalloc_against_oracle(cfg, 43, objective=objective, loss_mode=loss_mode)


def test_noalloc_fp16_scattered_mask_against_oracle():
    # fp16 inputs, ragged V and d, a mask that is not a prefix of each completion
    cfg = synth.make_config("tiny", dtype="fp16", G=4, L=200, d=320, V=777, sigma_ref=0.1)
    mask = (np.random.default_rng(47).random(cfg.N) < 0.45).astype(np.uint8)
    _noalloc_against_oracle(cfg, 47, mask=mask)


def test_noalloc_rejects_shapes_beyond_its_array():
    cfg = synth.make_config("tiny", G=8, L=4097, d=128, V=1024)      # 32776 rows > 32768
    shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V)
    dummy = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(rg.GrpoError) as e:
        rg.grpo_loss_fwd_noalloc(dummy, dummy, dummy, dummy, dummy, dummy, shape, dummy, None, dummy)
    assert e.value.code == 3          # GRPO_ERR_WORKSPACE
