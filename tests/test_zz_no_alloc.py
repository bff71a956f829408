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


_LAZY_SCRIPT = r"""
import os, sys
sys.path.insert(0, os.environ["GRPO_ROOT"]); sys.path.insert(0, os.path.join(os.environ["GRPO_ROOT"], "tests"))
import torch
import rl_fine_tuning_gb300 as rg
import synth
from gpu_harness import DeviceWorkload
cfg = synth.make_config("tiny", G=8, L=512, d=256, V=3000, len_lo=1, len_hi=512)
dw = DeviceWorkload(synth.generate(cfg, seed=2))
outs = [(torch.full((1,), float("nan"), device="cuda"), torch.full((cfg.N, 5), float("nan"), device="cuda"),
         torch.full((1,), -1, dtype=torch.int32, device="cuda")) for _ in range(2)]
def call(o):
    rg.grpo_loss_fwd_noalloc(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, o[0], o[1], o[2])
    torch.cuda.synchronize()
call(outs[0])                                   # first call on the device: the library's set-up
free, _ = torch.cuda.mem_get_info()
hold = torch.empty(free - (256 << 20), dtype=torch.uint8, device="cuda")   # the device's memory handed elsewhere
free_after, _ = torch.cuda.mem_get_info()
call(outs[1])
assert int(outs[0][2].item()) == 0 and int(outs[1][2].item()) == 0
assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
del hold
print("OK", free_after >> 20)
"""


def test_noalloc_second_call_needs_no_free_memory_under_lazy_loading():
    # In a fresh process with lazy module loading: after the first call, all but
    # 256 MiB of the device's free memory is taken by someone else; the next
    # call must still run and give the same bits.
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY", GRPO_ROOT=root)
    r = subprocess.run([sys.executable, "-c", _LAZY_SCRIPT], env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "OK" in r.stdout, (r.stdout[-2000:], r.stderr[-4000:])
