"""The build with device-side index checks (libgrpo_checked.so): a check made
to fail on purpose reports GRPO_ERR_BOUNDS, and the parity cases with every
tail (ragged V and d, several chunks, scattered and empty masks, degenerate
shapes, fp16, 8-bit inputs forward and backward, data-parallel shards, the
workspace-free forward) run through it with no check firing and the same
results as the oracle."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import rl_fine_tuning_gb300 as rg  # noqa: E402
from rl_fine_tuning_gb300 import build  # noqa: E402
from gpu_harness import DeviceWorkload  # noqa: E402
from test_gpu_parity import assert_fwd_parity, assert_grad_parity  # noqa: E402
from test_gpu_fp8 import assert_fp8_grad_parity, run_fp8, run_fp8_bwd  # noqa: E402


@pytest.fixture()
def checked(monkeypatch):
    build.build()
    monkeypatch.setattr(build, "LIB", build.LIB_CHECKED)
    monkeypatch.setattr(rg, "_lib", None)
    assert rg.grpo_device_checks()
    yield


def test_a_failing_check_reports_bounds(checked):
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    rg.grpo_selftest_bounds_check(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 8, rg.grpo_status_string(int(status.item()))


CASES = [
    ("tiny", dict(), 0, None),
    ("ragged", dict(G=3, L=333, d=320, V=1000, len_lo=1, len_hi=333), 256, None),
    ("scattered", dict(G=2, L=200, d=128, V=777), 128, "scattered"),
    ("v1", dict(V=1), 0, None),
    ("d64", dict(d=64, V=200), 0, None),
    ("no_even_split", dict(G=2, L=100, d=64, V=257 * 256, len_lo=40, len_hi=100), 0, None),
    ("all_masked", dict(), 0, "empty"),
    ("wide_dh", dict(G=4, L=4096, d=768, V=1000, len_lo=1500, len_hi=4096), 76 * 128, None),   # 512-column dH units
]


@pytest.mark.parametrize("name,over,chunk_rows,mask_kind", CASES, ids=[c[0] for c in CASES])
def test_parity_cases_pass_the_checks(checked, name, over, chunk_rows, mask_kind):
    cfg = synth.make_config("tiny", **over)
    wl = synth.generate(cfg, seed=21)
    mask = None
    if mask_kind == "scattered":
        mask = (np.random.default_rng(5).random(cfg.N) < 0.45).astype(np.uint8)
    elif mask_kind == "empty":
        mask = np.zeros(cfg.N, np.uint8)
    dw = DeviceWorkload(wl, mask=mask, chunk_rows=chunk_rows)
    res = dw.fwd_bwd().results()
    assert res["status"] == 0, rg.grpo_status_string(res["status"])
    exp = oracle.expected(wl, mask=res["mask"])
    if mask_kind == "empty":
        assert res["loss"] == 0.0 and np.all(res["dH"] == 0) and np.all(res["dW"] == 0)
        return
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)
    res2 = dw.fwd().results()
    assert res2["status"] == 0 and res2["loss"] == res["loss"]


def test_fp16_scaled_through_the_checks(checked):
    cfg = synth.make_config("tiny", dtype="fp16", sigma_ref=0.05)
    wl = synth.generate(cfg, seed=8)
    res = DeviceWorkload(wl).fwd_bwd(loss_scale=256.0).results()
    assert res["status"] == 0 and res["found_inf"] == 0
    exp = oracle.expected(wl, mask=res["mask"])
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp, loss_scale=256.0)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_forward_through_the_checks(checked, fmt):
    cfg = synth.make_config("tiny", G=4, L=500, d=384, V=3000, len_lo=1, len_hi=500)
    res, exp = run_fp8(synth.generate_fp8(cfg, seed=41, fmt=fmt))
    assert res["status"] == 0
    assert_fwd_parity(res, exp)


def test_workspace_free_forward_through_the_checks(checked):
    cfg = synth.make_config("tiny", G=3, L=333, d=320, V=1000, len_lo=1, len_hi=333)
    wl = synth.generate(cfg, seed=2)
    dw = DeviceWorkload(wl)
    rg.grpo_loss_fwd_noalloc(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, dw.loss, dw.row_stats,
                             dw.status)
    torch.cuda.synchronize()
    res = dw.results()
    assert res["status"] == 0
    assert_fwd_parity(res, oracle.expected(wl, mask=res["mask"], want_dH=False, want_dW=False))


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_backward_through_the_checks(checked, fmt):
    # ragged V over several chunks, and many rows per token (the sorted keys of the dW epilogue)
    for over, chunk_rows in ((dict(G=4, L=500, d=384, V=3000, len_lo=1, len_hi=500), 256),
                             (dict(G=4, L=256, d=256, V=200, len_lo=64, len_hi=256), 128)):
        cfg = synth.make_config("tiny", **over)
        res, exp = run_fp8_bwd(synth.generate_fp8(cfg, seed=43, fmt=fmt), chunk_rows=chunk_rows)
        assert res["status"] == 0
        assert_fp8_grad_parity(res, exp)


def test_shards_through_the_checks(checked):
    cfg = synth.make_config("tiny", n_groups=2, G=4, L=300, d=320, V=777, len_lo=40, len_hi=300)
    wl = synth.generate(cfg, seed=4)
    whole = DeviceWorkload(wl, chunk_rows=256).fwd_bwd()
    dws = [DeviceWorkload(s, chunk_rows=256) for s in synth.split_groups(wl, 2)]
    counts = [torch.zeros(2, dtype=torch.int32, device="cuda") for _ in dws]
    for d, c in zip(dws, counts):
        rg.grpo_shard_counts(d.mask, d.shape, c)
    total = counts[0] + counts[1]
    for d in dws:
        rg.grpo_loss_fwd_bwd_shard(d.h_pol, d.h_ref, d.W, d.tokens, d.mask, d.adv, d.shape, total, 1.0, d.ws, d.loss,
                                   d.dH, d.dW, d.found_inf, d.row_stats, d.status)
    torch.cuda.synchronize()
    assert all(int(d.status.item()) == 0 for d in dws)
    n = dws[0].cfg.N
    for r, d in enumerate(dws):
        assert torch.equal(d.dH.view(torch.int16), whole.dH[r * n:(r + 1) * n].view(torch.int16))
    loss = sum(float(d.loss.item()) for d in dws)
    assert abs(loss - float(whole.loss.item())) <= 1e-6 * abs(float(whole.loss.item()))
