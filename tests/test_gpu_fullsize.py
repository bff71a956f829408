"""GPU path vs the fp64 oracle at the full sizes of the model-head workloads.

Two runs per workload, on the full-size tensors:
  * sub-mask: the mask cut to three runs of consecutive rows (1, 9 and 130
    rows, the last spanning two 128-row tiles), so the oracle can compute
    everything -- loss, per-row terms, dH rows and all V x d entries of dW;
  * full mask, in the launch configuration bench.py times (default chunking):
    per-row terms and dH on sampled rows, which the oracle computes one by
    one, plus properties that hold at any size (the loss is the mean of the
    per-row objective, sum over the vocabulary of dW is zero, masked dH rows
    are zero).
The fp16 workload starts at loss scale 2^15 and halves while found_inf is set.
"""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

from gpu_harness import DeviceWorkload, host_f64  # noqa: E402
from test_gpu_parity import assert_fwd_parity  # noqa: E402

BIG = ["qwen2.5-1.5b-head", "llama-3.1-8b-head", "llama-3.1-8b-20k", "phi-4-14b-head-fp16"]


@pytest.fixture(scope="module", params=BIG)
def big(request):
    cfg = synth.CONFIGS[request.param]
    return synth.generate(cfg, seed=0)


def run_scaled(dw, cfg):
    scale = cfg.loss_scale
    dw.fwd_bwd(scale)
    halvings = 0
    while int(dw.found_inf.item()) == 1:
        assert cfg.dtype == "fp16", "bf16 gradients overflowed"
        scale /= 2
        halvings += 1
        assert halvings < 40
        dw.fwd_bwd(scale)
    return scale


def light_results(dw, rows):
    """What the full-size checks need, without copying the whole dH to the host."""
    cfg = dw.cfg
    idx = torch.from_numpy(np.asarray(rows, np.int64)).cuda()
    masked = dw.mask == 0
    return dict(
        loss=float(dw.loss.item()), status=int(dw.status.item()), found_inf=int(dw.found_inf.item()),
        row_stats=dw.row_stats.cpu().numpy().astype(np.float64), mask=dw.mask.cpu().numpy(),
        dH_rows=host_f64(dw.dH.index_select(0, idx), cfg.dtype),
        dH_masked_zero=bool((dw.dH[masked] == 0).all().item()) if bool(masked.any().item()) else True,
        dH_finite=bool(torch.isfinite(dw.dH).all().item()),
        dW=dw.dW.cpu().numpy(),
    )


def compare_dW(dW32, ref, scale):
    """max |dW/s - ref| <= 2e-2 max|ref|, in row blocks to bound host memory."""
    worst, top = 0.0, 0.0
    for v0 in range(0, ref.shape[0], 8192):
        a = dW32[v0:v0 + 8192].astype(np.float64) / scale
        b = ref[v0:v0 + 8192]
        worst = max(worst, float(np.abs(a - b).max()))
        top = max(top, float(np.abs(b).max()))
    assert worst <= 2e-2 * top, ("dW", worst, top)


def test_submask_full_shape(big):
    cfg = big.cfg
    rng = np.random.default_rng(17)
    full = oracle.build_mask(big.lengths, cfg.L)
    live = np.flatnonzero(big.lengths >= 140)
    mask = np.zeros(cfg.N, np.uint8)
    for run in (1, 9, 130):
        i = int(rng.choice(live))
        j = int(rng.integers(0, big.lengths[i] - run + 1))
        mask[i * cfg.L + j: i * cfg.L + j + run] = 1
    assert np.all(full[mask == 1] == 1)
    dw = DeviceWorkload(big, mask=mask)
    scale = run_scaled(dw, cfg)
    rows = np.flatnonzero(mask)
    res = light_results(dw, rows)
    del dw
    torch.cuda.empty_cache()
    exp = oracle.expected(big, mask=mask)
    assert_fwd_parity(res, exp)
    assert res["dH_masked_zero"] and res["dH_finite"]
    err = np.abs(res["dH_rows"] / scale - exp["dH"]).max()
    assert err <= 2e-2 * np.abs(exp["dH"]).max(), ("dH", err)
    compare_dW(res["dW"], exp["dW"], scale)


def test_full_mask_sampled_rows(big):
    cfg = big.cfg
    mask = oracle.build_mask(big.lengths, cfg.L)
    rows = oracle.valid_rows(mask)
    rng = np.random.default_rng(23)
    pick = set(rng.choice(rows, size=16, replace=False).tolist())
    for i, ln in enumerate(big.lengths):
        if ln > 0:
            pick.update({i * cfg.L, i * cfg.L + int(ln) - 1})
    sample = np.array(sorted(pick), np.int32)
    dw = DeviceWorkload(big)
    scale = run_scaled(dw, cfg)
    res = light_results(dw, sample)
    del dw
    torch.cuda.empty_cache()
    assert res["status"] == 0
    assert np.array_equal(res["mask"], mask)
    exp = oracle.expected(big, mask=mask, eval_rows=sample, want_dW=False)
    # per-row terms and dH rows on the sample
    rs = res["row_stats"][sample]
    for col, key in ((0, "lse_pol"), (1, "lse_ref"), (2, "q"), (3, "p")):
        ref = exp["terms"][key]
        assert np.all(np.abs(rs[:, col] - ref) <= 1e-3 * np.maximum(1.0, np.abs(ref))), key
    assert np.all(np.abs(rs[:, 4] - exp["terms"]["pen"]) <= 1e-5 + 1e-2 * np.abs(exp["terms"]["pen"]))
    dH = res["dH_rows"] / scale
    assert np.abs(dH - exp["dH"]).max() <= 2e-2 * np.abs(exp["dH"]).max()
    # the loss is the token mean of the per-row objective; its advantage part is exact
    A = exp["adv"][rows // cfg.L].astype(np.float64)
    ell = -A + cfg.beta * res["row_stats"][rows, 4]
    assert abs(res["loss"] - ell.mean()) <= 1e-5 * max(1e-3, abs(ell.mean()))
    a_part = -float(np.sum(big.lengths * exp["adv"].astype(np.float64))) / rows.size
    kl_ref_mean = float(np.mean(exp["terms"]["pen"]))
    assert res["loss"] - a_part >= 0
    # the KL part of the loss is beta times a mean KL of the size the sampled rows show
    kl_gpu_mean = (res["loss"] - a_part) / cfg.beta
    assert kl_ref_mean / 4 <= kl_gpu_mean <= 4 * kl_ref_mean + 1e-6
    # sum over the vocabulary of dW vanishes; masked rows of dH are exactly zero
    dW = res["dW"].astype(np.float64) / scale
    assert np.all(np.isfinite(dW)) and res["dH_finite"]
    assert np.abs(dW.sum(0)).max() <= 1e-3 * np.abs(dW).max() * np.sqrt(cfg.V)
    assert res["dH_masked_zero"]
