"""GPU path vs the fp64 oracle at the full sizes of the model-head workloads.

Runs per workload, on the full-size tensors:
  * sub-mask: the mask cut to four runs of consecutive rows (1, 9, 130 and
    260 rows in different completions, 400 rows), so the oracle can compute
    everything -- loss, per-row terms, every dH row and all V x d entries of
    dW.  It runs at the default chunk height (one chunk) and at 128-row
    chunks (four chunks: dW read-modify-written four times at the full V x d);
  * full mask, in the launch configuration bench.py times (default
    chunking): per-row terms and dH on sampled rows, which the oracle
    computes one by one; where tests/golden holds the oracle's full-mask
    values (written offline by tests/golden/make_fullmask_golden.py), the
    loss, the per-row terms of every row and dW at 16 vocabulary rows; and
    properties that hold at any size: the loss is the mean of the per-row
    objective, masked dH rows are zero, and the two gradients satisfy
    sum_t <dH_t, h_t> = sum_v <dW_v, W_v> (both equal (1/N_v) sum of
    dS * Z over the kept dlogits, reached through different GEMMs).
The fp16 workload starts at loss scale 2^15 and halves while found_inf is set.
"""
import os

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
GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


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


def gradient_pairing(dw, scale):
    """(sum_t <dH_t, h_t>, sum_v <dW_v, W_v>, sqrt(sum_tk (dH_tk h_tk)^2)) in fp64, in row blocks."""
    t_h, t_w, s2 = 0.0, 0.0, 0.0
    for r0 in range(0, dw.dH.shape[0], 8192):
        prod = dw.dH[r0:r0 + 8192].double() * dw.h_pol[r0:r0 + 8192].double()
        t_h += float(prod.sum().item())
        s2 += float((prod * prod).sum().item())
    for v0 in range(0, dw.dW.shape[0], 8192):
        t_w += float((dw.dW[v0:v0 + 8192].double() * dw.W[v0:v0 + 8192].double()).sum().item())
    return t_h / scale, t_w / scale, np.sqrt(s2) / scale


def light_results(dw, rows, scale=1.0):
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
        pairing=gradient_pairing(dw, scale),
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


def assert_pairing(pairing):
    """Both sides are (1/N_v) sum dS * Z over the same stored 16-bit dlogits; they
    differ by the rounding of dH to 16 bits (relative error <= 2^-8 per
    element, of random sign), whose sum over N_v * d products has a standard
    deviation near 2^-8 / sqrt(3) * sqrt(sum (dH h)^2).  The bound is ten times
    2^-8 * sqrt(sum (dH h)^2), about 17 standard deviations; a dW that misses
    one chunk of rows, or a dH with a wrong row, moves the difference by several
    times the bound."""
    t_h, t_w, s2 = pairing
    assert s2 > 0
    assert abs(t_h - t_w) <= 10 * 2.0 ** -8 * s2, pairing


_submask_expected = {}


def submask(big):
    """The 400-row sub-mask of a workload and the oracle's values for it (computed once)."""
    cfg = big.cfg
    if cfg.name not in _submask_expected:
        rng = np.random.default_rng(17)
        full = oracle.build_mask(big.lengths, cfg.L)
        live = list(np.flatnonzero(big.lengths >= 270))
        mask = np.zeros(cfg.N, np.uint8)
        for run in (1, 9, 130, 260):
            i = int(rng.choice(live))
            live.remove(i)
            j = int(rng.integers(0, big.lengths[i] - run + 1))
            mask[i * cfg.L + j: i * cfg.L + j + run] = 1
        assert np.all(full[mask == 1] == 1) and int(mask.sum()) == 400
        _submask_expected.clear()
        _submask_expected[cfg.name] = (mask, oracle.expected(big, mask=mask))
    return _submask_expected[cfg.name]


@pytest.mark.parametrize("chunk_rows", [0, 128])
def test_submask_full_shape(big, chunk_rows):
    cfg = big.cfg
    mask, exp = submask(big)
    dw = DeviceWorkload(big, mask=mask, chunk_rows=chunk_rows)
    scale = run_scaled(dw, cfg)
    rows = np.flatnonzero(mask)
    res = light_results(dw, rows, scale)
    del dw
    torch.cuda.empty_cache()
    assert_fwd_parity(res, exp)
    assert res["dH_masked_zero"] and res["dH_finite"]
    err = np.abs(res["dH_rows"] / scale - exp["dH"]).max()
    assert err <= 2e-2 * np.abs(exp["dH"]).max(), ("dH", err)
    compare_dW(res["dW"], exp["dW"], scale)
    assert_pairing(res["pairing"])


def load_golden(cfg):
    path = os.path.join(GOLDEN, f"fullmask_{cfg.name}.npz")
    if not os.path.exists(path):
        return None
    g = np.load(path)
    assert str(g["workload"]) == cfg.name and int(g["seed"]) == 0
    return g


def _completion_golden_workloads():
    """Workloads for which tests/golden holds single-completion values (completion<I>_<workload>.npz)."""
    import glob
    names = {os.path.basename(f)[:-4].split("_", 1)[1] for f in glob.glob(os.path.join(GOLDEN, "completion*_*.npz"))}
    return [n for n in BIG if n in names]


@pytest.mark.parametrize("big", _completion_golden_workloads(), indirect=True)
def test_single_completion_against_golden(big):
    """The full-size shape in the benchmark's launch configuration, masked to one completion whose rows fill
    several backward chunks (default height), against the oracle's values for every row, where
    tests/golden holds them (completion<I>_<workload>.npz, written by make_fullmask_golden.py --completion I)."""
    import glob
    cfg = big.cfg
    files = sorted(glob.glob(os.path.join(GOLDEN, f"completion*_{cfg.name}.npz")))
    import sys
    sys.path.insert(0, GOLDEN)
    from make_fullmask_golden import completion_mask, fingerprint
    g = np.load(files[0])
    assert str(g["workload"]) == cfg.name and int(g["seed"]) == 0
    assert fingerprint(big) == str(g["fingerprint"]), "regenerated inputs differ from the golden file's"
    mask = completion_mask(cfg, big.lengths, int(g["completion"]))
    rows = oracle.valid_rows(mask)
    assert np.array_equal(rows, g["rows"]) and rows.size == int(g["n_valid"])
    dw = DeviceWorkload(big, mask=mask)
    assert rows.size > 2 * rg_chunk_rows(dw)                 # at least two full chunks and a partial one
    scale = run_scaled(dw, cfg)
    sample = rows[np.random.default_rng(29).choice(rows.size, size=8, replace=False)]
    res = light_results(dw, np.sort(sample), scale)
    vr = torch.from_numpy(g["vrows"].astype(np.int64)).cuda()
    dW_rows = dw.dW.index_select(0, vr).cpu().numpy().astype(np.float64) / scale
    del dw
    torch.cuda.empty_cache()
    assert res["status"] == 0
    g_loss = float(g["loss"])
    assert abs(res["loss"] - g_loss) <= 1e-3 * abs(g_loss), (res["loss"], g_loss)
    rs = res["row_stats"][rows]
    for col, key in ((0, "lse_pol"), (1, "lse_ref"), (2, "q"), (3, "p")):
        ref = g[key].astype(np.float64)
        assert np.all(np.abs(rs[:, col] - ref) <= 1e-3 * np.maximum(1.0, np.abs(ref))), key
    pen = g["pen"].astype(np.float64)
    assert np.all(np.abs(rs[:, 4] - pen) <= 1e-5 + 1e-2 * np.abs(pen))
    ref_dW = g["dW_rows"].astype(np.float64)
    assert np.abs(dW_rows - ref_dW).max() <= 2e-2 * np.abs(ref_dW).max()
    exp = oracle.expected(big, mask=mask, eval_rows=np.sort(sample), want_dW=False)
    assert np.abs(res["dH_rows"] / scale - exp["dH"]).max() <= 2e-2 * np.abs(exp["dH"]).max()
    assert res["dH_masked_zero"] and res["dH_finite"]
    assert_pairing(res["pairing"])


def rg_chunk_rows(dw):
    import rl_fine_tuning_gb300 as rg
    return rg.grpo_chunk_rows(dw.shape)


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
    golden = load_golden(cfg)
    if golden is not None:
        import sys
        sys.path.insert(0, GOLDEN)
        from make_fullmask_golden import fingerprint
        assert fingerprint(big) == str(golden["fingerprint"]), "regenerated inputs differ from the golden file's"
    dw = DeviceWorkload(big)
    scale = run_scaled(dw, cfg)
    res = light_results(dw, sample, scale)
    if golden is not None:
        vr = torch.from_numpy(golden["vrows"].astype(np.int64)).cuda()
        res["dW_golden_rows"] = dw.dW.index_select(0, vr).cpu().numpy().astype(np.float64)
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
    assert res["loss"] - a_part >= 0
    if golden is not None:
        # the oracle's full-mask values: the loss, every row's terms, dW at sampled vocabulary rows
        assert int(golden["n_valid"]) == rows.size
        assert np.array_equal(golden["rows"], rows)
        g_loss = float(golden["loss"])
        assert abs(res["loss"] - g_loss) <= 1e-3 * abs(g_loss), (res["loss"], g_loss)
        kl_gpu = (res["loss"] - a_part) / cfg.beta
        assert abs(kl_gpu - float(golden["pen_mean"])) <= 2e-2 * float(golden["pen_mean"])
        rs = res["row_stats"][rows]
        for col, key in ((0, "lse_pol"), (1, "lse_ref"), (2, "q"), (3, "p")):
            ref = golden[key].astype(np.float64)
            assert np.all(np.abs(rs[:, col] - ref) <= 1e-3 * np.maximum(1.0, np.abs(ref))), key
        pen = golden["pen"].astype(np.float64)
        assert np.all(np.abs(rs[:, 4] - pen) <= 1e-5 + 1e-2 * np.abs(pen))
        ref_dW = golden["dW_rows"].astype(np.float64)
        err = np.abs(res["dW_golden_rows"] / scale - ref_dW).max()
        assert err <= 2e-2 * np.abs(ref_dW).max(), ("dW", err)
    else:
        # the KL part of the loss is beta times a mean KL of the size the sampled rows show
        kl_ref_mean = float(np.mean(exp["terms"]["pen"]))
        kl_gpu_mean = (res["loss"] - a_part) / cfg.beta
        assert kl_ref_mean / 4 <= kl_gpu_mean <= 4 * kl_ref_mean + 1e-6
    # masked rows of dH are exactly zero; the two gradients pair up
    assert np.all(np.isfinite(res["dW"])) and res["dH_finite"]
    assert res["dH_masked_zero"]
    assert_pairing(res["pairing"])
