"""GPU path vs the fp64 oracle, element by element, through the C ABI.

Tolerances (floating point): loss relative error <= 1e-3; dH and dW max-abs
error <= 2e-2 * max|reference|; per-row lse/q/p abs error <= 1e-3 * max(1,
|reference|).  Integer outputs (advantage bits, mask, row index) are exact.
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
from gpu_harness import DeviceWorkload, shape_for  # noqa: E402

LOSS_RTOL = 1e-3
GRAD_TOL = 2e-2
STAT_TOL = 1e-3


def assert_fwd_parity(res, exp):
    assert res["status"] == 0, rg.grpo_status_string(res["status"])
    rel = abs(res["loss"] - exp["loss"]) / max(abs(exp["loss"]), 1e-30)
    assert rel <= LOSS_RTOL, (res["loss"], exp["loss"], rel)
    rs = res["row_stats"][exp["eval_rows"]]
    for col, key in ((0, "lse_pol"), (1, "lse_ref"), (2, "q"), (3, "p")):
        ref = exp["terms"][key]
        err = np.abs(rs[:, col] - ref)
        lim = STAT_TOL * np.maximum(1.0, np.abs(ref))
        assert np.all(err <= lim), (key, float(err.max()), int(np.argmax(err - lim)))
    kerr = np.abs(rs[:, 4] - exp["terms"]["pen"])
    assert np.all(kerr <= 1e-5 + 1e-2 * np.abs(exp["terms"]["pen"])), float(kerr.max())
    masked = np.flatnonzero(exp["mask"] == 0)
    assert np.all(res["row_stats"][masked] == 0)


def assert_grad_parity(res, exp, loss_scale=1.0, check_dw=True):
    dH = res["dH"] / loss_scale
    ref = exp["dH"]
    rows = exp["eval_rows"]
    err = np.abs(dH[rows] - ref).max()
    assert err <= GRAD_TOL * np.abs(ref).max(), ("dH", err, np.abs(ref).max())
    masked = np.flatnonzero(exp["mask"] == 0)
    assert np.all(res["dH"][masked] == 0), "masked rows of dH must be exactly 0"
    if check_dw:
        dW = res["dW"] / loss_scale
        refw = exp["dW"]
        errw = np.abs(dW - refw).max()
        assert errw <= GRAD_TOL * np.abs(refw).max(), ("dW", errw, np.abs(refw).max())


# ------------------------------------------------------------------ integer paths

def test_advantages_bit_exact():
    rng = np.random.default_rng(0)
    for G, n_groups in ((1, 3), (2, 5), (4, 1), (8, 1), (8, 37), (16, 4), (64, 2)):
        r = (rng.integers(0, 2, G * n_groups) + 0.1 * rng.normal(size=G * n_groups)).astype(np.float32)
        for unb in (True, False):
            exp = oracle.group_advantages(r, n_groups, G, 1e-4, unb)
            out = torch.empty(G * n_groups, dtype=torch.float32, device="cuda")
            rg.grpo_group_advantages(torch.from_numpy(r).cuda(), n_groups, G, 1e-4, unb, out)
            torch.cuda.synchronize()
            assert np.array_equal(out.cpu().numpy().view(np.uint32), exp.view(np.uint32)), (G, n_groups, unb)


@pytest.mark.parametrize("case", ["prefix", "random", "empty", "full", "alternating", "long"])
def test_mask_and_valid_rows_bit_exact(case):
    rng = np.random.default_rng(1)
    G, L = 8, 1000
    if case == "long":
        G, L = 8, 20000
    lengths = rng.integers(0, L + 1, G).astype(np.int32)
    shape = rg.make_shape(1, G, L, 64, 128)
    N = G * L
    if case == "prefix" or case == "long":
        exp_mask = oracle.build_mask(lengths, L)
        d_mask = torch.empty(N, dtype=torch.uint8, device="cuda")
        rg.grpo_build_mask(torch.from_numpy(lengths).cuda(), shape, d_mask)
        torch.cuda.synchronize()
        assert np.array_equal(d_mask.cpu().numpy(), exp_mask)
        mask = exp_mask
    elif case == "random":
        mask = (rng.random(N) < 0.37).astype(np.uint8)
    elif case == "empty":
        mask = np.zeros(N, np.uint8)
    elif case == "full":
        mask = np.ones(N, np.uint8)
    else:
        mask = (np.arange(N) % 2).astype(np.uint8)
    exp_rows = oracle.valid_rows(mask)
    ws = torch.empty(rg.grpo_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    rows = torch.full((N,), -7, dtype=torch.int32, device="cuda")
    nv = torch.zeros(1, dtype=torch.int32, device="cuda")
    rg.grpo_valid_rows(torch.from_numpy(mask).cuda(), shape, rows, nv, ws)
    torch.cuda.synchronize()
    n = int(nv.item())
    assert n == exp_rows.size
    assert np.array_equal(rows.cpu().numpy()[:n], exp_rows)


# ------------------------------------------------------------------ fused loss

def _run(cfg, seed=0, mask=None, chunk_rows=0, loss_scale=1.0, fwd_only=False, eval_rows=None, vrows=None,
         objective=0, loss_mode=0, std_unbiased=True):
    wl = synth.generate(cfg, seed=seed)
    dw = DeviceWorkload(wl, mask=mask, chunk_rows=chunk_rows, objective=objective, loss_mode=loss_mode,
                        std_unbiased=std_unbiased)
    (dw.fwd() if fwd_only else dw.fwd_bwd(loss_scale))
    res = dw.results()
    exp = oracle.expected(wl, mask=res["mask"], eval_rows=eval_rows, vrows=vrows,
                          want_dH=not fwd_only, want_dW=not fwd_only, objective=objective,
                          loss_mode=loss_mode, std_unbiased=std_unbiased)
    assert np.array_equal(res["adv"].view(np.uint32), exp["adv"].view(np.uint32))
    return wl, dw, res, exp


def test_fwd_tiny():
    _, _, res, exp = _run(synth.CONFIGS["tiny"], fwd_only=True)
    assert_fwd_parity(res, exp)


def test_fwd_bwd_tiny():
    _, _, res, exp = _run(synth.CONFIGS["tiny"])
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)


def test_fwd_bwd_ragged_multi_tile_multi_chunk():
    # V not a multiple of the 256-wide vocabulary tile nor of 64; d spans a partial 256 tile;
    # rows span several 128-row tiles per completion; several backward chunks.
    cfg = synth.make_config("tiny", G=3, L=333, d=320, V=1000, len_lo=1, len_hi=333)
    _, _, res, exp = _run(cfg, seed=3, chunk_rows=256)
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)


@pytest.mark.parametrize("chunk_rows", [128, 384, 640, 1152])
def test_chunk_heights_with_odd_tile_counts(chunk_rows):
    # 1, 3, 5 and 9 tiles per chunk: dH's last SM pair gets a phantom tile, and the
    # last chunk is partial (N_valid is not a multiple of the chunk height)
    cfg = synth.make_config("tiny", G=4, L=700, d=192, V=1500, len_lo=100, len_hi=700)
    _, dw, res, exp = _run(cfg, seed=13, chunk_rows=chunk_rows)
    assert rg.grpo_chunk_rows(dw.shape) == chunk_rows
    assert int(exp["mask"].sum()) % chunk_rows != 0
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_wide_dh_units(dtype):
    # 76-tile chunks with d = 768: 38 tile pairs x 2 wide d tiles of 512 columns divide over the 76 SM
    # pairs, so dH runs in 512-column units, the second one half past d; two chunks, the second partial
    cfg = synth.make_config("tiny", dtype=dtype, G=4, L=4096, d=768, V=1000, len_lo=1500, len_hi=4096)
    _, dw, res, exp = _run(cfg, seed=31, chunk_rows=76 * 128, loss_scale=256.0 if dtype == "fp16" else 1.0)
    assert exp["n_valid"] > 76 * 128
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp, loss_scale=256.0 if dtype == "fp16" else 1.0)


def test_fwd_bwd_scattered_mask():
    cfg = synth.make_config("tiny", G=2, L=200, d=128, V=777)
    rng = np.random.default_rng(5)
    mask = (rng.random(cfg.N) < 0.45).astype(np.uint8)
    _, _, res, exp = _run(cfg, seed=5, mask=mask, chunk_rows=128)
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)


@pytest.mark.parametrize("over", [
    dict(V=1),                                               # one vocabulary entry: softmax is 1, dS is 0
    dict(d=64, V=200),                                       # smallest d, one partial vocabulary tile
    dict(G=1, sigma_ref=0.3),                                # one completion: A = 0, only the KL term acts
    dict(G=2, L=100, d=64, V=257 * 256, len_lo=40, len_hi=100),   # 257 vocabulary tiles: no even split exists
    dict(G=2, L=160, d=8192, V=600, len_lo=60, len_hi=160),      # d of a 70B-class head: 32 d tiles, K = 128 stages
    dict(w_sigma=2.0),                                       # logits up to ~110: near one-hot softmax
    dict(w_sigma=6.0),                                       # logits up to ~330, p - q of order 10
])
def test_degenerate_shapes(over):
    cfg = synth.make_config("tiny", **over)
    _, _, res, exp = _run(cfg, seed=11)
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)
    if cfg.V == 1:
        # lse = z, q = p = 0, and every dlogit is s*g*(1 - 1) = 0: the gradients are exactly zero
        rows = exp["eval_rows"]
        assert np.all(res["row_stats"][rows, 2:5] == 0)
        assert np.all(res["dH"] == 0) and np.all(res["dW"] == 0)
    if cfg.G == 1:
        assert np.all(res["adv"] == 0)


def test_kl_stress():
    cfg = synth.make_config("tiny", sigma_ref=0.5)
    _, _, res, exp = _run(cfg, seed=7)
    # the KL term now moves the loss and the gradient
    assert np.abs(exp["terms"]["p"] - exp["terms"]["q"]).max() > 0.1
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)


def test_fp16_scaled_gradients():
    cfg = synth.make_config("tiny", dtype="fp16", d=192, V=900, sigma_ref=0.05)
    _, _, res, exp = _run(cfg, seed=9, loss_scale=256.0)
    assert res["found_inf"] == 0
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp, loss_scale=256.0)


def test_fp16_overflow_sets_found_inf_and_halving_recovers():
    cfg = synth.make_config("tiny", dtype="fp16")
    wl = synth.generate(cfg, seed=11)
    dw = DeviceWorkload(wl)
    scale = 2.0 ** 40
    dw.fwd_bwd(scale)
    assert int(dw.found_inf.item()) == 1
    halvings = 0
    while int(dw.found_inf.item()) == 1:
        scale /= 2
        halvings += 1
        assert halvings < 64
        dw.fwd_bwd(scale)
    res = dw.results()
    exp = oracle.expected(wl, mask=res["mask"])
    assert scale <= 2.0 ** 16
    assert_grad_parity(res, exp, loss_scale=scale)


def test_deterministic_and_fwd_matches_fwd_bwd():
    cfg = synth.make_config("tiny", G=4, L=300, d=256, V=3000)
    wl = synth.generate(cfg, seed=13)
    dw = DeviceWorkload(wl, chunk_rows=256)
    dw.fwd()
    loss_fwd = dw.loss.clone()
    stats_fwd = dw.row_stats.clone()
    dw.fwd()
    assert torch.equal(loss_fwd.view(torch.int32), dw.loss.view(torch.int32))
    assert torch.equal(stats_fwd, dw.row_stats)
    dw.fwd_bwd()
    a = {k: v.clone() for k, v in (("loss", dw.loss), ("dH", dw.dH), ("dW", dw.dW), ("rs", dw.row_stats))}
    dw.fwd_bwd()
    # the forward-only entry point runs the same chunked kernels: equal bit for bit
    assert torch.equal(loss_fwd.view(torch.int32), a["loss"].view(torch.int32))
    assert torch.equal(stats_fwd, a["rs"])
    # every entry point is bitwise reproducible
    assert torch.equal(a["loss"].view(torch.int32), dw.loss.view(torch.int32))
    assert torch.equal(a["rs"], dw.row_stats)
    assert torch.equal(a["dH"].view(torch.int16), dw.dH.view(torch.int16))
    assert torch.equal(a["dW"].view(torch.int32), dw.dW.view(torch.int32))


@pytest.mark.parametrize("objective", ["grpo", "no_detach", "reverse_kl_q", "forward_kl"])
@pytest.mark.parametrize("loss_mode", [0, 1])
def test_objective_variants_and_means(objective, loss_mode):
    # several prompt groups, one fully masked completion, KL large enough to matter
    cfg = synth.make_config("tiny", n_groups=3, G=4, L=150, d=192, V=1000, len_lo=1, len_hi=150,
                            n_zero_seq=1, sigma_ref=0.3)
    _, _, res, exp = _run(cfg, seed=31, chunk_rows=256, objective=objective, loss_mode=loss_mode)
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)


@pytest.mark.parametrize("fwd_only", [True, False])
def test_population_std_and_sequence_mean_forward(fwd_only):
    cfg = synth.make_config("tiny", n_groups=2, G=8, L=96, d=128, V=2048, len_lo=0, len_hi=96)
    _, _, res, exp = _run(cfg, seed=37, std_unbiased=False, loss_mode=1, fwd_only=fwd_only)
    assert_fwd_parity(res, exp)
    if not fwd_only:
        assert_grad_parity(res, exp)


def test_all_rows_masked():
    cfg = synth.CONFIGS["tiny"]
    wl = synth.generate(cfg, seed=2)
    dw = DeviceWorkload(wl, mask=np.zeros(cfg.N, np.uint8))
    dw.dH.fill_(7)
    dw.dW.fill_(7)
    dw.fwd_bwd()
    res = dw.results()
    assert res["status"] == 0 and res["loss"] == 0.0 and res["found_inf"] == 0
    assert np.all(res["dH"] == 0) and np.all(res["dW"] == 0)


def test_token_out_of_range_reports_status():
    cfg = synth.CONFIGS["tiny"]
    wl = synth.generate(cfg, seed=2)
    wl.tokens[3] = cfg.V + 5          # row 3 is inside the first completion (lengths >= 16)
    dw = DeviceWorkload(wl)
    dw.fwd()
    assert int(dw.status.item()) == 2          # bad shape or token id


def test_host_validation_errors():
    cfg = synth.CONFIGS["tiny"]
    wl = synth.generate(cfg, seed=2)
    dw = DeviceWorkload(wl)
    small = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(rg.GrpoError) as e:
        rg.grpo_loss_fwd(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, small, dw.loss, None,
                         dw.status)
    assert e.value.code == 3
    bad = shape_for(cfg)
    bad.d = 100
    with pytest.raises(rg.GrpoError) as e:
        rg.grpo_loss_fwd(dw.h_pol, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, bad, dw.ws, dw.loss, None, dw.status)
    assert e.value.code == 2
    with pytest.raises(rg.GrpoError) as e:
        rg.grpo_loss_fwd(dw.h_pol.data_ptr() + 2, dw.h_ref, dw.W, dw.tokens, dw.mask, dw.adv, dw.shape, dw.ws,
                         dw.loss, None, dw.status)
    assert e.value.code == 1


def test_bounded_wait_times_out_and_context_stays_usable():
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    waited = torch.zeros(1, dtype=torch.int64, device="cuda")
    rg.grpo_selftest_wait_timeout(status, waited)
    torch.cuda.synchronize()
    assert int(status.item()) == 6                      # GRPO_ERR_TIMEOUT
    assert 0.9e9 <= int(waited.item()) <= 5e9           # about one second, then it gave up
    # the context still runs the real path
    _, _, res, exp = _run(synth.CONFIGS["tiny"])
    assert_fwd_parity(res, exp)
    assert_grad_parity(res, exp)
