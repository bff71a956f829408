"""The 8-bit entry points (E4M3 and E5M2 inputs) against the fp64 oracle on
the same 8-bit inputs: the oracle reads every code times its tensor's scale
exactly in fp64.  The forward (grpo_loss_fwd_fp8) meets the bar of the 16-bit
forward.  The forward+backward (grpo_loss_fwd_bwd_fp8) is held to the 16-bit
tolerances too (loss relative 1e-3, dH and dW 2e-2 x max|ref|) against the
exact gradient of the decoded inputs: its 8-bit dlogits carry only the
softmax part of each row, the one-hot part being added exactly."""
import numpy as np
import pytest

import oracle
import synth

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import rl_fine_tuning_gb300 as rg  # noqa: E402
from test_gpu_parity import assert_fwd_parity  # noqa: E402


def run_fp8(wl8, mask=None, eval_rows=None):
    cfg = wl8.cfg
    s_pol, s_ref, s_w = wl8.extra["scales"]
    dtype = rg.E5M2 if wl8.extra.get("fp8") == "e5m2" else rg.E4M3
    shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V, dtype, beta=cfg.beta, eps=cfg.eps)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    h_pol, h_ref, W = dev(wl8.h_pol), dev(wl8.h_ref), dev(wl8.W)
    tokens, lengths, rewards = dev(wl8.tokens), dev(wl8.lengths), dev(wl8.rewards)
    adv = torch.empty(cfg.n_seq, dtype=torch.float32, device="cuda")
    rg.grpo_group_advantages(rewards, cfg.n_groups, cfg.G, cfg.eps, True, adv)
    if mask is None:
        m = torch.empty(cfg.N, dtype=torch.uint8, device="cuda")
        rg.grpo_build_mask(lengths, shape, m)
    else:
        m = dev(mask.astype(np.uint8))
    ws = torch.empty(rg.grpo_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    stats = torch.zeros((cfg.N, 5), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    rg.grpo_loss_fwd_fp8(h_pol, h_ref, W, s_pol, s_ref, s_w, tokens, m, adv, shape, ws, loss, stats, status)
    torch.cuda.synchronize()
    res = dict(loss=float(loss.item()), status=int(status.item()), row_stats=stats.cpu().numpy().astype(np.float64),
               adv=adv.cpu().numpy(), mask=m.cpu().numpy())
    exp = oracle.expected(oracle.dequantized_workload(wl8), mask=res["mask"], eval_rows=eval_rows,
                          want_dH=False, want_dW=False)
    return res, exp


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("over", [dict(), dict(G=4, L=500, d=384, V=3000, len_lo=1, len_hi=500),
                                  dict(G=2, L=300, d=256, V=777, sigma_ref=0.4)])
def test_fp8_forward_parity(over, fmt):
    cfg = synth.make_config("tiny", **over)
    res, exp = run_fp8(synth.generate_fp8(cfg, seed=41, fmt=fmt))
    assert np.array_equal(res["adv"].view(np.uint32), exp["adv"].view(np.uint32))
    assert_fwd_parity(res, exp)


def test_fp8_rejects_bad_arguments():
    cfg = synth.make_config("tiny", d=192)
    wl8 = synth.generate_e4m3(synth.make_config("tiny"), seed=1)
    with pytest.raises(rg.GrpoError) as e:            # d not a multiple of 128
        shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, 192, cfg.V, rg.E4M3)
        t = torch.zeros(16, dtype=torch.int32, device="cuda")
        rg.grpo_loss_fwd_fp8(t, t, t, 1.0, 1.0, 1.0, t, t, t, shape, torch.zeros(64, dtype=torch.uint8, device="cuda"),
                             t, None, t)
    assert e.value.code == 2
    with pytest.raises(rg.GrpoError) as e:            # 16-bit shape handed to the 8-bit entry point
        shape = rg.make_shape(1, 4, 64, 128, 1024, rg.BF16)
        t = torch.zeros(16, dtype=torch.int32, device="cuda")
        rg.grpo_loss_fwd_fp8(t, t, t, 1.0, 1.0, 1.0, t, t, t, shape, torch.zeros(64, dtype=torch.uint8, device="cuda"),
                             t, None, t)
    assert e.value.code == 5
    del wl8


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_forward_full_size_sampled_rows(fmt):
    cfg = synth.CONFIGS["llama-3.1-8b-head"]
    wl8 = synth.generate_fp8(cfg, seed=0, fmt=fmt)
    mask = oracle.build_mask(wl8.lengths, cfg.L)
    rows = oracle.valid_rows(mask)
    rng = np.random.default_rng(5)
    sample = np.sort(rng.choice(rows, size=12, replace=False)).astype(np.int32)
    res, exp = run_fp8(wl8, eval_rows=sample)
    assert res["status"] == 0
    rs = res["row_stats"][sample]
    for col, key in ((0, "lse_pol"), (1, "lse_ref"), (2, "q"), (3, "p")):
        ref = exp["terms"][key]
        assert np.all(np.abs(rs[:, col] - ref) <= 1e-3 * np.maximum(1.0, np.abs(ref))), key
    A = exp["adv"][rows // cfg.L].astype(np.float64)
    ell = -A + cfg.beta * res["row_stats"][rows, 4]
    assert abs(res["loss"] - ell.mean()) <= 1e-5 * max(1e-3, abs(ell.mean()))


def run_fp8_bwd(wl8, mask=None, chunk_rows=0, want_expected=True, objective=0, loss_mode=0):
    cfg = wl8.cfg
    s_pol, s_ref, s_w = wl8.extra["scales"]
    dtype = rg.E5M2 if wl8.extra.get("fp8") == "e5m2" else rg.E4M3
    shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V, dtype, beta=cfg.beta, eps=cfg.eps,
                          chunk_rows=chunk_rows, objective=objective, loss_mode=loss_mode)
    dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()  # noqa: E731
    h_pol, h_ref, W = dev(wl8.h_pol), dev(wl8.h_ref), dev(wl8.W)
    tokens, lengths, rewards = dev(wl8.tokens), dev(wl8.lengths), dev(wl8.rewards)
    adv = torch.empty(cfg.n_seq, dtype=torch.float32, device="cuda")
    rg.grpo_group_advantages(rewards, cfg.n_groups, cfg.G, cfg.eps, True, adv)
    if mask is None:
        m = torch.empty(cfg.N, dtype=torch.uint8, device="cuda")
        rg.grpo_build_mask(lengths, shape, m)
    else:
        m = dev(mask.astype(np.uint8))
    ws = torch.empty(rg.grpo_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
    loss = torch.zeros(1, dtype=torch.float32, device="cuda")
    stats = torch.zeros((cfg.N, 5), dtype=torch.float32, device="cuda")
    status = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    # sentinels: every element must be written (masked dH rows with 0)
    dH = torch.full((cfg.N, cfg.d), 7.0, dtype=torch.bfloat16, device="cuda")
    dW = torch.full((cfg.V, cfg.d), 7.0, dtype=torch.float32, device="cuda")
    rg.grpo_loss_fwd_bwd_fp8(h_pol, h_ref, W, s_pol, s_ref, s_w, tokens, m, adv, shape, ws, loss, dH, dW, stats,
                             status)
    torch.cuda.synchronize()
    res = dict(loss=float(loss.item()), status=int(status.item()), row_stats=stats.cpu().numpy().astype(np.float64),
               adv=adv.cpu().numpy(), mask=m.cpu().numpy(), dH=dH.float().cpu().numpy().astype(np.float64),
               dW=dW.cpu().numpy().astype(np.float64))
    exp = (oracle.expected(oracle.dequantized_workload(wl8), mask=res["mask"], objective=objective,
                           loss_mode=loss_mode) if want_expected else None)
    return res, exp


def assert_fp8_grad_parity(res, exp):
    assert_fwd_parity(res, exp)
    rows = exp["eval_rows"]
    err_h = np.abs(res["dH"][rows] - exp["dH"]).max()
    assert err_h <= 2e-2 * np.abs(exp["dH"]).max(), ("dH", err_h, np.abs(exp["dH"]).max())
    masked = np.flatnonzero(exp["mask"] == 0)
    assert np.all(res["dH"][masked] == 0)
    err_w = np.abs(res["dW"] - exp["dW"]).max()
    assert err_w <= 2e-2 * np.abs(exp["dW"]).max(), ("dW", err_w, np.abs(exp["dW"]).max())
    rel_h, rel_w = err_h / np.abs(exp["dH"]).max(), err_w / np.abs(exp["dW"]).max()
    print(f"8-bit gradients: max|dH - ref| = {rel_h:.2e} max|ref|, max|dW - ref| = {rel_w:.2e} max|ref|")
    return rel_h, rel_w


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
@pytest.mark.parametrize("over,chunk_rows", [
    (dict(), 0),
    (dict(G=4, L=500, d=384, V=3000, len_lo=1, len_hi=500), 256),          # ragged V, several chunks
    (dict(G=4, L=256, d=256, V=200, len_lo=64, len_hi=256), 128),          # many rows per token in a chunk
    (dict(G=2, L=300, d=256, V=777, sigma_ref=0.4), 0),                    # a KL large enough to matter
])
def test_fp8_forward_backward_parity(over, chunk_rows, fmt):
    cfg = synth.make_config("tiny", **over)
    res, exp = run_fp8_bwd(synth.generate_fp8(cfg, seed=43, fmt=fmt), chunk_rows=chunk_rows)
    assert np.array_equal(res["adv"].view(np.uint32), exp["adv"].view(np.uint32))
    assert_fp8_grad_parity(res, exp)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_forward_backward_full_shape_submask(fmt):
    # the Llama-3.1-8B head shape with 400 masked-in rows in four runs, 128-row chunks
    cfg = synth.CONFIGS["llama-3.1-8b-head"]
    wl8 = synth.generate_fp8(cfg, seed=0, fmt=fmt)
    rng = np.random.default_rng(17)
    live = list(np.flatnonzero(wl8.lengths >= 270))
    mask = np.zeros(cfg.N, np.uint8)
    for run in (1, 9, 130, 260):
        i = int(rng.choice(live))
        live.remove(i)
        j = int(rng.integers(0, wl8.lengths[i] - run + 1))
        mask[i * cfg.L + j: i * cfg.L + j + run] = 1
    res, exp = run_fp8_bwd(wl8, mask=mask, chunk_rows=128)
    assert_fp8_grad_parity(res, exp)


def test_fp8_backward_forward_loss_equals_the_forward_entry_point():
    cfg = synth.make_config("tiny", G=4, L=300, d=256, V=1500, len_lo=1, len_hi=300)
    wl8 = synth.generate_fp8(cfg, seed=44, fmt="e4m3")
    res_b, _ = run_fp8_bwd(wl8)
    res_f, _ = run_fp8(wl8)
    assert res_b["status"] == 0 and res_f["status"] == 0
    assert res_b["loss"] == res_f["loss"]
    assert np.array_equal(res_b["row_stats"], res_f["row_stats"])


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_backward_edge_cases(fmt):
    # every row masked: loss 0, dH and dW exactly 0
    cfg = synth.make_config("tiny", G=2, L=128, d=128, V=1000)
    wl8 = synth.generate_fp8(cfg, seed=45, fmt=fmt)
    res, _ = run_fp8_bwd(wl8, mask=np.zeros(cfg.N, np.uint8))
    assert res["status"] == 0 and res["loss"] == 0.0
    assert np.all(res["dH"] == 0) and np.all(res["dW"] == 0)
    # a one-token vocabulary: softmax = 1, so the dlogits and both gradients are 0.  The one-hot
    # part (added exactly) and the softmax part (from 8-bit codes with fp32 scales) cancel
    # to fp32 rounding: the residue is held to 1e-5 of the one-hot terms' size
    cfg1 = synth.make_config("tiny", G=2, L=64, d=128, V=1)
    wl1 = synth.generate_fp8(cfg1, seed=46, fmt=fmt)
    res, exp = run_fp8_bwd(wl1)
    assert res["status"] == 0
    s_pol, _, s_w = wl1.extra["scales"]
    g_max = np.abs(exp["terms"]["g"]).max()
    w_max = np.abs(oracle.fp8_values(wl1.W, s_w, fmt)).max()
    h_max = np.abs(oracle.fp8_values(wl1.h_pol, s_pol, fmt)).max()
    assert np.abs(res["dH"]).max() <= 1e-5 * g_max * w_max / exp["n_valid"]
    assert np.abs(res["dW"]).max() <= 1e-5 * g_max * h_max       # every row's token is 0: N_v terms of g h / N_v
    assert abs(res["loss"] - exp["loss"]) <= 1e-3 * max(abs(exp["loss"]), 1e-30)


def test_fp8_backward_bad_token_and_reproducibility():
    cfg = synth.make_config("tiny", G=4, L=200, d=256, V=900, len_lo=20, len_hi=200)
    wl8 = synth.generate_fp8(cfg, seed=47, fmt="e4m3")
    a, _ = run_fp8_bwd(wl8, chunk_rows=256)
    b, _ = run_fp8_bwd(wl8, chunk_rows=256)
    assert a["status"] == 0 and b["status"] == 0
    assert a["loss"] == b["loss"] and np.array_equal(a["dH"], b["dH"]) and np.array_equal(a["dW"], b["dW"])
    # a sampled token outside [0, V) on a masked-in row: reported as status 2, nothing read out of bounds
    mask = oracle.build_mask(wl8.lengths, cfg.L)
    bad = int(oracle.valid_rows(mask)[3])
    wl8.tokens = wl8.tokens.copy()
    wl8.tokens[bad] = cfg.V + 5
    res, _ = run_fp8_bwd(wl8, chunk_rows=256, want_expected=False)
    assert res["status"] == 2
    assert np.all(np.isfinite(res["dH"])) and np.all(np.isfinite(res["dW"]))


@pytest.mark.parametrize("objective", ["no_detach", "reverse_kl_q", "forward_kl"])
def test_fp8_backward_objective_variants_and_sequence_mean(objective):
    # three prompt groups, a fully masked completion, a KL large enough to matter, per-completion mean
    cfg = synth.make_config("tiny", n_groups=3, G=4, L=150, d=256, V=1000, len_lo=1, len_hi=150, n_zero_seq=1,
                            sigma_ref=0.3)
    res, exp = run_fp8_bwd(synth.generate_fp8(cfg, seed=48, fmt="e4m3"), chunk_rows=256, objective=objective,
                           loss_mode=1)
    assert_fp8_grad_parity(res, exp)


@pytest.mark.parametrize("fmt", ["e4m3", "e5m2"])
def test_fp8_backward_wide_dh_units(fmt):
    # the default 76-tile chunks with d = 768: 38 tile pairs x 2 wide d tiles of 512 columns divide over
    # the 76 SM pairs, so the 8-bit dH runs in 512-column units, the second one half past d
    cfg = synth.make_config("tiny", G=4, L=4096, d=768, V=1000, len_lo=1500, len_hi=4096)
    res, exp = run_fp8_bwd(synth.generate_fp8(cfg, seed=31, fmt=fmt))
    assert exp["n_valid"] > 76 * 128             # two chunks
    assert_fp8_grad_parity(res, exp)
