"""Pins of the fp64 CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: a value the
pages print, a closed form, an invariant, brute force in higher precision or
an independent library routine.  A plausible slip in the oracle (a dropped
term, a wrong sign or index, a transposed operand) fails at least one.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth

HERE = os.path.dirname(os.path.abspath(__file__))


# --------------------------------------------------------------------------
# memory arithmetic printed on the pages ("Long-context GRPO", section 2)
# --------------------------------------------------------------------------

def test_logits_memory_figures_match_pages():
    g = json.load(open(os.path.join(HERE, "golden", "memory_figures.json")))
    f = g["logits_factors"]
    ctx = 20 * 1024                                   # "20K" read as 20480
    b = f["tensors"] * f["bytes"] * f["generations"] * ctx * f["vocab"]
    assert b == 84_053_852_160
    gib = b / 2**30
    assert round(gib, 1) == g["logits_two_tensors_gb"]          # 78.28 -> 78.3
    assert round(gib / 8, 1) == g["unsloth_extra_gb"]           # one generation: 9.8
    assert round(g["logits_two_tensors_gb"] - g["unsloth_extra_gb"], 1) == g["linear_algorithm_saving_gb"]
    assert g["logits_two_tensors_gb"] / g["unsloth_extra_gb"] >= g["linear_algorithm_reduction_at_least"] - 0.05
    # total VRAM difference = the three savings listed in the same section
    diff = g["total_vram_trl_fa2_gb"] - g["total_vram_unsloth_gb"]
    assert abs(diff - (g["linear_algorithm_saving_gb"] + g["gradient_checkpointing_saving_gb"]
                       + g["vllm_shared_memory_saving_gb"])) < 1e-9
    # a 20000-token reading gives a different figure: the pages used 20480
    assert round(2 * 2 * 8 * 20000 * 128256 / 2**30, 1) != g["logits_two_tensors_gb"]


def test_kv_cache_figure_matches_pages():
    g = json.load(open(os.path.join(HERE, "golden", "memory_figures.json")))
    f = g["kv_cache_factors"]
    b = f["kv"] * f["bytes"] * f["layers"] * 20 * 1024 * f["width"]
    assert b / 2**30 == g["kv_cache_per_batch_gb"]
    assert 8 * b / 2**30 == g["kv_cache_batch8_gb"]


# --------------------------------------------------------------------------
# storage-type widening and the generator's rounding
# --------------------------------------------------------------------------

def test_f16_widening_all_patterns():
    lib = oracle._L()
    bits = np.arange(65536, dtype=np.uint16)
    ref = bits.view(np.float16).astype(np.float64)
    got = np.array([lib.oracle_f16_to_f64(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))
    assert np.array_equal(np.isinf(got), np.isinf(ref))


def test_bf16_widening_all_patterns():
    torch = pytest.importorskip("torch")
    lib = oracle._L()
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([lib.oracle_bf16_to_f64(int(b)) for b in bits])
    fin = np.isfinite(ref)
    assert np.array_equal(got[fin], ref[fin])
    assert np.array_equal(np.isnan(got), np.isnan(ref))


@pytest.mark.filterwarnings("ignore:overflow encountered in cast")
def test_generator_rounding_matches_libraries():
    torch = pytest.importorskip("torch")
    x = synth.normal_f32(7, 11, 200_000, 3.0)
    x = np.concatenate([x, np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 1e-8, 2.0**-25, 2.0**-24,
                                     3 * 2.0**-26, 6.0e-5, -6.1e-5, 1e30, -1e30], np.float32)])
    assert np.array_equal(synth.to_f16_bits(x), x.astype(np.float16).view(np.uint16))
    tb = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(synth.to_bf16_bits(x), tb)


def test_e4m3_decoding_special_values():
    """OCP FP8 E4M3: bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN."""
    lib = oracle._L()
    dec = np.array([lib.oracle_e4m3_to_f64(i) for i in range(256)])
    assert dec[0x38] == 1.0 and dec[0x7E] == 448.0 and dec[0x08] == 2.0 ** -6 and dec[0x01] == 2.0 ** -9
    assert dec[0x07] == 7 * 2.0 ** -9 and dec[0x40] == 2.0 and dec[0x3C] == 1.5
    assert np.isnan(dec[0x7F]) and np.isnan(dec[0xFF])
    assert dec[0x00] == 0.0 and dec[0x80] == 0.0 and np.signbit(dec[0x80])
    assert np.array_equal(dec[0x80:0xFF], -dec[0x00:0x7F])
    assert np.all(np.diff(dec[0x00:0x7F]) > 0)                 # codes are ordered like their values


def test_generator_e4m3_rounding_brute_force():
    """Each code is the nearest e4m3 value to x/scale (ties to an even mantissa), saturating at 448."""
    lib = oracle._L()
    dec = np.array([lib.oracle_e4m3_to_f64(i) for i in range(256)])
    pos = np.arange(0x7F)                                       # finite non-negative codes
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.normal(0, 40, 4000), rng.uniform(-500, 500, 2000), rng.normal(0, 1e-2, 2000),
                        dec[pos] + 0.5 * np.diff(np.append(dec[pos], 480.0))])     # exact midpoints
    x = x.astype(np.float32)
    codes = synth.to_e4m3_bits(x, 1.0)
    for xi, c in zip(x.astype(np.float64), codes):
        a = abs(xi)
        err = np.abs(dec[pos] - min(a, 448.0))
        best = pos[err == err.min()]
        if best.size > 1:
            best = best[(best & 1) == 0]
        assert (c & 0x7F) == best[0], (xi, hex(c), hex(best[0]))
        assert (c >> 7) == (1 if (xi < 0 and (c & 0x7F) != 0) else (c >> 7))
    s = synth.e4m3_scale(x)
    assert np.max(np.abs(oracle.e4m3_values(synth.to_e4m3_bits(x, s), s))) <= 448.0 * s * (1 + 1e-7)


def test_e5m2_decoding_special_values():
    """OCP FP8 E5M2: bias 15, 2 mantissa bits, IEEE-style infinities and NaNs."""
    lib = oracle._L()
    dec = np.array([lib.oracle_e5m2_to_f64(i) for i in range(256)])
    assert dec[0x3C] == 1.0 and dec[0x7B] == 57344.0 and dec[0x04] == 2.0 ** -14 and dec[0x01] == 2.0 ** -16
    assert dec[0x03] == 3 * 2.0 ** -16 and dec[0x40] == 2.0 and dec[0x3E] == 1.5 and dec[0x3F] == 1.75
    assert dec[0x7C] == np.inf and dec[0xFC] == -np.inf
    assert all(np.isnan(dec[c]) for c in (0x7D, 0x7E, 0x7F, 0xFD, 0xFE, 0xFF))
    assert dec[0x00] == 0.0 and np.signbit(dec[0x80])
    assert np.array_equal(dec[0x80:0xFD], -dec[0x00:0x7D])
    assert np.all(np.diff(dec[0x00:0x7D]) > 0)
    # an E5M2 code is the high byte of an IEEE binary16 value: numpy's half decoder agrees on every code
    half = (np.arange(256, dtype=np.uint16) << 8).view(np.float16).astype(np.float64)
    finite = ~np.isnan(half)
    assert np.array_equal(dec[finite], half[finite]) and np.array_equal(np.isnan(dec), ~finite)


def test_generator_e5m2_rounding_brute_force():
    """Each code is the nearest e5m2 value to x/scale (ties to an even mantissa), saturating at 57344."""
    lib = oracle._L()
    dec = np.array([lib.oracle_e5m2_to_f64(i) for i in range(256)])
    pos = np.arange(0x7C)                                       # finite non-negative codes
    rng = np.random.default_rng(4)
    x = np.concatenate([rng.normal(0, 3000, 4000), rng.uniform(-70000, 70000, 2000), rng.normal(0, 1e-4, 2000),
                        dec[pos] + 0.5 * np.diff(np.append(dec[pos], 61440.0))])     # exact midpoints
    x = x.astype(np.float32)
    codes = synth.to_fp8_bits(x, 1.0, "e5m2")
    for xi, c in zip(x.astype(np.float64), codes):
        a = abs(xi)
        err = np.abs(dec[pos] - min(a, 57344.0))
        best = pos[err == err.min()]
        if best.size > 1:
            best = best[(best & 1) == 0]
        assert (c & 0x7F) == best[0], (xi, hex(c), hex(best[0]))
        if xi > 0:
            assert c >> 7 == 0
    s = synth.fp8_scale(x, "e5m2")
    vals = oracle.fp8_values(synth.to_fp8_bits(x, s, "e5m2"), s, "e5m2")
    assert np.all(np.isfinite(vals)) and np.max(np.abs(vals)) <= 57344.0 * s * (1 + 1e-7)


def test_generator_is_counter_based():
    a = synth.normal_f32(0, 1, 1000)
    b = synth.normal_f32(0, 1, 500, offset=500)
    assert np.array_equal(a[500:], b)
    assert abs(a.mean()) < 0.15 and abs(a.std() - 1) < 0.1
    t = synth.uniform_int(0, 4, 100000, 0, 9)
    assert t.min() == 0 and t.max() == 9
    p = synth.permutation(0, 8, 8)
    assert sorted(p.tolist()) == list(range(8))


# --------------------------------------------------------------------------
# group-relative advantages ("Train your own R1 ...", section 3, steps 3-5)
# --------------------------------------------------------------------------

def test_advantages_closed_form_bernoulli():
    r = np.array([0, 1, 0, 1], np.float32)
    a = oracle.group_advantages(r, 1, 4, eps=1e-4)
    # sample std of {0,1,0,1} is sqrt(1/3); standardised scores are +-sqrt(3)/2
    expect = 0.5 / (math.sqrt(1.0 / 3.0) + float(np.float32(1e-4)))
    assert np.allclose(a, [-expect, expect, -expect, expect], rtol=1e-7, atol=0)
    assert abs(abs(a[0]) - math.sqrt(3) / 2) < 2e-4


def test_advantages_invariants_and_numpy():
    rng = np.random.default_rng(0)
    for G in (2, 3, 4, 8, 16):
        r = rng.normal(size=5 * G).astype(np.float32)
        a = oracle.group_advantages(r, 5, G).reshape(5, G)
        rr = r.reshape(5, G).astype(np.float64)
        ref = (rr - rr.mean(1, keepdims=True)) / (rr.std(1, ddof=1, keepdims=True) + float(np.float32(1e-4)))
        assert np.allclose(a, ref.astype(np.float32), rtol=2e-7, atol=1e-7)
        assert np.all(np.abs(a.astype(np.float64).sum(1)) < 1e-5)        # centred
        # population std option matches numpy ddof=0
        ap = oracle.group_advantages(r, 5, G, std_unbiased=False).reshape(5, G)
        refp = (rr - rr.mean(1, keepdims=True)) / (rr.std(1, ddof=0, keepdims=True) + float(np.float32(1e-4)))
        assert np.allclose(ap, refp.astype(np.float32), rtol=2e-7, atol=1e-7)
    # all-equal rewards -> zero advantage; G = 1 -> zero
    assert np.all(oracle.group_advantages(np.full(8, 0.7, np.float32), 1, 8) == 0)
    assert np.all(oracle.group_advantages(np.array([3.0], np.float32), 1, 1) == 0)
    # shift invariance (exact for shifts that keep r - mu exact)
    r = np.array([0, 1, 1, 0, 1, 0, 0, 0], np.float32)
    assert np.array_equal(oracle.group_advantages(r, 1, 8), oracle.group_advantages(r + 2, 1, 8))


# --------------------------------------------------------------------------
# mask and valid-row index
# --------------------------------------------------------------------------

def test_mask_and_rows():
    lens = np.array([0, 3, 5, 1], np.int32)
    m = oracle.build_mask(lens, 5)
    assert m.tolist() == [0, 0, 0, 0, 0, 1, 1, 1, 0, 0, 1, 1, 1, 1, 1, 1, 0, 0, 0, 0]
    assert oracle.valid_rows(m).tolist() == [5, 6, 7, 10, 11, 12, 13, 14, 15]
    assert oracle.valid_rows(np.zeros(7, np.uint8)).size == 0
    rng = np.random.default_rng(1)
    mm = (rng.random(1000) < 0.3).astype(np.uint8)
    assert np.array_equal(oracle.valid_rows(mm), np.flatnonzero(mm))


# --------------------------------------------------------------------------
# logsumexp ("Long-context GRPO", section 4: the logsumexp trick)
# --------------------------------------------------------------------------

def test_logsumexp_against_brute_force():
    mp = pytest.importorskip("mpmath")
    mp.mp.dps = 50
    rng = np.random.default_rng(2)
    for V in (1, 2, 7, 1000):
        z = rng.uniform(-20, 20, V)
        brute = float(mp.log(mp.fsum([mp.exp(mp.mpf(float(v))) for v in z])))
        assert abs(oracle.logsumexp(z) - brute) <= 1e-13 * max(1.0, abs(brute))
        # shift invariance, including shifts that would overflow a naive sum
        assert abs(oracle.logsumexp(z + 800.0) - (brute + 800.0)) <= 1e-12 * (800 + abs(brute))
    assert oracle.logsumexp(np.array([3.25])) == 3.25
    assert oracle.logsumexp(np.zeros(1024)) == pytest.approx(math.log(1024), abs=1e-14)


# --------------------------------------------------------------------------
# per-row terms
# --------------------------------------------------------------------------

def _tiny_problem(seed=0, G=2, L=3, d=4, V=5, w_scale=0.5, ref_noise=0.3, lens=(2, 3)):
    rng = np.random.default_rng(seed)
    N = G * L
    h_pol = rng.normal(size=(N, d))
    h_ref = h_pol + ref_noise * rng.normal(size=(N, d))
    W = w_scale * rng.normal(size=(V, d))
    tokens = rng.integers(0, V, N).astype(np.int32)
    rewards = rng.normal(size=G).astype(np.float32)
    adv = oracle.group_advantages(rewards, 1, G)
    mask = oracle.build_mask(np.array(lens, np.int32), L)
    return h_pol, h_ref, W, tokens, adv, mask, L


def test_row_terms_against_numpy_scipy():
    scipy_special = pytest.importorskip("scipy.special")
    h_pol, h_ref, W, tok, adv, mask, L = _tiny_problem(seed=3, G=3, L=4, d=6, V=9)
    rows = np.arange(h_pol.shape[0], dtype=np.int32)
    t = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows)
    zp = h_pol @ W.T
    zr = h_ref @ W.T
    lp = scipy_special.logsumexp(zp, axis=1)
    lr = scipy_special.logsumexp(zr, axis=1)
    q = zp[rows, tok] - lp
    p = zr[rows, tok] - lr
    A = adv[rows // L].astype(np.float64)
    x = p - q
    assert np.allclose(t["lse_pol"], lp, rtol=0, atol=1e-12)
    assert np.allclose(t["lse_ref"], lr, rtol=0, atol=1e-12)
    assert np.allclose(t["q"], q, atol=1e-12) and np.allclose(t["p"], p, atol=1e-12)
    # KL estimator: e^x - x - 1 >= 0
    assert np.all(t["pen"] >= 0)
    assert np.allclose(t["pen"], np.exp(x) - x - 1, atol=1e-12)
    assert np.allclose(t["ell"], -A + 0.04 * (np.exp(x) - x - 1), atol=1e-12)
    assert np.allclose(t["g"], -A + 0.04 * (1 - np.exp(x)), atol=1e-12)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
def test_16bit_row_loops_read_storage_as_numpy_and_torch_widen_it(dtype):
    # The row loops read 16-bit storage (fp16 through its table of all 65536 patterns).  Given the bit
    # patterns, every row term and gradient must equal, bit for bit, the fp64 path on the values that numpy
    # (fp16) or torch (bf16) widens the same patterns to: same values, same ascending-index sums.
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(12)
    G, L, d, V = 3, 4, 40, 70
    N = G * L
    h = rng.normal(size=(N, d)) * 3.0
    x = {"h_pol": h, "h_ref": h + 0.1 * rng.normal(size=(N, d)), "W": rng.normal(size=(V, d)) * 0.3}
    if dtype == "fp16":
        for k in x:                                      # fp16 subnormals and a large normal value
            x[k][0, :3] = [1e-6, -3e-8, 900.0]
    bits = {}
    for name, v in x.items():
        if dtype == "fp16":
            bits[name] = v.astype(np.float16).view(np.uint16)
        else:
            bits[name] = torch.from_numpy(v.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy() \
                .view(np.uint16)
    if dtype == "fp16":
        val = {k: b.view(np.float16).astype(np.float64) for k, b in bits.items()}
    else:
        val = {k: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
               for k, b in bits.items()}
    tok = rng.integers(0, V, N).astype(np.int32)
    adv = oracle.group_advantages(rng.normal(size=G).astype(np.float32), 1, G)
    rows = np.arange(N, dtype=np.int32)
    t16 = oracle.row_terms(bits["h_pol"], bits["h_ref"], bits["W"], dtype, tok, adv, L, rows)
    t64 = oracle.row_terms(val["h_pol"], val["h_ref"], val["W"], "f64", tok, adv, L, rows)
    for k in t16:
        assert np.all(np.isfinite(t16[k])) and np.array_equal(t16[k], t64[k]), k
    w = oracle.row_weights(rows, L)
    g16 = oracle.grad(bits["h_pol"], bits["W"], dtype, tok, rows, t16["lse_pol"], t16["g"], w)
    g64 = oracle.grad(val["h_pol"], val["W"], "f64", tok, rows, t64["lse_pol"], t64["g"], w)
    for a16, a64 in zip(g16, g64):
        assert np.all(np.isfinite(a16)) and np.array_equal(a16, a64)


def test_kl_small_argument_taylor():
    # p - q tiny: KL ~ x^2/2 + x^3/6 with no cancellation loss
    rng = np.random.default_rng(4)
    h_pol, _, W, tok, adv, mask, L = _tiny_problem(seed=4)
    h_ref = h_pol + 1e-7 * rng.normal(size=h_pol.shape)
    rows = np.arange(h_pol.shape[0], dtype=np.int32)
    t = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows)
    x = t["p"] - t["q"]
    assert np.all(np.abs(x) < 1e-5) and np.any(np.abs(x) > 1e-9)
    assert np.allclose(t["pen"], x * x / 2 + x ** 3 / 6, rtol=1e-6, atol=0)


def test_policy_equals_reference_closed_form():
    """H_ref == H_pol: KL = 0, g = -A exactly, loss = -sum_i len_i A_i / sum_i len_i."""
    wl = synth.generate(synth.CONFIGS["tiny"], seed=5)
    cfg = wl.cfg
    adv = oracle.group_advantages(wl.rewards, 1, cfg.G)
    mask = oracle.build_mask(wl.lengths, cfg.L)
    rows = oracle.valid_rows(mask)
    t = oracle.row_terms(wl.h_pol, wl.h_pol, wl.W, "bf16", wl.tokens, adv, cfg.L, rows)
    assert np.all(t["pen"] == 0.0)
    assert np.array_equal(t["g"], -adv[rows // cfg.L].astype(np.float64))
    loss, nv = oracle.loss(wl.h_pol, wl.h_pol, wl.W, "bf16", wl.tokens, mask, adv, cfg.L)
    lens = wl.lengths.astype(np.float64)
    closed = -float(np.sum(lens * adv.astype(np.float64))) / float(lens.sum())
    assert nv == int(lens.sum())
    assert abs(loss - closed) <= 1e-15 * max(1.0, abs(closed)) + 1e-16


def test_zero_weight_closed_form():
    """W = 0: uniform softmax -> lse = log V, q = p = -log V, dH = 0 and a closed-form dW."""
    h_pol, h_ref, W, tok, adv, mask, L = _tiny_problem(seed=6, G=2, L=4, d=3, V=7, lens=(3, 4))
    W = np.zeros_like(W)
    rows = oracle.valid_rows(mask)
    t = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows)
    V = W.shape[0]
    assert np.allclose(t["lse_pol"], math.log(V), atol=1e-15)
    assert np.allclose(t["q"], -math.log(V), atol=1e-15) and np.allclose(t["p"], -math.log(V), atol=1e-15)
    w = 1.0 / rows.size
    dH, dW = oracle.grad(h_pol, W, "f64", tok, rows, t["lse_pol"], t["g"], w)
    assert np.all(dH == 0.0)
    A = adv[rows // L].astype(np.float64)
    closed = np.zeros((V, h_pol.shape[1]))
    for i, r in enumerate(rows):
        for v in range(V):
            closed[v] += w * (-A[i]) * ((v == tok[r]) - 1.0 / V) * h_pol[r]
    assert np.allclose(dW, closed, rtol=1e-13, atol=1e-16)


# --------------------------------------------------------------------------
# gradients: central finite differences of the detached surrogate
# --------------------------------------------------------------------------

def _fd(fun, x, idx, h=1e-6):
    x0 = x[idx]
    x[idx] = x0 + h
    fp = fun()
    x[idx] = x0 - h
    fm = fun()
    x[idx] = x0
    return (fp - fm) / (2 * h)


@pytest.mark.parametrize("seed", [0, 1])
def test_gradient_finite_differences(seed):
    h_pol, h_ref, W, tok, adv, mask, L = _tiny_problem(seed=seed)
    rows = oracle.valid_rows(mask)
    w = 1.0 / rows.size
    t = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows)
    c = t["q"].copy()                       # the detached value of q
    W_ref = W.copy()                        # frozen reference weight
    # the surrogate at c = q is the loss itself
    loss, nv = oracle.loss(h_pol, h_ref, W, "f64", tok, mask, adv, L)
    J0 = oracle.surrogate(h_pol, h_ref, W, "f64", tok, adv, L, rows, c, w, W_ref=W_ref)
    assert nv == rows.size and abs(J0 - loss) <= 1e-15 * max(1, abs(loss))

    dH, dW = oracle.grad(h_pol, W, "f64", tok, rows, t["lse_pol"], t["g"], w)

    def J():
        return oracle.surrogate(h_pol, h_ref, W, "f64", tok, adv, L, rows, c, w, W_ref=W_ref)

    for i, r in enumerate(rows):
        for k in range(h_pol.shape[1]):
            fd = _fd(J, h_pol, (r, k))
            assert abs(fd - dH[i, k]) <= 1e-6 * max(1e-3, abs(dH[i, k])) + 1e-10
    for v in range(W.shape[0]):
        for k in range(W.shape[1]):
            fd = _fd(J, W, (v, k))
            assert abs(fd - dW[v, k]) <= 1e-6 * max(1e-3, abs(dW[v, k])) + 1e-10
    # masked rows carry no gradient
    for r in np.flatnonzero(mask == 0):
        assert abs(_fd(J, h_pol, (r, 0))) < 1e-12
    # sum over the vocabulary of dW vanishes (each dS row sums to zero)
    assert np.all(np.abs(dW.sum(0)) < 1e-14)


def test_without_detach_policy_gradient_vanishes():
    """exp(q - q) with no detach is the constant 1: only the KL gradient is left."""
    h_pol, h_ref, W, tok, adv, mask, L = _tiny_problem(seed=9)
    rows = oracle.valid_rows(mask)
    w = 1.0 / rows.size
    W_ref = W.copy()
    t = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows)
    x = t["p"] - t["q"]
    g_kl = 0.04 * (1 - np.exp(x))           # d/dq of beta KL only
    dH_kl, _ = oracle.grad(h_pol, W, "f64", tok, rows, t["lse_pol"], g_kl, w, want_dW=False)
    dH_full, _ = oracle.grad(h_pol, W, "f64", tok, rows, t["lse_pol"], t["g"], w, want_dW=False)

    def Jnd():
        return oracle.surrogate(h_pol, h_ref, W, "f64", tok, adv, L, rows, None, w, W_ref=W_ref)

    for i, r in enumerate(rows):
        for k in range(h_pol.shape[1]):
            fd = _fd(Jnd, h_pol, (r, k))
            assert abs(fd - dH_kl[i, k]) <= 1e-6 * max(1e-3, abs(dH_kl[i, k])) + 1e-10
    assert np.max(np.abs(dH_full - dH_kl)) > 1e-3


def _fd_check(fun, h_pol, W, rows, dH, dW):
    for i, r in enumerate(rows):
        for k in range(h_pol.shape[1]):
            fd = _fd(fun, h_pol, (r, k))
            assert abs(fd - dH[i, k]) <= 1e-6 * max(1e-3, abs(dH[i, k])) + 1e-10, (r, k, fd, dH[i, k])
    for v in range(W.shape[0]):
        for k in range(W.shape[1]):
            fd = _fd(fun, W, (v, k))
            assert abs(fd - dW[v, k]) <= 1e-6 * max(1e-3, abs(dW[v, k])) + 1e-10, (v, k, fd, dW[v, k])


@pytest.mark.parametrize("objective", ["grpo", "no_detach", "reverse_kl_q", "forward_kl"])
@pytest.mark.parametrize("loss_mode", ["token_mean", "sequence_mean"])
def test_variant_gradients_finite_differences(objective, loss_mode):
    """Each objective variant and each mean: g and the weights give the surrogate's gradient."""
    h_pol, h_ref, W, tok, adv, mask, L = _tiny_problem(seed=21, G=3, L=3, d=3, V=4, lens=(1, 3, 2), ref_noise=0.5)
    rows = oracle.valid_rows(mask)
    w = oracle.row_weights(rows, L, loss_mode)
    t = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows, objective=objective)
    c = None if objective == "no_detach" else t["q"].copy()
    W_ref = W.copy()
    loss, _ = oracle.loss(h_pol, h_ref, W, "f64", tok, mask, adv, L, objective=objective, loss_mode=loss_mode)
    J0 = oracle.surrogate(h_pol, h_ref, W, "f64", tok, adv, L, rows, c, w, W_ref=W_ref, objective=objective)
    assert abs(J0 - loss) <= 1e-14 * max(1, abs(loss))          # surrogate value = the loss
    dH, dW = oracle.grad(h_pol, W, "f64", tok, rows, t["lse_pol"], t["g"], w)

    def J():
        return oracle.surrogate(h_pol, h_ref, W, "f64", tok, adv, L, rows, c, w, W_ref=W_ref, objective=objective)

    _fd_check(J, h_pol, W, rows, dH, dW)


def test_variant_values():
    """Penalty terms of the variants against their definitions at chosen x = p - q."""
    h_pol, h_ref, W, tok, adv, mask, L = _tiny_problem(seed=22, ref_noise=0.7)
    rows = np.arange(h_pol.shape[0], dtype=np.int32)
    base = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows, objective="grpo")
    x = base["p"] - base["q"]
    assert np.any(np.abs(x) > 0.1)
    k_rev = np.exp(x) - x - 1
    A = adv[rows // L].astype(np.float64)
    nd = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows, objective="no_detach")
    assert np.array_equal(nd["ell"], base["ell"])                       # same value
    assert np.allclose(nd["g"], 0.04 * (1 - np.exp(x)), atol=1e-15)     # the A term has no gradient
    rq = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows, objective="reverse_kl_q")
    assert np.allclose(rq["pen"], np.exp(base["q"]) * k_rev, rtol=1e-12, atol=1e-15)
    fk = oracle.row_terms(h_pol, h_ref, W, "f64", tok, adv, L, rows, objective="forward_kl")
    assert np.allclose(fk["pen"], np.exp(-x) + x - 1, rtol=1e-10, atol=1e-15)
    assert np.all(fk["pen"] >= 0) and np.all(rq["pen"] >= 0)
    for t in (nd, rq, fk):
        assert np.allclose(t["ell"], -A + 0.04 * t["pen"], atol=1e-15)
    # policy = reference: every penalty vanishes
    for obj in ("grpo", "no_detach", "reverse_kl_q", "forward_kl"):
        same = oracle.row_terms(h_pol, h_pol, W, "f64", tok, adv, L, rows, objective=obj)
        assert np.all(same["pen"] == 0)


def test_sequence_mean_closed_form():
    """Policy = reference under the per-completion mean: loss = -mean of A over completions with tokens."""
    wl = synth.generate(synth.make_config("tiny", n_zero_seq=1), seed=8)
    cfg = wl.cfg
    adv = oracle.group_advantages(wl.rewards, 1, cfg.G)
    mask = oracle.build_mask(wl.lengths, cfg.L)
    loss, _ = oracle.loss(wl.h_pol, wl.h_pol, wl.W, "bf16", wl.tokens, mask, adv, cfg.L, loss_mode="sequence_mean")
    active = wl.lengths > 0
    assert active.sum() == cfg.G - 1
    closed = -float(np.mean(adv[active].astype(np.float64)))
    assert abs(loss - closed) <= 1e-15
    rows = oracle.valid_rows(mask)
    w = oracle.row_weights(rows, cfg.L, "sequence_mean")
    assert abs(w.sum() - 1.0) <= 1e-15
    for i in np.flatnonzero(active):
        sel = (rows // cfg.L) == i
        assert np.allclose(w[sel], 1.0 / (active.sum() * wl.lengths[i]), rtol=1e-15)


def test_expected_bundle_consistency():
    wl = synth.generate(synth.CONFIGS["tiny"], seed=0)
    e = oracle.expected(wl)
    cfg = wl.cfg
    loss, nv = oracle.loss(wl.h_pol, wl.h_ref, wl.W, "bf16", wl.tokens, e["mask"], e["adv"], cfg.L)
    assert nv == e["n_valid"] == int(wl.lengths.sum())
    assert abs(loss - e["loss"]) <= 1e-14
    # A-part of the loss is exact from the lengths; the KL part is small and >= 0
    a_part = -float(np.sum(wl.lengths * e["adv"].astype(np.float64))) / nv
    assert 0 <= e["loss"] - a_part < 0.04 * 0.1
    assert np.all(np.abs(e["dW"].sum(0)) < 1e-15)
    # sub-sampled rows give the same per-row terms
    sub = e["rows"][::7]
    e2 = oracle.expected(wl, eval_rows=sub, want_dW=False)
    for k in oracle.ROW_FIELDS:
        assert np.array_equal(e2["terms"][k], e["terms"][k][::7])
    assert np.array_equal(e2["dH"], e["dH"][::7])
