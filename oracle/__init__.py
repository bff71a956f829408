"""fp64 CPU oracle of the linear GRPO loss -- TEST INFRASTRUCTURE ONLY.

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The library (``rl_fine_tuning_gb300``)
neither imports nor links it, and shares no code with it.

The arithmetic lives in ``grpo_oracle.c`` (plain loops, fp64, ascending-index
sums).  This module only compiles it and marshals numpy arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libgrpo_oracle.so")

TYPE_CODE = {"f64": 0, "bf16": 1, "fp16": 2}
ROW_FIELDS = ("lse_pol", "lse_ref", "zt_pol", "zt_ref", "q", "p", "pen", "ell", "g")
OBJECTIVES = {"grpo": 0, "no_detach": 1, "reverse_kl_q": 2, "forward_kl": 3}
LOSS_MODES = {"token_mean": 0, "sequence_mean": 1}


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "grpo_oracle.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
                               "-fPIC", "-shared", src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        p, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_set_threads.argtypes = [i32]
        lib.oracle_max_threads.restype = i32
        lib.oracle_bf16_to_f64.restype = f64
        lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_f64.restype = f64
        lib.oracle_f16_to_f64.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_to_f64.restype = f64
        lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_e5m2_to_f64.restype = f64
        lib.oracle_e5m2_to_f64.argtypes = [ctypes.c_uint8]
        lib.oracle_group_advantages.argtypes = [p, i32, i32, ctypes.c_float, i32, p]
        lib.oracle_build_mask.argtypes = [p, i32, i32, p]
        lib.oracle_valid_rows.restype = i64
        lib.oracle_valid_rows.argtypes = [p, i64, p]
        lib.oracle_logsumexp.restype = f64
        lib.oracle_logsumexp.argtypes = [p, i32]
        lib.oracle_row_terms.argtypes = [p, p, p, p, i32, p, p, i32, i32, i32, f64, i32, p, i64, p]
        lib.oracle_row_weights.argtypes = [p, i64, i32, i32, p]
        lib.oracle_shard_counts.argtypes = [p, i32, i32, p]
        lib.oracle_row_weights_shard.argtypes = [p, i64, i32, i32, i64, i64, p]
        lib.oracle_weighted_sum.restype = f64
        lib.oracle_weighted_sum.argtypes = [p, p, i64]
        lib.oracle_reduce_loss.restype = f64
        lib.oracle_reduce_loss.argtypes = [p, p, i64, i32, i32]
        lib.oracle_loss.restype = f64
        lib.oracle_loss.argtypes = [p, p, p, i32, p, p, p, i64, i32, i32, i32, f64, i32, i32, p]
        lib.oracle_surrogate.restype = f64
        lib.oracle_surrogate.argtypes = [p, p, p, p, i32, p, p, i32, i32, i32, f64, i32, p, i64, p, p]
        lib.oracle_grad.argtypes = [p, p, i32, p, i32, i32, p, i64, p, p, p, p, p, i64, p]
        _lib = lib
    return _lib


def _p(a):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"], "oracle wants C-contiguous arrays"
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int):
    _L().oracle_set_threads(int(n))


def max_threads() -> int:
    return int(_L().oracle_max_threads())


def _mat(a, dtype):
    """H / W argument: uint16 bit patterns for bf16/fp16, float64 for f64."""
    if dtype == "f64":
        return np.ascontiguousarray(a, np.float64)
    return np.ascontiguousarray(a, np.uint16)


def fp8_values(codes, scale, fmt="e4m3"):
    """OCP FP8 codes ("e4m3" / "e5m2") -> float64 values code * scale (exact in
    fp64), via the oracle's decoders."""
    dec = {"e4m3": _L().oracle_e4m3_to_f64, "e5m2": _L().oracle_e5m2_to_f64}[fmt]
    lut = np.array([dec(i) for i in range(256)], np.float64)
    return lut[np.ascontiguousarray(codes, np.uint8)] * float(scale)


def e4m3_values(codes, scale):
    return fp8_values(codes, scale, "e4m3")


def dequantized_workload(wl):
    """A copy of an 8-bit workload whose matrices are the exact float64 values."""
    from copy import copy
    s_pol, s_ref, s_w = wl.extra["scales"]
    fmt = wl.extra.get("fp8", "e4m3")
    out = copy(wl)
    out.h_pol = fp8_values(wl.h_pol, s_pol, fmt)
    out.h_ref = fp8_values(wl.h_ref, s_ref, fmt)
    out.W = fp8_values(wl.W, s_w, fmt)
    return out


def group_advantages(rewards, n_groups, G, eps=1e-4, std_unbiased=True):
    r = np.ascontiguousarray(rewards, np.float32)
    out = np.empty(n_groups * G, np.float32)
    _L().oracle_group_advantages(_p(r), n_groups, G, eps, int(bool(std_unbiased)), _p(out))
    return out


def build_mask(lengths, L):
    lens = np.ascontiguousarray(lengths, np.int32)
    out = np.empty(lens.size * L, np.uint8)
    _L().oracle_build_mask(_p(lens), lens.size, L, _p(out))
    return out


def valid_rows(mask):
    m = np.ascontiguousarray(mask, np.uint8)
    out = np.empty(max(m.size, 1), np.int32)
    n = _L().oracle_valid_rows(_p(m), m.size, _p(out))
    return out[:n].copy()


def logsumexp(z):
    z = np.ascontiguousarray(z, np.float64)
    return float(_L().oracle_logsumexp(_p(z), z.size))


def _obj(objective):
    return OBJECTIVES[objective] if isinstance(objective, str) else int(objective)


def _mode(loss_mode):
    return LOSS_MODES[loss_mode] if isinstance(loss_mode, str) else int(loss_mode)


def row_terms(h_pol, h_ref, W, dtype, tokens, adv, L, rows, beta=0.04, W_ref=None, objective=0):
    """Per-row forward terms for the listed rows -> dict of float64 arrays."""
    h_pol, h_ref, W = _mat(h_pol, dtype), _mat(h_ref, dtype), _mat(W, dtype)
    Wr = None if W_ref is None else _mat(W_ref, dtype)
    V, d = W.shape
    tok = np.ascontiguousarray(tokens, np.int32)
    adv = np.ascontiguousarray(adv, np.float32)
    rows = np.ascontiguousarray(rows, np.int32)
    out = np.empty((rows.size, 9), np.float64)
    _L().oracle_row_terms(_p(h_pol), _p(h_ref), _p(W), _p(Wr), TYPE_CODE[dtype], _p(tok), _p(adv),
                          L, d, V, beta, _obj(objective), _p(rows), rows.size, _p(out))
    return {k: out[:, i].copy() for i, k in enumerate(ROW_FIELDS)}


def row_weights(rows, L, loss_mode=0):
    """Loss weight of each listed masked-in row (ascending)."""
    rows = np.ascontiguousarray(rows, np.int32)
    out = np.empty(rows.size, np.float64)
    _L().oracle_row_weights(_p(rows), rows.size, L, _mode(loss_mode), _p(out))
    return out


def shard_counts(mask, n_seq, L):
    """(masked-in rows, completions with a masked-in row) of one shard's mask."""
    m = np.ascontiguousarray(mask, np.uint8)
    out = np.zeros(2, np.int64)
    _L().oracle_shard_counts(_p(m), int(n_seq), int(L), _p(out))
    return int(out[0]), int(out[1])


def row_weights_shard(rows, L, n_valid_batch, n_active_batch, loss_mode=0):
    """Loss weights of one shard's masked-in rows when the batch's divisors
    (all shards' masked-in rows and active completions) are given."""
    rows = np.ascontiguousarray(rows, np.int32)
    out = np.empty(rows.size, np.float64)
    _L().oracle_row_weights_shard(_p(rows), rows.size, L, _mode(loss_mode), int(n_valid_batch),
                                  int(n_active_batch), _p(out))
    return out


def weighted_sum(ell, w):
    """sum_i w_i ell_i (a shard's share of the batch loss)."""
    ell = np.ascontiguousarray(ell, np.float64)
    w = np.ascontiguousarray(w, np.float64)
    return float(_L().oracle_weighted_sum(_p(ell), _p(w), ell.size))


def reduce_loss(ell, rows, L, loss_mode=0):
    ell = np.ascontiguousarray(ell, np.float64)
    rows = np.ascontiguousarray(rows, np.int32)
    return float(_L().oracle_reduce_loss(_p(ell), _p(rows), rows.size, L, _mode(loss_mode)))


def loss(h_pol, h_ref, W, dtype, tokens, mask, adv, L, beta=0.04, objective=0, loss_mode=0):
    """Loss over the masked rows (token mean or sequence mean) and N_v."""
    h_pol, h_ref, W = _mat(h_pol, dtype), _mat(h_ref, dtype), _mat(W, dtype)
    V, d = W.shape
    tok = np.ascontiguousarray(tokens, np.int32)
    mask = np.ascontiguousarray(mask, np.uint8)
    adv = np.ascontiguousarray(adv, np.float32)
    nv = ctypes.c_int64(0)
    val = _L().oracle_loss(_p(h_pol), _p(h_ref), _p(W), TYPE_CODE[dtype], _p(tok), _p(mask), _p(adv),
                           mask.size, L, d, V, beta, _obj(objective), _mode(loss_mode), ctypes.byref(nv))
    return float(val), int(nv.value)


def surrogate(h_pol, h_ref, W, dtype, tokens, adv, L, rows, c, w, beta=0.04, W_ref=None, objective=0):
    """sum_i w_i [-A exp(q_i - c_i) + beta pen_i]; c=None re-evaluates c = q (no detach).

    w: per-row weights (or one scalar for all rows); W_ref: weight of the
    frozen reference (None: W itself)."""
    h_pol, h_ref, W = _mat(h_pol, dtype), _mat(h_ref, dtype), _mat(W, dtype)
    Wr = None if W_ref is None else _mat(W_ref, dtype)
    V, d = W.shape
    tok = np.ascontiguousarray(tokens, np.int32)
    adv = np.ascontiguousarray(adv, np.float32)
    rows = np.ascontiguousarray(rows, np.int32)
    cc = None if c is None else np.ascontiguousarray(c, np.float64)
    ww = np.ascontiguousarray(np.broadcast_to(np.asarray(w, np.float64), (rows.size,)))
    return float(_L().oracle_surrogate(_p(h_pol), _p(h_ref), _p(W), _p(Wr), TYPE_CODE[dtype], _p(tok),
                                       _p(adv), L, d, V, beta, _obj(objective), _p(rows), rows.size, _p(cc),
                                       _p(ww)))


def grad(h_pol, W, dtype, tokens, rows, lse, g, w, want_dH=True, vrows=None, want_dW=True):
    """dH for the listed rows ([n_rows, d]) and dW for vocabulary rows vrows (all if None).

    w: per-row loss weights (or one scalar for all rows)."""
    h_pol, W = _mat(h_pol, dtype), _mat(W, dtype)
    V, d = W.shape
    tok = np.ascontiguousarray(tokens, np.int32)
    rows = np.ascontiguousarray(rows, np.int32)
    lse = np.ascontiguousarray(lse, np.float64)
    g = np.ascontiguousarray(g, np.float64)
    ww = np.ascontiguousarray(np.broadcast_to(np.asarray(w, np.float64), (rows.size,)))
    dH = np.empty((rows.size, d), np.float64) if want_dH else None
    vr = None if vrows is None else np.ascontiguousarray(vrows, np.int32)
    n_v = V if vr is None else vr.size
    dW = np.empty((n_v, d), np.float64) if want_dW else None
    _L().oracle_grad(_p(h_pol), _p(W), TYPE_CODE[dtype], _p(tok), d, V, _p(rows), rows.size,
                     _p(lse), _p(g), _p(ww), _p(dH), _p(vr), 0 if vr is None else vr.size, _p(dW))
    return dH, dW


def expected(wl, eval_rows=None, vrows=None, mask=None, want_dH=True, want_dW=True,
             std_unbiased=True, objective=0, loss_mode=0):
    """Everything the library computes for a synthetic workload, in fp64.

    eval_rows: the valid rows whose per-row terms (and dH) are computed; None
    means every valid row, in which case the loss is the full masked mean.
    mask: overrides the mask built from the workload's lengths.
    """
    cfg = wl.cfg
    adv = group_advantages(wl.rewards, cfg.n_groups, cfg.G, cfg.eps, std_unbiased)
    if mask is None:
        mask = build_mask(wl.lengths, cfg.L)
    rows_all = valid_rows(mask)
    n_valid = rows_all.size
    w_all = row_weights(rows_all, cfg.L, loss_mode)
    full = eval_rows is None
    rows = rows_all if full else np.ascontiguousarray(eval_rows, np.int32)
    w = w_all if full else w_all[np.searchsorted(rows_all, rows)]
    mtype = "f64" if wl.h_pol.dtype == np.float64 else cfg.dtype
    terms = row_terms(wl.h_pol, wl.h_ref, wl.W, mtype, wl.tokens, adv, cfg.L, rows, cfg.beta,
                      objective=objective)
    out = dict(adv=adv, mask=mask, rows=rows_all, n_valid=n_valid, w=w, eval_rows=rows, terms=terms)
    if full:
        out["loss"] = reduce_loss(terms["ell"], rows_all, cfg.L, loss_mode)
    if want_dH or want_dW:
        dH, dW = grad(wl.h_pol, wl.W, mtype, wl.tokens, rows, terms["lse_pol"], terms["g"], w,
                      want_dH=want_dH, vrows=vrows, want_dW=want_dW and full)
        out["dH"] = dH
        out["dW"] = dW
    return out
