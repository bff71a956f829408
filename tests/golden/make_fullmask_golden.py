"""Writes the full-mask expected values of a model-head workload, from the fp64 oracle only.

    python tests/golden/make_fullmask_golden.py WORKLOAD [WORKLOAD ...]
    python tests/golden/make_fullmask_golden.py --completion I WORKLOAD

The second form masks the workload to the rows of completion I alone (all its
generated rows, the other completions masked out) and writes
``tests/golden/completion<I>_<WORKLOAD>.npz``: the same values for a batch
whose masked-in rows fill several backward chunks of the full-size shape, at
an oracle cost of one completion.

For each workload (a name in ``synth.CONFIGS``) it generates the seeded
inputs (seed 0), builds the completion mask from the generated lengths and
asks the oracle (``oracle/``, on the host cores) for:

  * the loss over every masked-in row (token mean, GRPO objective),
  * the per-row terms of every masked-in row: lse of the policy and reference
    logits, q, p and the KL penalty (the library's ``row_stats`` columns),
  * the gradient dW for a seeded sample of 16 vocabulary rows, summed over
    every masked-in row -- the one output that no single row determines.

The result goes to ``tests/golden/fullmask_<WORKLOAD>.npz`` with a
fingerprint of the generated inputs, so a test can first check that it
regenerated the same inputs.  Nothing here reads the library or a GPU.
Per-row values are stored as float32 and dW rows as float32: their rounding
(relative 6e-8) is far below every tolerance the tests apply.
"""
from __future__ import annotations

import hashlib
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402

SEED = 0
N_VROWS = 16


def out_path(name: str) -> str:
    return os.path.join(HERE, f"fullmask_{name}.npz")


def fingerprint(wl) -> str:
    """sha256 over the generated inputs' bytes (hidden states, weight, tokens, lengths, rewards)."""
    h = hashlib.sha256()
    for a in (wl.h_pol, wl.h_ref, wl.W, wl.tokens, wl.lengths, wl.rewards):
        h.update(np.ascontiguousarray(a).tobytes())
    return h.hexdigest()


def pick_vrows(cfg, tokens_valid: np.ndarray) -> np.ndarray:
    """First, middle and last vocabulary rows, four rows that are sampled tokens
    of masked-in rows, and random rows up to N_VROWS (seeded)."""
    rng = np.random.default_rng(29)
    pick = {0, cfg.V // 2, cfg.V - 1}
    hits = np.unique(tokens_valid)
    pick.update(int(v) for v in rng.choice(hits, size=4, replace=False))
    while len(pick) < N_VROWS:
        pick.add(int(rng.integers(0, cfg.V)))
    return np.array(sorted(pick), np.int32)


def completion_mask(cfg, lengths, i: int) -> np.ndarray:
    """The completion mask of the workload with every completion but i masked out."""
    full = oracle.build_mask(lengths, cfg.L)
    mask = np.zeros_like(full)
    mask[i * cfg.L:(i + 1) * cfg.L] = full[i * cfg.L:(i + 1) * cfg.L]
    return mask


def make(name: str, completion=None) -> str:
    cfg = synth.CONFIGS[name]
    t0 = time.time()
    wl = synth.generate(cfg, seed=SEED)
    adv = oracle.group_advantages(wl.rewards, cfg.n_groups, cfg.G, cfg.eps, True)
    if completion is None:
        mask = oracle.build_mask(wl.lengths, cfg.L)
    else:
        mask = completion_mask(cfg, wl.lengths, completion)
    rows = oracle.valid_rows(mask)
    terms = oracle.row_terms(wl.h_pol, wl.h_ref, wl.W, cfg.dtype, wl.tokens, adv, cfg.L, rows, cfg.beta)
    loss = oracle.reduce_loss(terms["ell"], rows, cfg.L)
    w = oracle.row_weights(rows, cfg.L)
    vrows = pick_vrows(cfg, wl.tokens[rows])
    _, dW = oracle.grad(wl.h_pol, wl.W, cfg.dtype, wl.tokens, rows, terms["lse_pol"], terms["g"], w,
                        want_dH=False, vrows=vrows, want_dW=True)
    path = out_path(name) if completion is None else os.path.join(HERE, f"completion{completion}_{name}.npz")
    cmd = f"python tests/golden/make_fullmask_golden.py {name}" if completion is None else \
        f"python tests/golden/make_fullmask_golden.py --completion {completion} {name}"
    np.savez(path, workload=np.array(name), seed=np.array(SEED), fingerprint=np.array(fingerprint(wl)),
             completion=np.array(-1 if completion is None else completion),
             n_valid=np.array(rows.size, np.int64), loss=np.array(loss, np.float64),
             pen_mean=np.array(float(np.mean(terms["pen"])), np.float64), rows=rows.astype(np.int32),
             lse_pol=terms["lse_pol"].astype(np.float32), lse_ref=terms["lse_ref"].astype(np.float32),
             q=terms["q"].astype(np.float32), p=terms["p"].astype(np.float32),
             pen=terms["pen"].astype(np.float32), vrows=vrows, dW_rows=dW.astype(np.float32),
             command=np.array(cmd))
    print(f"{name}: N_v {rows.size}, loss {loss:.9f}, {time.time() - t0:.0f} s -> {path}", flush=True)
    return path


if __name__ == "__main__":
    args = sys.argv[1:]
    if not args:
        raise SystemExit(__doc__)
    oracle.build()
    synth.build()
    if args[0] == "--completion":
        make(args[2], completion=int(args[1]))
    else:
        for n in args:
            make(n)
