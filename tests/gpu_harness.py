"""Host-side glue for the GPU tests: moves a synthetic workload to the device,
calls libgrpo through its C ABI (the ctypes binding) and brings the results
back as numpy arrays.  No arithmetic of the method lives here."""
from __future__ import annotations

import numpy as np

import rl_fine_tuning_gb300 as rg
import synth


def torch():
    import torch as t
    return t


def dev_bits(a: np.ndarray, dtype: str):
    """uint16 bit patterns -> device tensor of bf16/fp16."""
    t = torch()
    x = t.from_numpy(np.ascontiguousarray(a).view(np.int16)).cuda()
    return x.view(t.bfloat16 if dtype == "bf16" else t.float16)


def host_f64(x, dtype: str) -> np.ndarray:
    """device bf16/fp16 tensor -> float64 numpy (exact)."""
    t = torch()
    b = x.contiguous().view(t.int16).cpu().numpy().view(np.uint16)
    return synth.bits_to_f32(b, dtype).astype(np.float64)


def shape_for(cfg, chunk_rows=0, beta=None, objective=0, loss_mode=0, std_unbiased=True):
    return rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V, rg.BF16 if cfg.dtype == "bf16" else rg.FP16,
                         beta=cfg.beta if beta is None else beta, eps=cfg.eps, chunk_rows=chunk_rows,
                         objective=objective, loss_mode=loss_mode, std_unbiased=std_unbiased)


class DeviceWorkload:
    def __init__(self, wl, mask=None, chunk_rows=0, objective=0, loss_mode=0, std_unbiased=True):
        t = torch()
        cfg = wl.cfg
        self.cfg = cfg
        self.shape = shape_for(cfg, chunk_rows, objective=objective, loss_mode=loss_mode, std_unbiased=std_unbiased)
        self.h_pol = dev_bits(wl.h_pol, cfg.dtype)
        self.h_ref = dev_bits(wl.h_ref, cfg.dtype)
        self.W = dev_bits(wl.W, cfg.dtype)
        self.tokens = t.from_numpy(wl.tokens).cuda()
        self.lengths = t.from_numpy(wl.lengths).cuda()
        self.rewards = t.from_numpy(wl.rewards).cuda()
        self.adv = t.empty(cfg.n_seq, dtype=t.float32, device="cuda")
        rg.grpo_group_advantages(self.rewards, cfg.n_groups, cfg.G, cfg.eps, std_unbiased, self.adv)
        if mask is None:
            self.mask = t.empty(cfg.N, dtype=t.uint8, device="cuda")
            rg.grpo_build_mask(self.lengths, self.shape, self.mask)
        else:
            self.mask = t.from_numpy(np.ascontiguousarray(mask, np.uint8)).cuda()
        nbytes = rg.grpo_workspace_bytes(self.shape)
        assert nbytes > 0
        self.ws = t.empty(nbytes, dtype=t.uint8, device="cuda")
        self.loss = t.zeros(1, dtype=t.float32, device="cuda")
        self.status = t.zeros(1, dtype=t.int32, device="cuda")
        self.found_inf = t.zeros(1, dtype=t.int32, device="cuda")
        self.row_stats = t.zeros((cfg.N, 5), dtype=t.float32, device="cuda")
        dt = t.bfloat16 if cfg.dtype == "bf16" else t.float16
        # a finite sentinel: a backward must overwrite every element (masked dH rows with 0)
        self.dH = t.full((cfg.N, cfg.d), 7.0, dtype=dt, device="cuda")
        self.dW = t.full((cfg.V, cfg.d), 7.0, dtype=t.float32, device="cuda")

    def fwd(self):
        rg.grpo_loss_fwd(self.h_pol, self.h_ref, self.W, self.tokens, self.mask, self.adv, self.shape, self.ws,
                         self.loss, self.row_stats, self.status)
        torch().cuda.synchronize()
        return self

    def fwd_bwd(self, loss_scale=1.0):
        rg.grpo_loss_fwd_bwd(self.h_pol, self.h_ref, self.W, self.tokens, self.mask, self.adv, self.shape,
                             loss_scale, self.ws, self.loss, self.dH, self.dW, self.found_inf, self.row_stats,
                             self.status)
        torch().cuda.synchronize()
        return self

    def results(self):
        cfg = self.cfg
        return dict(
            loss=float(self.loss.item()),
            status=int(self.status.item()),
            found_inf=int(self.found_inf.item()),
            row_stats=self.row_stats.cpu().numpy().astype(np.float64),
            adv=self.adv.cpu().numpy(),
            mask=self.mask.cpu().numpy(),
            dH=host_f64(self.dH, cfg.dtype),
            dW=self.dW.cpu().numpy().astype(np.float64),
        )
