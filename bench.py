#!/usr/bin/env python
"""Benchmark: fused linear GRPO loss forward+backward on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl ours|reference]

One step = the whole hot path on one batch: group advantages, completion
mask, row index, policy+reference lm_head logits with streaming logsumexp,
objective and masked mean, and the backward: dlogits from the exponentials
the forward kept, then dH and dW.  The
default workload is the Llama-3.1-8B head at 20K context with 8 completions
(G=8, L=20000, d=4096, V=128256, bf16), synthetic seeded inputs shaped like
the pages' long-context run.  Inputs (W 1 GB, hidden states 1.3 GB each) are
larger than L2, so steps need no L2 flush.

Prints one JSON line (rank 0).  With N>1 (torchrun) each rank runs an
independent replica of the same workload by default; with --split the N
ranks hold one batch of N prompt groups as data-parallel shards (each rank
one group, the same synthetic inputs on every rank): every step sums the
batch's counts before the loss and the loss shares and dW after it over the
ranks (NCCL), so each rank ends the step with the batch's loss and dW.
value = all ranks' tokens / max-over-ranks time.

--impl reference times the fp64 CPU oracle on the host cores on a bounded
sample of rows of the same workload, each step a different sample.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "GRPO loss fwd+bwd tokens/s and % of bf16 tensor peak on 1 GB300; peak extra HBM"
DEFAULT_CONFIG = "llama-3.1-8b-20k"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
DATASHEET_BF16_TFLOPS = 2250.0   # GB300 dense bf16 tensor peak (without sparsity)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--chunk-rows", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-graph", action="store_true", help="skip the CUDA-graph replay timing")
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="target length of one oracle sample")
    ap.add_argument("--forward", action="store_true",
                    help="time the forward-only entry points (bf16 and e4m3 inputs) instead of fwd+bwd")
    ap.add_argument("--split", action="store_true",
                    help="with N>1: one batch of N prompt groups split over the ranks (data-parallel shards), "
                         "the batch counts and dW summed over the ranks every step; default: N replicas")
    return ap.parse_args()


# --------------------------------------------------------------------------- ranks

class Ranks:
    """The ranks of a torchrun launch: a gloo group for barriers and timings and,
    for the data-parallel split, a second group (NCCL on GPUs) that sums the
    shards' counts, loss shares and dW."""

    def __init__(self, n_gpus, split=False, device_backend="nccl"):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        self.dev_group = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist
            if split:
                if device_backend == "nccl":
                    import torch
                    torch.cuda.set_device(self.local)
                self.dev_group = dist.new_group(backend=device_backend)

    def sum_(self, *tensors):
        """In-place sum over the ranks (the shards' exchange); nothing on one rank."""
        if not self.dev_group:
            return
        for t in tensors:
            self.pg.all_reduce(t, group=self.dev_group)

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, x: float) -> float:
        if not self.pg:
            return x
        import torch
        t = torch.tensor([x], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


# --------------------------------------------------------------------------- clocks

CLOCK_FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASON_NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons every 200 ms."""

    def __init__(self, gpu_uuid=None):
        self.proc = None
        self.path = None
        self.out = None
        try:
            import tempfile
            fd, self.path = tempfile.mkstemp(prefix="grpo_clocks_", suffix=".csv")
            os.close(fd)
            cmd = ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits", "-lms", "200"]
            if gpu_uuid:
                cmd += ["-i", gpu_uuid]
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(cmd, stdout=self.out, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
            self._discard()

    def _discard(self):
        """Close and remove the sample file (no sampler is running)."""
        if self.out is not None:
            self.out.close()
            self.out = None
        if self.path and os.path.exists(self.path):
            os.unlink(self.path)
        self.path = None

    def stop(self):
        if not self.proc:
            self._discard()
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.out.close()
        sm, smax, reasons = [], [], set()
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    smax.append(float(parts[2]))
                except ValueError:
                    continue
                for name, val in zip(REASON_NAMES, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(name)
        os.unlink(self.path)
        self.path = None
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def gpu_uuid():
    try:
        import torch
        u = torch.cuda.get_device_properties(torch.cuda.current_device()).uuid
        s = str(u)
        return s if s.startswith("GPU-") else "GPU-" + s
    except Exception:
        return None


# --------------------------------------------------------------------------- helpers

def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def kernel_source_hash():
    h = hashlib.sha256()
    for f in ("tc_kernels.cu", "ptx.cuh"):
        h.update(open(os.path.join(ROOT, "rl_fine_tuning_gb300", "csrc", f), "rb").read())
    return h.hexdigest()[:16]


def ncu_traffic(kind, chunk_rows, field="dram_bytes_per_launch_full_workload"):
    """DRAM bytes per launch of `kind` from the committed ncu summary (the median of
    its captures; field="spread" gives their range), if it was taken on the current
    kernel source with chunks of the same height; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
    except Exception:
        return None
    if d.get("kernel_source_hash") != kernel_source_hash() or d.get("chunk_rows") != chunk_rows:
        return None
    ent = d.get("kernels", {}).get(kind)
    if not ent:
        return None
    return ent.get(field)


def cfg_dict(cfg, extra=None):
    d = {"workload": cfg.name, "G": cfg.G, "L": cfg.L, "N": cfg.N, "d": cfg.d, "V": cfg.V,
         "global_batch": cfg.N, "seq_len": cfg.L, "beta": cfg.beta, "lengths": [cfg.len_lo, cfg.len_hi],
         "parallelism": "replicas", "l2": "inputs larger than L2 (no flush)"}
    if extra:
        d.update(extra)
    return d


def sample_rows(valid_rows, n, seed):
    import numpy as np
    rng = np.random.default_rng(seed)
    n = min(n, valid_rows.size)
    return np.sort(rng.choice(valid_rows, size=n, replace=False)).astype(np.int32)


def oracle_sample(cfg, wl, rows, adv):
    """One bounded oracle run: per-row terms, dH and the dW contribution of the sampled rows."""
    import oracle
    t0 = time.perf_counter()
    terms = oracle.row_terms(wl.h_pol, wl.h_ref, wl.W, cfg.dtype, wl.tokens, adv, cfg.L, rows, cfg.beta)
    oracle.grad(wl.h_pol, wl.W, cfg.dtype, wl.tokens, rows, terms["lse_pol"], terms["g"], 1.0 / rows.size)
    return time.perf_counter() - t0


# --------------------------------------------------------------------------- reference arm

def run_reference(args, ranks):
    import numpy as np

    import oracle
    import synth
    cfg = synth.make_config(args.config)
    if ranks.rank != 0:
        return
    oracle.build()
    synth.build()
    wl = synth.generate(cfg, seed=0)
    adv = oracle.group_advantages(wl.rewards, cfg.n_groups, cfg.G, cfg.eps, True)
    mask = oracle.build_mask(wl.lengths, cfg.L)
    valid = oracle.valid_rows(mask)
    budget = max(2.0, min(args.cpu_seconds, 150.0 / max(1, args.steps + args.warmup)))
    # calibrate on a small sample, then size each step to the budget
    cal = sample_rows(valid, max(1, oracle.max_threads()), 12345)
    t_cal = oracle_sample(cfg, wl, cal, adv)
    n_rows = max(1, int(budget / (t_cal / cal.size)))
    times = []
    for i in range(args.warmup + args.steps):
        rows = sample_rows(valid, n_rows, 1000 + i)
        dt = oracle_sample(cfg, wl, rows, adv)
        if i >= args.warmup:
            times.append((rows.size, dt))
    toks = sum(n for n, _ in times)
    secs = sum(t for _, t in times)
    value = toks / secs
    cores = oracle.max_threads()
    sample = (f"{n_rows} seeded valid rows per step of {cfg.name} (of {valid.size}); per-row lse, q, p, KL, "
              f"dH and dW contribution in fp64")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * secs / len(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": cfg_dict(cfg, {"sample_rows_per_step": n_rows}),
        "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# --------------------------------------------------------------------------- our arm

def run_ours(args, ranks):
    import numpy as np
    import torch

    import rl_fine_tuning_gb300 as rg
    import synth

    torch.cuda.set_device(ranks.local)
    rg.load(build_if_missing=True)
    cfg = synth.make_config(args.config)
    wl = synth.generate(cfg, seed=0)
    lengths_np = wl.lengths
    n_valid = int(np.minimum(np.maximum(lengths_np, 0), cfg.L).sum())

    tdt = torch.bfloat16 if cfg.dtype == "bf16" else torch.float16
    shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V, rg.BF16 if cfg.dtype == "bf16" else rg.FP16,
                          beta=cfg.beta, eps=cfg.eps, chunk_rows=args.chunk_rows)

    def pinned(a):
        t = torch.from_numpy(a.view(np.int16) if a.dtype == np.uint16 else a)
        return t.pin_memory()

    host = {"h_pol": pinned(wl.h_pol), "h_ref": pinned(wl.h_ref), "tokens": pinned(wl.tokens),
            "lengths": pinned(wl.lengths), "rewards": pinned(wl.rewards)}
    dev = {k: v.cuda() for k, v in host.items()}
    dev["h_pol"] = dev["h_pol"].view(tdt)
    dev["h_ref"] = dev["h_ref"].view(tdt)
    W = torch.from_numpy(wl.W.view(np.int16)).cuda().view(tdt)
    N, d, V = cfg.N, cfg.d, cfg.V
    adv = torch.empty(cfg.n_seq, dtype=torch.float32, device="cuda")
    mask = torch.empty(N, dtype=torch.uint8, device="cuda")
    # (with one rank the split is the whole batch, still through the shard entry points)
    split = args.split

    def outputs():
        return {"dH": torch.empty((N, d), dtype=tdt, device="cuda"),
                "dW": torch.empty((V, d), dtype=torch.float32, device="cuda"),
                "loss": torch.zeros(1, dtype=torch.float32, device="cuda")}

    out = outputs()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    found_inf = torch.zeros(1, dtype=torch.int32, device="cuda")
    counts = torch.zeros(2, dtype=torch.int32, device="cuda")
    ws_bytes = rg.grpo_workspace_bytes(shape)
    ws = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()
    scale = [cfg.loss_scale]

    def step(d_in, o=None):
        o = out if o is None else o
        rg.grpo_group_advantages(d_in["rewards"], cfg.n_groups, cfg.G, cfg.eps, True, adv)
        rg.grpo_build_mask(d_in["lengths"], shape, mask)
        if not split:
            rg.grpo_loss_fwd_bwd(d_in["h_pol"], d_in["h_ref"], W, d_in["tokens"], mask, adv, shape, scale[0], ws,
                                 o["loss"], o["dH"], o["dW"], found_inf, None, status)
            return
        # one shard of the batch: the batch's counts, then this rank's share, then the sums
        rg.grpo_shard_counts(mask, shape, counts)
        ranks.sum_(counts)
        rg.grpo_loss_fwd_bwd_shard(d_in["h_pol"], d_in["h_ref"], W, d_in["tokens"], mask, adv, shape, counts,
                                   scale[0], ws, o["loss"], o["dH"], o["dW"], found_inf, None, status)
        ranks.sum_(o["dW"], o["loss"])

    # warm-up (also settles the fp16 loss scale: halve while the scaled gradients overflow)
    for _ in range(max(args.warmup, 1)):
        step(dev)
    torch.cuda.synchronize()
    while cfg.dtype == "fp16" and int(found_inf.item()) == 1 and scale[0] > 1.0:
        scale[0] /= 2
        step(dev)
        torch.cuda.synchronize()
    st_code = int(status.item())
    if st_code != 0:
        raise SystemExit(f"device status {st_code}: {rg.grpo_status_string(st_code)}")
    if not np.isfinite(out["loss"].item()):
        raise SystemExit("non-finite loss")

    # ---------------- device-resident timed region
    torch.cuda.reset_peak_memory_stats()
    mem_base = torch.cuda.memory_allocated()
    ranks.barrier()
    torch.cuda.synchronize()
    sampler = ClockSampler(gpu_uuid())
    launches0 = rg.grpo_kernel_launches()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(args.steps):
        step(dev)
    e1.record(stream)
    torch.cuda.synchronize()
    launches = rg.grpo_kernel_launches() - launches0
    clocks = sampler.stop()
    # the timed steps repeat the warm-up's inputs at its settled loss scale, so
    # none may overflow; a step that did would need a retry the timing lacks
    if int(found_inf.item()) != 0 or int(status.item()) != 0:
        raise SystemExit("a timed step overflowed or reported a device error")
    ranks.barrier()
    ms = e0.elapsed_time(e1)
    # the per-kernel breakdown comes from a second pass over the same steps with
    # the library's launch events on (they cost about 1% of the step, so they
    # stay out of the timed region above)
    rg.grpo_profile_enable(True)
    for _ in range(args.steps):
        step(dev)
    torch.cuda.synchronize()
    rg.grpo_profile_enable(False)
    prof = rg.grpo_profile_collect()
    ms_max = ranks.max(ms)
    peak_extra = torch.cuda.max_memory_allocated() - mem_base
    ms_step = ms_max / args.steps
    value = ranks.world * n_valid * args.steps / (ms_max / 1e3)

    # ---------------- the same step captured once into a CUDA graph and replayed
    graph = None
    if not args.no_graph and not split:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            step(dev)
        stream.wait_stream(side)
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            step(dev)
        g.replay()
        torch.cuda.synchronize()
        ranks.barrier()
        g0 = torch.cuda.Event(enable_timing=True)
        g1 = torch.cuda.Event(enable_timing=True)
        g0.record(stream)
        for _ in range(args.steps):
            g.replay()
        g1.record(stream)
        torch.cuda.synchronize()
        ms_g = ranks.max(g0.elapsed_time(g1))
        graph = {"value": ranks.world * n_valid * args.steps / (ms_g / 1e3), "unit": "tokens/s",
                 "ms_per_step": ms_g / args.steps, "what": "one step captured into a CUDA graph, replayed"}
        del g

    # ---------------- end to end: host inputs copied in, results read back, every step
    # Through the public API with every step's inputs copied from pinned host
    # memory inside the timed region: serially before each step, and overlapped
    # the way a training loop prefetches its next batch (step i+1's inputs
    # copied on a second stream into a second device buffer set while step i
    # computes).  The headline reads back the loss only: the gradients stay on
    # the device, where the optimizer step of a trainer consumes them.  A third
    # variant also copies dH and dW of every step back to pinned host memory (on
    # a third stream, from two alternating output sets, while the next step runs).
    e2e = None
    if not args.no_e2e:
        loss_host = torch.zeros(1, dtype=torch.float32).pin_memory()
        h2d = sum(host[k].numel() * host[k].element_size() for k in host)
        dev2 = {k: torch.empty_like(v) for k, v in dev.items()}

        def copy_in(d_in):
            for k in host:
                dev_raw = d_in[k].view(host[k].dtype) if k in ("h_pol", "h_ref") else d_in[k]
                dev_raw.copy_(host[k], non_blocking=True)

        def run_serial(n):
            for _ in range(n):
                copy_in(dev)
                step(dev)
                loss_host.copy_(out["loss"], non_blocking=True)

        copy_stream = torch.cuda.Stream()
        back_stream = torch.cuda.Stream()
        bufs = (dev, dev2)
        copied = [torch.cuda.Event() for _ in bufs]
        consumed = [torch.cuda.Event() for _ in bufs]
        outs = [out]
        grads_host = None

        def run_overlapped(n, grads_back=False):
            copy_stream.wait_stream(stream)
            with torch.cuda.stream(copy_stream):
                copy_in(bufs[0])
                copied[0].record(copy_stream)
            computed = [torch.cuda.Event() for _ in outs]
            drained = [None for _ in outs]
            for i in range(n):
                b = i % 2
                if i + 1 < n:
                    nb = (i + 1) % 2
                    with torch.cuda.stream(copy_stream):
                        if i >= 1:
                            copy_stream.wait_event(consumed[nb])   # step i-1 has finished with that buffer
                        copy_in(bufs[nb])
                        copied[nb].record(copy_stream)
                stream.wait_event(copied[b])
                if not grads_back:
                    step(bufs[b])
                    consumed[b].record(stream)
                    loss_host.copy_(out["loss"], non_blocking=True)
                    continue
                ob = i % 2
                if drained[ob] is not None:
                    stream.wait_event(drained[ob])              # step i-2's gradients have left this set
                step(bufs[b], outs[ob])
                consumed[b].record(stream)
                computed[ob].record(stream)
                back_stream.wait_event(computed[ob])
                with torch.cuda.stream(back_stream):
                    for k in ("dH", "dW", "loss"):
                        grads_host[k].copy_(outs[ob][k].view(grads_host[k].dtype), non_blocking=True)
                    ev = torch.cuda.Event()
                    ev.record(back_stream)
                    drained[ob] = ev
            stream.wait_stream(back_stream)

        def timed(fn):
            fn(1)
            torch.cuda.synchronize()
            ranks.barrier()
            a0 = torch.cuda.Event(enable_timing=True)
            a1 = torch.cuda.Event(enable_timing=True)
            a0.record(stream)
            fn(args.steps)
            a1.record(stream)
            torch.cuda.synchronize()
            return ranks.max(a0.elapsed_time(a1))

        ms_ser = timed(run_serial)
        ms_ovl = timed(run_overlapped)
        # the same loop with the gradients read back every step
        outs.append(outputs())
        grads_host = {"dH": torch.empty((N, d), dtype=torch.int16).pin_memory(),
                      "dW": torch.empty((V, d), dtype=torch.float32).pin_memory(),
                      "loss": torch.empty(1, dtype=torch.float32).pin_memory()}
        d2h_grads = sum(t.numel() * t.element_size() for t in grads_host.values())
        ms_grads = timed(lambda n: run_overlapped(n, grads_back=True))
        del dev2, grads_host
        outs.pop()
        e2e = {"value": ranks.world * n_valid * args.steps / (ms_ovl / 1e3), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": 4, "ms_per_step": ms_ovl / args.steps,
               "copies": "step i+1's inputs copied on a second stream during step i (two device input sets); "
                         "the loss read back every step; dH and dW stay on the device for the optimizer",
               "serial": {"value": ranks.world * n_valid * args.steps / (ms_ser / 1e3),
                          "ms_per_step": ms_ser / args.steps, "copies": "before each step, same stream"},
               "with_gradients": {"value": ranks.world * n_valid * args.steps / (ms_grads / 1e3),
                                  "ms_per_step": ms_grads / args.steps, "h2d_bytes_per_step": int(h2d),
                                  "d2h_bytes_per_step": int(d2h_grads),
                                  "copies": "as the headline, plus dH, dW and the loss of every step copied to "
                                            "pinned host memory on a third stream while the next step runs "
                                            "(two device output sets)"},
               "resident": "lm_head weight W"}

    # ---------------- roofline of the dominant kernel
    pk, pk_kind = peaks()
    # algorithmic work per kernel kind over the timed steps: the three GEMM kernels
    # in flops, the dlogits pass (read exponentials, write dlogits, in place) in bytes
    flops_kind = {"fwd": 4.0 * n_valid * V * d, "dh": 2.0 * n_valid * V * d, "dw": 2.0 * n_valid * V * d}
    v_pad = (V + 63) // 64 * 64
    bytes_kind = {"dlogits": n_valid * (v_pad * 2 * 2 + ((V + 31) // 32) * 4)}
    total_kernel_ms = sum(v[0] for v in prof.values())
    kernels = {}
    for k, (kms, cnt) in prof.items():
        if cnt == 0:
            continue
        ent = {"ms_per_step": kms / args.steps, "launches_per_step": cnt / args.steps,
               "share": kms / total_kernel_ms if total_kernel_ms > 0 else None}
        if k in flops_kind and kms > 0:
            ent["tflops"] = flops_kind[k] * args.steps / (kms / 1e3) / 1e12
        if k in bytes_kind and kms > 0:
            ent["gbs"] = bytes_kind[k] * args.steps / (kms / 1e3) / 1e9
        kernels[k] = ent
    dom = max(flops_kind, key=lambda k: prof[k][0])
    R = rg.grpo_chunk_rows(shape)
    n_chunks_work = (n_valid + R - 1) // R
    dom_ms, _ = prof[dom]
    sustained = pk.get("bf16_tflops_sustained", FALLBACK_PEAKS["bf16_tflops_sustained"])
    achieved = flops_kind[dom] * args.steps / (dom_ms / 1e3) / 1e12
    roofline = {"kernel": dom, "bound": "tensor", "achieved": achieved, "peak": sustained, "unit": "TFLOP/s",
                "frac": achieved / sustained, "peak_kind": f"bf16 dense sustained, {pk_kind}",
                "traffic": ncu_traffic(dom, rg.grpo_chunk_rows(shape)),
                "traffic_spread": ncu_traffic(dom, rg.grpo_chunk_rows(shape), "spread"),
                "traffic_per": "full chunk launch (ncu DRAM read+write bytes, median of captures in separate processes)",
                # per full chunk of R rows, like traffic: its algorithmic flops, and the kernel's
                # time per R rows (empty chunk slots exit at once and add nothing)
                "rows_per_launch": R, "launches_with_rows": n_chunks_work,
                "flops_per_launch": flops_kind[dom] / n_valid * R,
                "ms_per_launch": dom_ms / args.steps / n_valid * R}
    useful = 8.0 * n_valid * V * d
    t_step = ms_step / 1e3
    burst = pk.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"])
    useful_tf = useful / t_step / 1e12
    # the measured GEMM peaks were taken at their own clock under the power cap;
    # scaled to this run's median SM clock they compare like with like
    peak_mhz = (pk.get("clocks_under_load") or {}).get("sm_mhz_median")
    run_mhz = clocks["sm_mhz"] if clocks else None
    at_clock = (useful_tf / sustained * peak_mhz / run_mhz) if (peak_mhz and run_mhz) else None

    cpu = None
    if ranks.rank == 0 and ranks.world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(cfg, wl, args)

    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": ranks.world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": cfg.dtype, "data": "synthetic (seeded generator; random-init head)",
        "config": cfg_dict(cfg, {"n_valid": n_valid, "chunk_rows": rg.grpo_chunk_rows(shape),
                                 "loss_scale": scale[0]}),
        "pct_bf16_peak": {"useful_tflops": useful_tf,
                          "of_datasheet_dense": useful_tf / DATASHEET_BF16_TFLOPS,
                          "of_burst": useful_tf / burst,
                          "of_sustained": useful_tf / sustained,
                          "of_sustained_at_equal_clock": at_clock,
                          "executed_tflops": useful_tf,
                          "peaks": f"datasheet dense bf16 {DATASHEET_BF16_TFLOPS:.0f} TFLOP/s; burst and sustained: "
                                   f"cuBLAS bf16 GEMM, {pk_kind}; at equal clock: sustained x its median SM clock "
                                   f"({peak_mhz} MHz) / this run's ({run_mhz} MHz)"},
        "cycles_per_step": (ms_step * run_mhz * 1e3) if run_mhz else None,
        "peak_extra_hbm_gb": max(peak_extra, 0) / 1e9 + ws_bytes / 1e9,
        "workspace_gb": ws_bytes / 1e9,
        "logits_not_materialised_gb": 2 * 2 * N * V / 1e9,
        "e2e": e2e,
        "graph": graph,
        "gpu_launches": int(launches),
        "kernels": kernels,
        "roofline": roofline,
        "cpu_baseline": cpu,
        "clocks": clocks,
        "loss": float(out["loss"].item()),
        "parallelism": ("data-parallel shards: one prompt group per rank, batch counts, loss shares and dW summed "
                        "over the ranks every step" if split else "replicas"),
        "split": bool(split),
    }
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)


def run_forward_modes(args, ranks):
    """Forward-only throughput: grpo_loss_fwd on bf16 inputs and grpo_loss_fwd_fp8 on
    the same workload quantised to e4m3 and to e5m2 (one scale per tensor); and
    forward+backward on the 8-bit inputs (grpo_loss_fwd_bwd_fp8)."""
    import numpy as np
    import torch

    import rl_fine_tuning_gb300 as rg
    import synth

    torch.cuda.set_device(ranks.local)
    rg.load(build_if_missing=True)
    cfg = synth.make_config(args.config)
    n_valid = int(np.minimum(np.maximum(synth.lengths_for(cfg, 0), 0), cfg.L).sum())
    stream = torch.cuda.current_stream()
    out = {}
    for mode in ("bf16", "e4m3", "e5m2"):
        if mode == "bf16":
            wl = synth.generate(cfg, seed=0)
            mats = [torch.from_numpy(a.view(np.int16)).cuda().view(torch.bfloat16) for a in (wl.h_pol, wl.h_ref, wl.W)]
            shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V, rg.BF16, beta=cfg.beta, eps=cfg.eps,
                                  chunk_rows=args.chunk_rows)
        else:
            wl = synth.generate_fp8(cfg, seed=0, fmt=mode)
            mats = [torch.from_numpy(a).cuda() for a in (wl.h_pol, wl.h_ref, wl.W)]
            shape = rg.make_shape(cfg.n_groups, cfg.G, cfg.L, cfg.d, cfg.V, rg.E4M3 if mode == "e4m3" else rg.E5M2,
                                  beta=cfg.beta, eps=cfg.eps, chunk_rows=args.chunk_rows)
        tokens, lengths, rewards = (torch.from_numpy(a).cuda() for a in (wl.tokens, wl.lengths, wl.rewards))
        adv = torch.empty(cfg.n_seq, dtype=torch.float32, device="cuda")
        mask = torch.empty(cfg.N, dtype=torch.uint8, device="cuda")
        ws = torch.empty(rg.grpo_workspace_bytes(shape), dtype=torch.uint8, device="cuda")
        loss = torch.zeros(1, dtype=torch.float32, device="cuda")
        status = torch.zeros(1, dtype=torch.int32, device="cuda")

        def step():
            rg.grpo_group_advantages(rewards, cfg.n_groups, cfg.G, cfg.eps, True, adv)
            rg.grpo_build_mask(lengths, shape, mask)
            if mode == "bf16":
                rg.grpo_loss_fwd(*mats, tokens, mask, adv, shape, ws, loss, None, status)
            else:
                rg.grpo_loss_fwd_fp8(*mats, *wl.extra["scales"], tokens, mask, adv, shape, ws, loss, None, status)

        for _ in range(max(args.warmup, 1)):
            step()
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise SystemExit(f"device status {int(status.item())}")
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.steps):
            step()
        e1.record(stream)
        torch.cuda.synchronize()
        ms = e0.elapsed_time(e1) / args.steps
        flops = 4.0 * n_valid * cfg.V * cfg.d
        out[mode] = {"ms_per_step": ms, "tokens_per_s": n_valid / (ms / 1e3), "tflops": flops / (ms / 1e3) / 1e12,
                     "loss": float(loss.item())}
        if mode != "bf16":
            # the 8-bit forward+backward on the same inputs (dH bf16, dW fp32)
            dH = torch.empty((cfg.N, cfg.d), dtype=torch.bfloat16, device="cuda")
            dW = torch.empty((cfg.V, cfg.d), dtype=torch.float32, device="cuda")

            def step_bwd():
                rg.grpo_group_advantages(rewards, cfg.n_groups, cfg.G, cfg.eps, True, adv)
                rg.grpo_build_mask(lengths, shape, mask)
                rg.grpo_loss_fwd_bwd_fp8(*mats, *wl.extra["scales"], tokens, mask, adv, shape, ws, loss, dH, dW,
                                         None, status)

            for _ in range(max(args.warmup, 1)):
                step_bwd()
            torch.cuda.synchronize()
            if int(status.item()) != 0:
                raise SystemExit(f"device status {int(status.item())}")
            e0.record(stream)
            for _ in range(args.steps):
                step_bwd()
            e1.record(stream)
            torch.cuda.synchronize()
            ms = e0.elapsed_time(e1) / args.steps
            flops = 8.0 * n_valid * cfg.V * cfg.d
            # per-kernel breakdown from a second, instrumented pass
            rg.grpo_profile_enable(True)
            for _ in range(args.steps):
                step_bwd()
            torch.cuda.synchronize()
            rg.grpo_profile_enable(False)
            kern = {k: round(v[0] / args.steps, 3) for k, v in rg.grpo_profile_collect().items() if v[1]}
            out[mode + "_fwd_bwd"] = {"ms_per_step": ms, "tokens_per_s": n_valid / (ms / 1e3),
                                      "tflops": flops / (ms / 1e3) / 1e12, "loss": float(loss.item()),
                                      "kernel_ms_per_step": kern}
            del dH, dW
        del mats, ws, wl
        torch.cuda.empty_cache()
    pk, pk_kind = peaks()
    line = {"metric": "GRPO loss forward tokens/s (bf16, e4m3 and e5m2 inputs)", "value": out["e4m3"]["tokens_per_s"],
            "unit": "tokens/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": out["e4m3"]["ms_per_step"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "e4m3", "data": "synthetic", "config": cfg_dict(cfg, {"n_valid": n_valid}),
            "forward": out, "bf16_peak_tflops": pk.get("bf16_tflops"), "peaks": pk_kind}
    if ranks.rank == 0:
        print(json.dumps(line), flush=True)


def cpu_baseline(cfg, wl, args):
    """The oracle, as it stands, on the host cores: a bounded sample of rows."""
    import oracle
    oracle.build()
    adv = oracle.group_advantages(wl.rewards, cfg.n_groups, cfg.G, cfg.eps, True)
    valid = oracle.valid_rows(oracle.build_mask(wl.lengths, cfg.L))
    cal = sample_rows(valid, max(1, oracle.max_threads()), 12345)
    t_cal = oracle_sample(cfg, wl, cal, adv)
    n = max(1, int(args.cpu_seconds / (t_cal / cal.size)))
    rows = sample_rows(valid, n, 777)
    dt = oracle_sample(cfg, wl, rows, adv)
    return {"value": rows.size / dt, "unit": "tokens/s", "cores": oracle.max_threads(), "kind": "oracle",
            "sample": f"{rows.size} seeded valid rows of {cfg.name}: per-row lse/q/p/KL, dH and dW "
                      f"contribution in fp64 ({dt:.1f} s)"}


def main():
    args = parse()
    ranks = Ranks(args.gpus, split=args.split and args.impl == "ours")
    try:
        if args.impl == "reference":
            run_reference(args, ranks)
        elif args.forward:
            run_forward_modes(args, ranks)
        else:
            run_ours(args, ranks)
    finally:
        ranks.close()


if __name__ == "__main__":
    main()
