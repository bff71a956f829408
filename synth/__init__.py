"""Seeded synthetic workloads for the fused GRPO loss.

Holds no arithmetic of the loss: it draws hidden states, the lm_head weight,
sampled tokens, completion lengths and rewards from a counter-based
splitmix64 generator (``synth.c``) and rounds fp32 to bf16/fp16 storage.
Both the CPU oracle and the GPU path take their inputs from here.

Workload shapes follow the model heads the GRPO pages talk about: the
Llama 3.1 8B run at 20K context with 8 generations per prompt and a
128256-entry vocabulary ("Long-context GRPO", section 2), plus the Qwen2.5
1.5B and Phi-4 heads those pages train GRPO notebooks on.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass, field

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "libsynth.so")

# generator streams
S_HPOL, S_REFNOISE, S_W, S_TOK, S_LEN, S_RBIT, S_RNOISE, S_MASKSEQ = 1, 2, 3, 4, 5, 6, 7, 8


def build(force: bool = False) -> str:
    src = os.path.join(_HERE, "synth.c")
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < os.path.getmtime(src):
        os.makedirs(_BUILD, exist_ok=True)
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               src, "-o", tmp, "-lm"])
        os.replace(tmp, _SO)
    return _SO


_lib = None


def _L():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        u64, i64, p = ctypes.c_uint64, ctypes.c_int64, ctypes.c_void_p
        lib.synth_u64.restype = u64
        lib.synth_u64.argtypes = [u64, u64, u64]
        lib.synth_normal_f32.argtypes = [u64, u64, u64, i64, ctypes.c_float, p, p]
        lib.synth_uniform_int.argtypes = [u64, u64, i64, i64, i64, p]
        lib.synth_bits.argtypes = [u64, u64, i64, p]
        lib.synth_permutation.argtypes = [u64, u64, ctypes.c_int32, p]
        lib.synth_to_bf16.argtypes = [p, i64, p]
        lib.synth_to_f16.argtypes = [p, i64, p]
        lib.synth_to_e4m3.argtypes = [p, i64, ctypes.c_float, p]
        lib.synth_to_e5m2.argtypes = [p, i64, ctypes.c_float, p]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def u64(seed: int, stream: int, i: int) -> int:
    return int(_L().synth_u64(seed, stream, i))


def normal_f32(seed, stream, n, sigma=1.0, base=None, offset=0):
    out = np.empty(n, np.float32)
    if base is not None:
        base = np.ascontiguousarray(base, np.float32).reshape(-1)
        assert base.size == n
    _L().synth_normal_f32(seed, stream, offset, n, sigma, None if base is None else _ptr(base), _ptr(out))
    return out


def uniform_int(seed, stream, n, lo, hi):
    out = np.empty(n, np.int32)
    _L().synth_uniform_int(seed, stream, n, lo, hi, _ptr(out))
    return out


def bits(seed, stream, n):
    out = np.empty(n, np.int32)
    _L().synth_bits(seed, stream, n, _ptr(out))
    return out


def permutation(seed, stream, n):
    out = np.empty(n, np.int32)
    _L().synth_permutation(seed, stream, n, _ptr(out))
    return out


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _L().synth_to_bf16(_ptr(x), x.size, _ptr(out))
    return out


def to_f16_bits(x: np.ndarray) -> np.ndarray:
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint16)
    _L().synth_to_f16(_ptr(x), x.size, _ptr(out))
    return out


E4M3_MAX = 448.0
E5M2_MAX = 57344.0
FP8_MAX = {"e4m3": E4M3_MAX, "e5m2": E5M2_MAX}


def fp8_scale(x: np.ndarray, fmt: str = "e4m3") -> float:
    """Per-tensor scale that maps max|x| onto the largest finite value of the format."""
    amax = float(np.max(np.abs(x))) if x.size else 0.0
    return float(np.float32(amax / FP8_MAX[fmt])) if amax > 0 else 1.0


def e4m3_scale(x: np.ndarray) -> float:
    return fp8_scale(x, "e4m3")


def to_fp8_bits(x: np.ndarray, scale: float, fmt: str = "e4m3") -> np.ndarray:
    """fp32 values x -> OCP FP8 codes of x / scale (round to nearest even, saturating)."""
    x = np.ascontiguousarray(x, np.float32)
    out = np.empty(x.shape, np.uint8)
    fn = {"e4m3": _L().synth_to_e4m3, "e5m2": _L().synth_to_e5m2}[fmt]
    fn(_ptr(x), x.size, scale, _ptr(out))
    return out


def to_e4m3_bits(x: np.ndarray, scale: float) -> np.ndarray:
    return to_fp8_bits(x, scale, "e4m3")


def bits_to_f32(b: np.ndarray, dtype: str) -> np.ndarray:
    """Exact widening of bf16/fp16 bit patterns to float32."""
    if dtype == "bf16":
        return (b.astype(np.uint32) << 16).view(np.float32)
    return b.view(np.float16).astype(np.float32)


@dataclass(frozen=True)
class Config:
    name: str
    G: int
    L: int
    d: int
    V: int
    dtype: str = "bf16"          # storage/compute type of H and W
    sigma_ref: float = 0.02      # h_ref = h_pol + N(0, sigma_ref^2)
    len_lo: int = 1
    len_hi: int = 1
    n_zero_seq: int = 0          # sequences forced to length 0 (fully masked)
    n_groups: int = 1
    loss_scale: float = 1.0      # initial loss scale (fp16 path)
    w_sigma: float = 0.02
    beta: float = 0.04
    eps: float = 1e-4

    @property
    def n_seq(self):
        return self.n_groups * self.G

    @property
    def N(self):
        return self.n_seq * self.L


CONFIGS = {
    c.name: c for c in [
        Config("tiny", G=4, L=64, d=128, V=1024, sigma_ref=0.05, len_lo=16, len_hi=64),
        Config("qwen2.5-1.5b-head", G=8, L=1024, d=1536, V=151936, sigma_ref=0.02, len_lo=256, len_hi=1024),
        Config("llama-3.1-8b-head", G=8, L=4096, d=4096, V=128256, sigma_ref=0.02, len_lo=1024, len_hi=4096),
        Config("llama-3.1-8b-20k", G=8, L=20000, d=4096, V=128256, sigma_ref=0.02, len_lo=5000, len_hi=20000),
        Config("phi-4-14b-head-fp16", G=8, L=8192, d=5120, V=100352, dtype="fp16", sigma_ref=0.05,
               len_lo=512, len_hi=8192, n_zero_seq=2, loss_scale=2.0 ** 15),
    ]
}
CONFIG_ORDER = list(CONFIGS)


def make_config(name: str, **over) -> Config:
    from dataclasses import replace
    return replace(CONFIGS[name], **over) if over else CONFIGS[name]


@dataclass
class Workload:
    cfg: Config
    h_pol: np.ndarray            # [N, d] uint16 bits (bf16 or fp16)
    h_ref: np.ndarray            # [N, d] uint16 bits
    W: np.ndarray                # [V, d] uint16 bits
    tokens: np.ndarray           # [N] int32
    lengths: np.ndarray          # [n_seq] int32
    rewards: np.ndarray          # [n_seq] float32
    extra: dict = field(default_factory=dict)


def lengths_for(cfg: Config, seed: int = 0) -> np.ndarray:
    lens = uniform_int(seed, S_LEN, cfg.n_seq, cfg.len_lo, cfg.len_hi)
    if cfg.n_zero_seq:
        perm = permutation(seed, S_MASKSEQ, cfg.n_seq)
        lens[perm[:cfg.n_zero_seq]] = 0
    return lens


def rewards_for(cfg: Config, seed: int = 0) -> np.ndarray:
    b = bits(seed, S_RBIT, cfg.n_seq).astype(np.float32)
    return (b + normal_f32(seed, S_RNOISE, cfg.n_seq, 0.1)).astype(np.float32)


def generate_fp8(cfg: Config, seed: int = 0, fmt: str = "e4m3") -> Workload:
    """The workload of `generate` quantised to an OCP FP8 format ("e4m3" or
    "e5m2") with one scale per tensor.

    h_pol / h_ref / W hold the codes (uint8); extra["scales"] = (s_pol, s_ref, s_w)
    with value = decode(code) * scale, extra["fp8"] = fmt.  The reference rows
    are formed from the unrounded policy rows, as in `generate`."""
    N, d, V = cfg.N, cfg.d, cfg.V
    h32 = normal_f32(seed, S_HPOL, N * d, 1.0)
    r32 = normal_f32(seed, S_REFNOISE, N * d, cfg.sigma_ref, base=h32)
    w32 = normal_f32(seed, S_W, V * d, cfg.w_sigma)
    s_pol, s_ref, s_w = fp8_scale(h32, fmt), fp8_scale(r32, fmt), fp8_scale(w32, fmt)
    wl = Workload(cfg, to_fp8_bits(h32, s_pol, fmt).reshape(N, d), to_fp8_bits(r32, s_ref, fmt).reshape(N, d),
                  to_fp8_bits(w32, s_w, fmt).reshape(V, d), uniform_int(seed, S_TOK, N, 0, V - 1),
                  lengths_for(cfg, seed), rewards_for(cfg, seed))
    wl.extra["scales"] = (s_pol, s_ref, s_w)
    wl.extra["fp8"] = fmt
    return wl


def generate_e4m3(cfg: Config, seed: int = 0) -> Workload:
    return generate_fp8(cfg, seed, "e4m3")


def generate(cfg: Config, seed: int = 0, with_w: bool = True) -> Workload:
    N, d, V = cfg.N, cfg.d, cfg.V
    rnd = to_bf16_bits if cfg.dtype == "bf16" else to_f16_bits
    h32 = normal_f32(seed, S_HPOL, N * d, 1.0)
    h_pol = rnd(h32).reshape(N, d)
    h_ref = rnd(normal_f32(seed, S_REFNOISE, N * d, cfg.sigma_ref, base=h32)).reshape(N, d)
    del h32
    W = rnd(normal_f32(seed, S_W, V * d, cfg.w_sigma)).reshape(V, d) if with_w else None
    tokens = uniform_int(seed, S_TOK, N, 0, V - 1)
    return Workload(cfg, h_pol, h_ref, W, tokens, lengths_for(cfg, seed), rewards_for(cfg, seed))



def split_groups(wl: Workload, n_shards: int) -> list:
    """The workload cut into n_shards consecutive runs of whole prompt groups
    (the data-parallel split): shard r holds groups [r*g, (r+1)*g) with
    g = n_groups / n_shards, i.e. their rows, tokens, lengths and rewards;
    every shard keeps the whole W."""
    from dataclasses import replace
    cfg = wl.cfg
    assert cfg.n_groups % n_shards == 0, "shards hold whole prompt groups"
    g = cfg.n_groups // n_shards
    scfg = replace(cfg, n_groups=g)
    rows, seqs = scfg.N, scfg.n_seq
    out = []
    for r in range(n_shards):
        rs, ss = slice(r * rows, (r + 1) * rows), slice(r * seqs, (r + 1) * seqs)
        out.append(Workload(scfg, np.ascontiguousarray(wl.h_pol[rs]), np.ascontiguousarray(wl.h_ref[rs]), wl.W,
                            np.ascontiguousarray(wl.tokens[rs]), np.ascontiguousarray(wl.lengths[ss]),
                            np.ascontiguousarray(wl.rewards[ss]), dict(wl.extra)))
    return out
