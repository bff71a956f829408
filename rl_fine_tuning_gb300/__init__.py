"""Python binding of libgrpo, the fused linear GRPO loss for GB300 (sm_103a).

Argument marshalling only: every function forwards to the C entry point of
the same name in libgrpo.so, whose kernels do all the work.  Tensors are
torch CUDA tensors (only their device pointers are passed); the stream
defaults to torch's current stream.  A nonzero return code raises
GrpoError.  There is no CPU fallback: importing the binding without the
built library raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

__all__ = [
    "GrpoError", "GrpoShape", "BF16", "FP16", "E4M3", "E5M2", "TOKEN_MEAN", "SEQUENCE_MEAN", "OBJECTIVES", "load",
    "make_shape", "grpo_workspace_bytes", "grpo_chunk_rows", "grpo_group_advantages", "grpo_build_mask",
    "grpo_valid_rows", "grpo_loss_fwd", "grpo_loss_fwd_bwd", "grpo_loss_fwd_fp8", "grpo_loss_fwd_noalloc",
    "grpo_shard_counts", "grpo_loss_fwd_shard", "grpo_loss_fwd_bwd_shard", "grpo_loss_fwd_bwd_fp8",
    "grpo_status_string", "grpo_version", "library_path", "grpo_profile_enable", "grpo_profile_collect",
    "grpo_kernel_launches", "grpo_device_checks", "grpo_selftest_bounds_check", "grpo_selftest_wait_timeout",
    "PROF_KINDS",
]

# kernel kinds of the diagnostics interface, in the order of the GRPO_PROF_* enum
PROF_KINDS = ("advantages", "mask", "index", "fwd", "merge", "clear", "gather", "dlogits", "dh", "dw", "f8_prep")

BF16, FP16, E4M3, E5M2 = 0, 1, 2, 3
TOKEN_MEAN, SEQUENCE_MEAN = 0, 1
OBJECTIVES = {"grpo": 0, "no_detach": 1, "reverse_kl_q": 2, "forward_kl": 3}


class GrpoError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"libgrpo {what} failed: {code} ({_status_string(code)})")


class GrpoShape(ctypes.Structure):
    """Mirror of grpo_shape in include/grpo.h."""
    _fields_ = [
        ("n_groups", ctypes.c_int), ("G", ctypes.c_int), ("L", ctypes.c_int), ("d", ctypes.c_int),
        ("V", ctypes.c_int), ("dtype", ctypes.c_int), ("beta", ctypes.c_float), ("eps", ctypes.c_float),
        ("std_unbiased", ctypes.c_int), ("chunk_rows", ctypes.c_int), ("loss_mode", ctypes.c_int),
        ("objective", ctypes.c_int),
    ]

    @property
    def N(self) -> int:
        return self.n_groups * self.G * self.L


_lib = None


def library_path() -> str:
    return _build.LIB


def load(build_if_missing: bool = False):
    """The loaded libgrpo.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    path = _build.LIB
    if build_if_missing:
        path = _build.build()
    if not os.path.exists(path):
        raise ImportError(f"libgrpo.so is not built ({path}); run `python -m rl_fine_tuning_gb300.build`")
    lib = ctypes.CDLL(path)
    _declare(lib)
    _lib = lib
    return lib


def _declare(lib):
    """Argument and result types of every entry point of include/grpo.h."""
    p, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t, ctypes.c_float
    sp = ctypes.POINTER(GrpoShape)
    sigs = {
        "grpo_shape_init": ([sp, i32, i32, i32, i32, i32, i32], None),
        "grpo_workspace_bytes": ([sp], sz),
        "grpo_chunk_rows": ([sp], i32),
        "grpo_group_advantages": ([p, i32, i32, f32, i32, p, p], i32),
        "grpo_build_mask": ([p, sp, p, p], i32),
        "grpo_valid_rows": ([p, sp, p, p, p, sz, p], i32),
        "grpo_loss_fwd": ([p, p, p, p, p, p, sp, p, sz, p, p, p, p], i32),
        "grpo_loss_fwd_bwd": ([p, p, p, p, p, p, sp, f32, p, sz, p, p, p, p, p, p, p], i32),
        "grpo_loss_fwd_fp8": ([p, p, p, f32, f32, f32, p, p, p, sp, p, sz, p, p, p, p], i32),
        "grpo_loss_fwd_bwd_fp8": ([p, p, p, f32, f32, f32, p, p, p, sp, p, sz, p, p, p, p, p, p], i32),
        "grpo_loss_fwd_noalloc": ([p, p, p, p, p, p, sp, p, p, p, p], i32),
        "grpo_shard_counts": ([p, sp, p, p], i32),
        "grpo_loss_fwd_shard": ([p, p, p, p, p, p, sp, p, p, sz, p, p, p, p], i32),
        "grpo_loss_fwd_bwd_shard": ([p, p, p, p, p, p, sp, p, f32, p, sz, p, p, p, p, p, p, p], i32),
        "grpo_profile_enable": ([i32], i32),
        "grpo_profile_collect": ([ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_longlong), i32], i32),
        "grpo_kernel_launches": ([], ctypes.c_ulonglong),
        "grpo_device_checks": ([], i32),
        "grpo_selftest_bounds_check": ([p, p], i32),
        "grpo_selftest_wait_timeout": ([p, p, p], i32),
        "grpo_status_string": ([i32], ctypes.c_char_p),
        "grpo_version": ([], i32),
    }
    for name, (args, res) in sigs.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res


def _status_string(code: int) -> str:
    try:
        return load().grpo_status_string(int(code)).decode()
    except Exception:
        return "?"


def _ptr(x):
    if x is None:
        return None
    if isinstance(x, int):
        return ctypes.c_void_p(x)
    return ctypes.c_void_p(x.data_ptr())


def _nbytes(x) -> int:
    return x.numel() * x.element_size()


def _stream(stream):
    if stream is None:
        import torch
        return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return ctypes.c_void_p(stream)
    return ctypes.c_void_p(stream.cuda_stream)


def _check(code: int, what: str):
    if code != 0:
        raise GrpoError(code, what)


def make_shape(n_groups, G, L, d, V, dtype=BF16, beta=0.04, eps=1e-4, std_unbiased=True, chunk_rows=0,
               loss_mode=TOKEN_MEAN, objective=0):
    s = GrpoShape()
    load().grpo_shape_init(ctypes.byref(s), n_groups, G, L, d, V, dtype)
    s.beta, s.eps, s.std_unbiased, s.chunk_rows = beta, eps, int(bool(std_unbiased)), chunk_rows
    s.loss_mode = int(loss_mode)
    s.objective = OBJECTIVES[objective] if isinstance(objective, str) else int(objective)
    return s


def grpo_workspace_bytes(shape: GrpoShape) -> int:
    return int(load().grpo_workspace_bytes(ctypes.byref(shape)))


def grpo_chunk_rows(shape: GrpoShape) -> int:
    return int(load().grpo_chunk_rows(ctypes.byref(shape)))


def grpo_group_advantages(rewards, n_groups, G, eps, std_unbiased, adv_out, stream=None):
    _check(load().grpo_group_advantages(_ptr(rewards), n_groups, G, eps, int(bool(std_unbiased)), _ptr(adv_out),
                                        _stream(stream)), "grpo_group_advantages")


def grpo_build_mask(lengths, shape, mask_out, stream=None):
    _check(load().grpo_build_mask(_ptr(lengths), ctypes.byref(shape), _ptr(mask_out), _stream(stream)),
           "grpo_build_mask")


def grpo_valid_rows(mask, shape, rows_out, n_valid_out, workspace, stream=None):
    _check(load().grpo_valid_rows(_ptr(mask), ctypes.byref(shape), _ptr(rows_out), _ptr(n_valid_out),
                                  _ptr(workspace), _nbytes(workspace), _stream(stream)), "grpo_valid_rows")


def grpo_loss_fwd(h_pol, h_ref, W, tokens, mask, adv, shape, workspace, loss_out, row_stats, status,
                  stream=None):
    _check(load().grpo_loss_fwd(_ptr(h_pol), _ptr(h_ref), _ptr(W), _ptr(tokens), _ptr(mask), _ptr(adv),
                                ctypes.byref(shape), _ptr(workspace), _nbytes(workspace), _ptr(loss_out),
                                _ptr(row_stats), _ptr(status), _stream(stream)), "grpo_loss_fwd")


def grpo_loss_fwd_bwd(h_pol, h_ref, W, tokens, mask, adv, shape, loss_scale, workspace, loss_out, dH, dW,
                      found_inf, row_stats, status, stream=None):
    _check(load().grpo_loss_fwd_bwd(_ptr(h_pol), _ptr(h_ref), _ptr(W), _ptr(tokens), _ptr(mask), _ptr(adv),
                                    ctypes.byref(shape), float(loss_scale), _ptr(workspace), _nbytes(workspace),
                                    _ptr(loss_out), _ptr(dH), _ptr(dW), _ptr(found_inf), _ptr(row_stats),
                                    _ptr(status), _stream(stream)), "grpo_loss_fwd_bwd")


def grpo_shard_counts(mask, shape, counts_out, stream=None):
    _check(load().grpo_shard_counts(_ptr(mask), ctypes.byref(shape), _ptr(counts_out), _stream(stream)),
           "grpo_shard_counts")


def grpo_loss_fwd_shard(h_pol, h_ref, W, tokens, mask, adv, shape, global_counts, workspace, loss_out, row_stats,
                        status, stream=None):
    _check(load().grpo_loss_fwd_shard(_ptr(h_pol), _ptr(h_ref), _ptr(W), _ptr(tokens), _ptr(mask), _ptr(adv),
                                      ctypes.byref(shape), _ptr(global_counts), _ptr(workspace), _nbytes(workspace),
                                      _ptr(loss_out), _ptr(row_stats), _ptr(status), _stream(stream)),
           "grpo_loss_fwd_shard")


def grpo_loss_fwd_bwd_shard(h_pol, h_ref, W, tokens, mask, adv, shape, global_counts, loss_scale, workspace,
                            loss_out, dH, dW, found_inf, row_stats, status, stream=None):
    _check(load().grpo_loss_fwd_bwd_shard(_ptr(h_pol), _ptr(h_ref), _ptr(W), _ptr(tokens), _ptr(mask), _ptr(adv),
                                          ctypes.byref(shape), _ptr(global_counts), float(loss_scale),
                                          _ptr(workspace), _nbytes(workspace), _ptr(loss_out), _ptr(dH), _ptr(dW),
                                          _ptr(found_inf), _ptr(row_stats), _ptr(status), _stream(stream)),
           "grpo_loss_fwd_bwd_shard")


def grpo_status_string(code: int) -> str:
    return _status_string(code)


def grpo_version() -> int:
    return int(load().grpo_version())


def grpo_profile_enable(on: bool = True):
    _check(load().grpo_profile_enable(int(bool(on))), "grpo_profile_enable")


def grpo_profile_collect() -> dict:
    """{kind: (milliseconds, launches)} accumulated since the last collect."""
    n = len(PROF_KINDS)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_longlong * n)()
    _check(load().grpo_profile_collect(ms, cnt, n), "grpo_profile_collect")
    return {k: (float(ms[i]), int(cnt[i])) for i, k in enumerate(PROF_KINDS)}


def grpo_kernel_launches() -> int:
    return int(load().grpo_kernel_launches())


def grpo_loss_fwd_noalloc(h_pol, h_ref, W, tokens, mask, adv, shape, loss_out, row_stats, status, stream=None):
    """grpo_loss_fwd on the library's own fixed scratch array (no workspace argument)."""
    _check(load().grpo_loss_fwd_noalloc(_ptr(h_pol), _ptr(h_ref), _ptr(W), _ptr(tokens), _ptr(mask), _ptr(adv),
                                        ctypes.byref(shape), _ptr(loss_out), _ptr(row_stats), _ptr(status),
                                        _stream(stream)), "grpo_loss_fwd_noalloc")


def grpo_loss_fwd_fp8(h_pol, h_ref, W, scale_h_pol, scale_h_ref, scale_w, tokens, mask, adv, shape, workspace,
                      loss_out, row_stats, status, stream=None):
    _check(load().grpo_loss_fwd_fp8(_ptr(h_pol), _ptr(h_ref), _ptr(W), float(scale_h_pol), float(scale_h_ref),
                                    float(scale_w), _ptr(tokens), _ptr(mask), _ptr(adv), ctypes.byref(shape),
                                    _ptr(workspace), _nbytes(workspace), _ptr(loss_out), _ptr(row_stats),
                                    _ptr(status), _stream(stream)), "grpo_loss_fwd_fp8")


def grpo_loss_fwd_bwd_fp8(h_pol, h_ref, W, scale_h_pol, scale_h_ref, scale_w, tokens, mask, adv, shape, workspace,
                          loss_out, dH, dW, row_stats, status, stream=None):
    _check(load().grpo_loss_fwd_bwd_fp8(_ptr(h_pol), _ptr(h_ref), _ptr(W), float(scale_h_pol), float(scale_h_ref),
                                        float(scale_w), _ptr(tokens), _ptr(mask), _ptr(adv), ctypes.byref(shape),
                                        _ptr(workspace), _nbytes(workspace), _ptr(loss_out), _ptr(dH), _ptr(dW),
                                        _ptr(row_stats), _ptr(status), _stream(stream)), "grpo_loss_fwd_bwd_fp8")


def grpo_device_checks() -> bool:
    """True when the loaded library is the build with device-side index checks."""
    return bool(load().grpo_device_checks())


def grpo_selftest_bounds_check(status, stream=None):
    _check(load().grpo_selftest_bounds_check(_ptr(status), _stream(stream)), "grpo_selftest_bounds_check")


def grpo_selftest_wait_timeout(status, waited_ns, stream=None):
    _check(load().grpo_selftest_wait_timeout(_ptr(status), _ptr(waited_ns), _stream(stream)),
           "grpo_selftest_wait_timeout")
