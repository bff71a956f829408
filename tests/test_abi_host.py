"""Host-side checks of libgrpo that need no GPU: the library loads, exports
every function include/grpo.h declares, agrees with the binding on the shape
struct, sizes its workspace, and rejects bad arguments before any launch."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "grpo.h")


@pytest.fixture(scope="module")
def lib():
    from rl_fine_tuning_gb300 import build
    build.build()
    import rl_fine_tuning_gb300 as rg
    return rg.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(grpo_[a-z0-9_]+)\s*\(", src)))


def test_every_declared_symbol_is_exported(lib):
    names = declared_functions()
    assert len(names) >= 12
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (grpo_\w+)", out))
    assert set(names) <= exported


def declared_parameter_counts():
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    counts = {}
    for name, params in re.findall(r"\b(grpo_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", src):
        params = params.strip()
        counts[name] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_declares_every_entry_point_with_the_header_arity(lib):
    counts = declared_parameter_counts()
    assert set(counts) == set(declared_functions())
    for name, n in counts.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, name
        assert len(fn.argtypes) == n, (name, len(fn.argtypes), n)


def test_checked_build_exports_the_same_symbols_and_says_so(lib):
    from rl_fine_tuning_gb300 import build
    names = declared_functions()
    checked = ctypes.CDLL(build.LIB_CHECKED)
    assert not [n for n in names if not hasattr(checked, n)]
    assert checked.grpo_device_checks() == 1 and lib.grpo_device_checks() == 0
    P = 1 << 20
    assert lib.grpo_selftest_bounds_check(None, None) == 1
    assert lib.grpo_selftest_bounds_check(ctypes.c_void_p(P), None) == 7      # normal build: nothing launched
    assert checked.grpo_selftest_bounds_check(None, None) == 1


def test_shape_struct_layout_matches_binding(tmp_path):
    import rl_fine_tuning_gb300 as rg
    prog = tmp_path / "sz.c"
    prog.write_text('#include <stdio.h>\n#include <stddef.h>\n#include "grpo.h"\n'
                    'int main(void){printf("%zu", sizeof(grpo_shape));'
                    'const char* n[]={"n_groups","G","L","d","V","dtype","beta","eps","std_unbiased","chunk_rows",'
                    '"loss_mode","objective"};'
                    'size_t o[]={offsetof(grpo_shape,n_groups),offsetof(grpo_shape,G),offsetof(grpo_shape,L),'
                    'offsetof(grpo_shape,d),offsetof(grpo_shape,V),offsetof(grpo_shape,dtype),'
                    'offsetof(grpo_shape,beta),offsetof(grpo_shape,eps),offsetof(grpo_shape,std_unbiased),'
                    'offsetof(grpo_shape,chunk_rows),offsetof(grpo_shape,loss_mode),offsetof(grpo_shape,objective)};'
                    'for(int i=0;i<12;i++)printf(" %s=%zu",n[i],o[i]);return 0;}\n')
    exe = tmp_path / "sz"
    subprocess.check_call(["gcc", "-I" + os.path.join(ROOT, "include"), str(prog), "-o", str(exe)])
    out = subprocess.check_output([str(exe)], text=True).split()
    assert int(out[0]) == ctypes.sizeof(rg.GrpoShape)
    for item in out[1:]:
        k, v = item.split("=")
        assert getattr(rg.GrpoShape, k).offset == int(v), k


def test_shape_defaults_and_workspace_bytes(lib):
    import rl_fine_tuning_gb300 as rg
    s = rg.make_shape(1, 8, 20000, 4096, 128256)
    assert (s.beta, s.std_unbiased, s.chunk_rows) == (pytest.approx(0.04), 1, 0)
    assert s.eps == pytest.approx(1e-4)
    n = rg.grpo_workspace_bytes(s)
    N, R, V, d = 160000, 38 * 128, 128256, 4096
    assert rg.grpo_chunk_rows(s) == R      # d/256 = 16: 19 tile pairs x 16 d tiles = 4 x 76 dH units
    # O(R*V + R*d + N) -- never O(N*V): dlogits chunk, three compact hidden-state chunks (policy,
    # reference, policy transposed), per-32-column maxima, per-split partials, per-row arrays
    assert R * V * 2 <= n < R * V * 2 + 3 * R * d * 2 + R * ((V + 31) // 32) * 4 + R * 256 * 16 + 300 * N + (1 << 20)
    assert n < 2 * 2 * N * V // 50          # > 50x below the two logit tensors
    s2 = rg.make_shape(1, 8, 20000, 4096, 128256, chunk_rows=4096)
    assert rg.grpo_workspace_bytes(s2) < n and rg.grpo_chunk_rows(s2) == 4096
    assert rg.grpo_chunk_rows(rg.make_shape(1, 8, 4096, 1536, 151936)) == 76 * 128   # 6 d tiles: 76 tiles balance
    assert rg.grpo_chunk_rows(rg.make_shape(1, 8, 8192, 5120, 100352)) == 38 * 128
    assert rg.grpo_chunk_rows(rg.make_shape(1, 8, 20000, 4096, 128256, chunk_rows=100)) == 128
    assert rg.grpo_chunk_rows(rg.make_shape(1, 4, 64, 128, 1024)) == 256            # capped at N
    assert rg.grpo_chunk_rows(rg.make_shape(1, 8, 20000, 100, 128256)) == 0         # invalid shape
    V_pad, nc32 = (V + 63) // 64 * 64, ((V + 31) // 32 + 7) // 8 * 8
    R8 = 76 * 128                            # 8-bit shapes default to 76-tile chunks
    n76 = rg.grpo_workspace_bytes(rg.make_shape(1, 8, 20000, 4096, 128256, chunk_rows=R8))
    for fp8 in (rg.E4M3, rg.E5M2):          # the 16-bit layout plus the 8-bit backward's buffers
        s8 = rg.make_shape(1, 8, 20000, 4096, 128256, fp8)
        assert rg.grpo_chunk_rows(s8) == R8
        n8 = rg.grpo_workspace_bytes(s8)
        # two code buffers, row maxima, group scales, keys, first key of each token
        max_chunks = (N + R8 - 1) // R8
        extra = 2 * R8 * V_pad + 4 * N + 4 * nc32 + 8 * max_chunks * R8 + 4 * V
        assert n76 + extra <= n8 <= n76 + extra + 6 * 256
    for bad in (dict(d=100), dict(d=0), dict(V=0), dict(G=0), dict(L=0)):
        b = rg.make_shape(1, 8, 20000, 4096, 128256)
        for k, v in bad.items():
            setattr(b, k, v)
        assert rg.grpo_workspace_bytes(b) == 0, bad


def test_validation_codes_without_a_device(lib):
    """Argument errors come back as status codes before anything touches a GPU."""
    import rl_fine_tuning_gb300 as rg
    s = rg.make_shape(1, 4, 64, 128, 1024)
    need = rg.grpo_workspace_bytes(s)
    P = 1 << 20                         # a 256-byte aligned stand-in address, never dereferenced
    f = lib.grpo_loss_fwd
    args = [P, P, P, P, P, P, ctypes.byref(s), P, need, P, None, P, None]
    assert f(*args[:7], None, need, *args[9:]) == 1                      # null workspace
    assert f(*args[:7], P + 8, need, *args[9:]) == 1                     # misaligned workspace
    assert f(P + 2, *args[1:]) == 1                                      # misaligned h_pol
    assert f(*args[:7], P, need - 1, *args[9:]) == 3                     # workspace too small
    bad = rg.make_shape(1, 4, 64, 100, 1024)
    assert f(*args[:6], ctypes.byref(bad), *args[7:]) == 2               # d not a multiple of 64
    bad.dtype = 7
    assert f(*args[:6], ctypes.byref(bad), *args[7:]) == 5               # unknown dtype
    for fp8 in (rg.E4M3, rg.E5M2):                                       # 8-bit codes: grpo_loss_fwd_fp8 only
        b8 = rg.make_shape(1, 4, 64, 128, 1024, fp8)
        assert f(*args[:6], ctypes.byref(b8), *args[7:]) == 5
    for field, val in (("loss_mode", 2), ("objective", 4), ("objective", -1)):
        b2 = rg.make_shape(1, 4, 64, 128, 1024)
        setattr(b2, field, val)
        assert f(*args[:6], ctypes.byref(b2), *args[7:]) == 2, field     # unknown mode / objective
    assert lib.grpo_group_advantages(P, 0, 4, ctypes.c_float(1e-4), 1, P, None) == 2
    assert lib.grpo_group_advantages(None, 1, 4, ctypes.c_float(1e-4), 1, P, None) == 1
    fb = lib.grpo_loss_fwd_bwd
    assert fb(P, P, P, P, P, P, ctypes.byref(s), ctypes.c_float(1.0), P, need, P, None, P, P, None, P, None) == 1
    assert fb(P, P, P, P, P, P, ctypes.byref(s), ctypes.c_float(1.0), P, need, P, P + 16, P, P, None, P, None) == 1
    assert fb(P, P, P, P, P, P, ctypes.byref(s), ctypes.c_float(1.0), P, need, P, P, P + 16, P, None, P, None) == 1
    assert fb(P, P, P, P, P, P, ctypes.byref(s), ctypes.c_float(0.0), P, need, P, P, P, P, None, P, None) == 2
    assert fb(P, P, P, P, P, P, ctypes.byref(s), ctypes.c_float(float("nan")), P, need, P, P, P, P, None, P,
              None) == 2


def test_validation_codes_of_the_added_entry_points_without_a_device(lib):
    """The shard and 8-bit backward entry points reject bad arguments before any launch."""
    import rl_fine_tuning_gb300 as rg
    P = 1 << 20
    s = rg.make_shape(1, 4, 64, 128, 1024)
    need = rg.grpo_workspace_bytes(s)
    one = ctypes.c_float(1.0)
    sh = lib.grpo_loss_fwd_bwd_shard
    assert sh(P, P, P, P, P, P, ctypes.byref(s), None, one, P, need, P, P, P, P, None, P, None) == 1   # no counts
    assert sh(P, P, P, P, P, P, ctypes.byref(s), P + 2, one, P, need, P, P, P, P, None, P, None) == 1  # misaligned
    assert sh(P, P, P, P, P, P, ctypes.byref(s), P, one, P, need - 1, P, P, P, P, None, P, None) == 3
    assert lib.grpo_loss_fwd_shard(P, P, P, P, P, P, ctypes.byref(s), None, P, need, P, None, P, None) == 1
    assert lib.grpo_shard_counts(P, ctypes.byref(s), None, None) == 1
    bad = rg.make_shape(1, 4, 64, 100, 1024)
    assert lib.grpo_shard_counts(P, ctypes.byref(bad), P, None) == 2
    f8 = lib.grpo_loss_fwd_bwd_fp8
    s8 = rg.make_shape(1, 4, 64, 128, 1024, rg.E4M3)
    n8 = rg.grpo_workspace_bytes(s8)
    assert n8 > need
    args = lambda shape, ws, dH=P, dW=P, scale=one: (P, P, P, scale, one, one, P, P, P, ctypes.byref(shape), P, ws,  # noqa: E731
                                                     P, dH, dW, None, P, None)
    assert f8(*args(s, need)) == 5                                       # 16-bit shape
    assert f8(*args(s8, n8 - 1)) == 3                                    # one byte short of the 8-bit layout
    assert f8(*args(s8, n8, dH=P + 16)) == 1                             # dH only 16-byte aligned
    assert f8(*args(s8, n8, dW=None)) == 1
    assert f8(*args(s8, n8, scale=ctypes.c_float(0.0))) == 2             # a scale must be positive
    b8 = rg.make_shape(1, 4, 64, 192, 1024, rg.E5M2)
    assert f8(*args(b8, rg.grpo_workspace_bytes(b8))) == 2               # d not a multiple of 128
    big = rg.make_shape(1, 8, 4096, 128, 1024, rg.E4M3, chunk_rows=16384 + 128)
    assert f8(*args(big, rg.grpo_workspace_bytes(big))) == 2             # chunks above the sort's 16384 rows


def test_status_strings_and_version(lib):
    import rl_fine_tuning_gb300 as rg
    assert rg.grpo_status_string(0) == "ok"
    assert "workspace" in rg.grpo_status_string(3)
    assert "timed out" in rg.grpo_status_string(6)
    assert "index check" in rg.grpo_status_string(8)
    assert rg.grpo_version() >= 100
    assert rg.grpo_kernel_launches() == 0 or rg.grpo_kernel_launches() > 0


def test_binding_refuses_to_run_without_the_library(tmp_path, monkeypatch):
    import rl_fine_tuning_gb300 as rg
    from rl_fine_tuning_gb300 import build
    monkeypatch.setattr(build, "LIB", str(tmp_path / "missing.so"))
    monkeypatch.setattr(rg, "_lib", None)
    with pytest.raises(ImportError):
        rg.load()
