"""The C ABI without a GPU: the library loads, exports every function the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import importlib.util
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "awq.h")
LIB = os.path.join(ROOT, "post_weight_quantization_32_b300", "libawq.so")


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(awq_\w+)\s*\(", src)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(LIB):
        path = os.path.join(ROOT, "post_weight_quantization_32_b300", "build.py")
        spec = importlib.util.spec_from_file_location("awq_build", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)
        mod.build()
    return ctypes.CDLL(LIB)


def test_header_declares_the_entry_points():
    names = _declared()
    for n in ("awq_channel_stats", "awq_search", "awq_search_ex", "awq_search_workspace_bytes",
              "awq_quantize_pack", "awq_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in _declared():
        assert hasattr(lib, n), n


def test_binding_names_match_abi(lib):
    import post_weight_quantization_32_b300 as pkg
    for n in ("awq_channel_stats", "awq_search", "awq_quantize_pack", "awq_search_workspace_bytes"):
        assert callable(getattr(pkg, n))
    for n in pkg.EXPORTS:
        assert n in _declared()


def test_status_strings(lib):
    lib.awq_status_string.restype = ctypes.c_char_p
    for code in range(6):
        assert lib.awq_status_string(code)
    assert b"unknown" in lib.awq_status_string(99)


def _ws(lib, *a, fn="awq_search_workspace_min_bytes"):
    f = getattr(lib, fn)
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                  ctypes.c_int]
    return f(*a)


def test_workspace_query(lib):
    # fp16 notebook-shaped layer: X is read in place; s and 1/s tables for 21 alphas
    n = _ws(lib, 1, 4096, 4096, 256, 128, 20)
    assert n >= 21 * 4096 * (4 + 4) and n % 256 == 0
    # bf16 and fp32 add the fp16 copy of X the tensor cores read
    assert _ws(lib, 2, 4096, 4096, 256, 128, 20) >= n + 256 * 4096 * 2
    assert _ws(lib, 0, 4096, 4096, 256, 128, 20) >= n + 256 * 4096 * 2
    # groups wider than a producer job add their precomputed ranges (two floats
    # per alpha, row and group)
    assert _ws(lib, 1, 4096, 4096, 256, 256, 20) >= n + 21 * 4096 * 16 * 8
    assert _ws(lib, 1, 4096, 4096, 256, 4096, 20) >= n + 21 * 4096 * 8
    for fn in ("awq_search_workspace_min_bytes", "awq_search_workspace_bytes"):
        assert _ws(lib, 2, 4096, 4096, 256, 100, 20, fn=fn) == 0      # group does not divide in
        assert _ws(lib, 2, 0, 4096, 256, 128, 20, fn=fn) == 0
        assert _ws(lib, 7, 16, 16, 16, 16, 20, fn=fn) == 0
        assert _ws(lib, 2, 16, 16, 16, 16, 5000, fn=fn) == 0


def test_workspace_of_the_pre_divided_path(lib):
    full = lambda *a: _ws(lib, *a, fn="awq_search_workspace_bytes")  # noqa: E731
    # 16-bit, more than 128 tokens, group 128 (or a group read from its
    # precomputed ranges), 21 copies of X / s within 64 MiB: the full
    # workspace adds the copies (fp16, N x in each) and the scaled s table
    for dt in (1, 2):
        for n_in, g in ((4096, 128), (4096, 256), (4096, 4096), (3072, 96)):
            assert full(dt, 4096, n_in, 256, g, 20) >= (
                _ws(lib, 1, 4096, n_in, 256, g, 20) + 21 * 256 * n_in * 2 + 21 * n_in * 4)
    # not eligible: fp32, 128 tokens or fewer, or copies beyond 64 MiB
    for args in ((0, 4096, 4096, 256, 128, 20), (1, 4096, 4096, 128, 128, 20),
                 (1, 4096, 3072, 128, 96, 20), (2, 8192, 28672, 1024, 128, 40)):
        assert full(*args) == _ws(lib, *args)


def test_search_rejects_bad_arguments_on_host(lib):
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.awq_search.restype = i32
    lib.awq_search.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, i32, vp, sz, vp, vp,
                               vp, vp, vp]
    fake = 1 << 20  # never dereferenced: the checks return before any launch
    ok = dict(W=fake, X=fake, dt=2, out=256, n_in=512, N=64, sx=None, bits=4, group=128, sym=1,
              grid=20, ws=fake, wsb=1 << 30, err=fake, best=fake, s_best=fake, st=fake, stream=None)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.awq_search(a["W"], a["X"], a["dt"], a["out"], a["n_in"], a["N"], a["sx"],
                              a["bits"], a["group"], a["sym"], a["grid"], a["ws"], a["wsb"],
                              a["err"], a["best"], a["s_best"], a["st"], a["stream"])

    assert call(W=None) == 1
    assert call(N=0) == 1
    assert call(bits=1) == 1 and call(bits=9) == 1
    assert call(grid=0) == 1
    assert call(group=100) == 1          # does not divide in
    assert call(wsb=16) == 1             # workspace too small
    assert call(ws=fake + 8) == 1        # workspace not 256-byte aligned
    # valid for the method, not handled by the search kernels: a group that is
    # not a multiple of 8 columns, or range-pass groups with in % 8 != 0
    assert call(group=12, n_in=768) == 2
    assert call(group=12, n_in=516) == 2
    assert call(group=516, n_in=516) == 2
    assert call(W=fake + 4) == 2         # TMA needs 16-byte aligned rows


def test_pack_rejects_bad_arguments_on_host(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.awq_quantize_pack.restype = i32
    lib.awq_quantize_pack.argtypes = [vp, i32, i64, i64, vp, i32, i32, i32, vp, vp, vp, vp, vp]
    f = 1 << 20
    assert lib.awq_quantize_pack(None, 2, 4, 8, f, 4, 8, 1, f, f, f, f, None) == 1
    assert lib.awq_quantize_pack(f, 2, 4, 8, f, 4, 3, 1, f, f, f, f, None) == 1
    assert lib.awq_quantize_pack(f, 2, 4, 8, f, 1, 8, 1, f, f, f, f, None) == 1
    assert lib.awq_quantize_pack(f, 5, 4, 8, f, 4, 8, 1, f, f, f, f, None) == 1


def test_stats_rejects_bad_arguments_on_host(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.awq_channel_stats.restype = i32
    lib.awq_channel_stats.argtypes = [vp, i32, i64, i64, vp, vp, vp]
    f = 1 << 20
    assert lib.awq_channel_stats(None, 2, 4, 8, f, None, None) == 1
    assert lib.awq_channel_stats(f, 2, 0, 8, f, None, None) == 1
    assert lib.awq_channel_stats(f, 9, 4, 8, f, None, None) == 1


def test_output_power_rejects_bad_arguments_on_host(lib):
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.awq_output_power.restype = i32
    lib.awq_output_power.argtypes = [vp, vp, i32, i64, i64, i64, vp, sz, vp, vp, vp]
    f = 1 << 20   # never dereferenced
    lib.awq_output_power_workspace_bytes.restype = sz
    lib.awq_output_power_workspace_bytes.argtypes = [i32, i64, i64, i64]
    need = lib.awq_output_power_workspace_bytes(2, 64, 256, 16)
    assert need >= 16 * 64 * 4 and need % 256 == 0   # the float32 product X W^T and a scratch
    assert lib.awq_output_power_workspace_bytes(7, 64, 256, 16) == 0
    ok = dict(W=f, X=f, dt=2, out=64, n_in=256, N=16, ws=f, wsb=need, p=f)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.awq_output_power(a["W"], a["X"], a["dt"], a["out"], a["n_in"], a["N"], a["ws"],
                                    a["wsb"], a["p"], None, None)

    assert call(W=None) == 1 and call(p=None) == 1
    assert call(N=0) == 1 and call(out=0) == 1 and call(dt=7) == 1
    assert call(wsb=need - 1) == 1 and call(ws=f + 16) == 1


def test_clip_search_rejects_bad_arguments_on_host(lib):
    vp, i64, i32, sz = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
    lib.awq_clip_search_workspace_bytes.restype = sz
    lib.awq_clip_search_workspace_bytes.argtypes = [i64, i64, i32]
    lib.awq_clip_search.restype = i32
    lib.awq_clip_search.argtypes = [vp, vp, i32, i64, i64, i64, vp, i32, i32, i32, i32, i32, vp, sz,
                                    vp, vp, vp, vp]
    # Gram matrices (one g x g float block per group and token split of 256),
    # or, for group 128 and at most 256 tokens, the tensor-core path's s * 2^e
    # and 2^m / s rows, control words and fp16 copy of X / s if larger
    assert lib.awq_clip_search_workspace_bytes(4096, 256, 128) == 2 * 4096 * 4 + 256 + 256 * 4096 * 2
    assert lib.awq_clip_search_workspace_bytes(4096, 64, 128) == 4096 * 128 * 4
    assert lib.awq_clip_search_workspace_bytes(4096, 2048, 128) == 8 * 4096 * 128 * 4
    assert lib.awq_clip_search_workspace_bytes(4096, 256, 64) == 4096 * 64 * 4
    assert lib.awq_clip_search_workspace_bytes(4096, 256, 256) == 0     # group not handled
    assert lib.awq_clip_search_workspace_bytes(100, 256, 32) == 0       # group does not divide in
    f = 1 << 20
    ok = dict(W=f, X=f, dt=1, out=8, n_in=256, N=4, s=f, bits=4, group=128, sym=1, n_grid=20,
              steps=10, ws=f, wsb=1 << 30, clip=f)

    def call(**kw):
        a = dict(ok)
        a.update(kw)
        return lib.awq_clip_search(a["W"], a["X"], a["dt"], a["out"], a["n_in"], a["N"], a["s"],
                                   a["bits"], a["group"], a["sym"], a["n_grid"], a["steps"],
                                   a["ws"], a["wsb"], a["clip"], None, None, None)

    assert call(clip=None) == 1 and call(s=None) == 1 and call(bits=9) == 1
    assert call(n_grid=0) == 1 and call(steps=-1) == 1 and call(steps=20) == 1
    assert call(wsb=16) == 1 and call(ws=f + 64) == 1
    assert call(group=64, n_in=256, steps=12) == 2     # more than twelve factors
    assert call(group=256, n_in=512) == 2              # groups wider than 128 columns


def test_export_and_clipped_pack_reject_bad_arguments_on_host(lib):
    vp, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.awq_export_checkpoint.restype = i32
    lib.awq_export_checkpoint.argtypes = [vp, vp, vp, i64, i64, i32, i32, vp, vp, vp, vp, vp]
    f = 1 << 20
    assert lib.awq_export_checkpoint(None, f, f, 4, 64, 4, 32, f, f, f, None, None) == 1
    assert lib.awq_export_checkpoint(f, f, f, 4, 64, 3, 32, f, f, f, None, None) == 1  # 3 bits
    assert lib.awq_export_checkpoint(f, f, f, 4, 60, 4, 30, f, f, f, None, None) == 1  # in % 8
    assert lib.awq_export_checkpoint(f, f, f, 4, 64, 4, 48, f, f, f, None, None) == 1  # group
    lib.awq_quantize_pack_clipped.restype = i32
    lib.awq_quantize_pack_clipped.argtypes = [vp, i32, i64, i64, vp, i32, i32, i32, vp, vp, vp, vp,
                                              vp, vp]
    assert lib.awq_quantize_pack_clipped(f, 2, 4, 8, f, 4, 8, 1, None, f, f, f, None, None) == 1
    assert lib.awq_quantize_pack_clipped(f, 2, 4, 8, f, 4, 3, 1, f, f, f, f, None, None) == 1


def test_binding_wrappers_pass_one_label_to_the_status_check():
    # every wrapper reports a failing C call under its own name
    import ast
    src = open(os.path.join(ROOT, "post_weight_quantization_32_b300", "__init__.py")).read()
    calls = [n for n in ast.walk(ast.parse(src))
             if isinstance(n, ast.Call) and getattr(n.func, "id", "") == "_check"]
    assert calls and all(len(c.args) == 2 and isinstance(c.args[1], ast.Constant) for c in calls)


def test_wait_limit_from_the_environment(monkeypatch):
    import post_weight_quantization_32_b300 as awq
    monkeypatch.delenv("AWQ_WAIT_LIMIT_MS", raising=False)
    assert awq._env_opts() is None
    monkeypatch.setenv("AWQ_WAIT_LIMIT_MS", "250")
    o = awq._env_opts()
    assert o.wait_limit_ns == 250_000_000 and o.test_timeout == 0 and not o.diag


def test_sweep_summary_rejects_bad_arguments_on_host(lib):
    vp, i32 = ctypes.c_void_p, ctypes.c_int
    lib.awq_sweep_summary.restype = i32
    lib.awq_sweep_summary.argtypes = [vp, vp, vp, i32, vp, vp]
    fake = 1 << 20  # never dereferenced
    assert lib.awq_sweep_summary(None, fake, fake, 20, fake, None) == 1
    assert lib.awq_sweep_summary(fake, fake, fake, 0, fake, None) == 1
    assert lib.awq_sweep_summary(fake, fake, fake, 5000, fake, None) == 1
    assert lib.awq_sweep_summary(fake, fake, None, 20, fake, None) == 1
