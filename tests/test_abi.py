"""The C ABI without a GPU: the library builds and loads, exports every entry point that
include/bitnet.h declares, and rejects bad arguments on the host before any CUDA call.
No kernel is launched here."""
import ctypes
import os
import re
import subprocess

import pytest

from ternary_weight_gb300 import _build, binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return binding.lib()


def declared_entry_points():
    names = []
    for fn in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if fn.endswith(".h"):
            src = open(os.path.join(ROOT, "include", fn)).read()
            names += re.findall(r"BITNET_API\s+[\w\s\*]+?\b(bitnet_\w+)\s*\(", src)
    return names


def test_header_declares_the_boundary():
    names = declared_entry_points()
    for required in ("bitnet_pack_i2s", "bitnet_quant_act", "bitnet_i2s_matmul"):
        assert required in names
    assert set(names) == set(binding.SIGNATURES), "binding and header disagree"


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", _build.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    for name in declared_entry_points():
        assert name in exported, name
        assert getattr(lib, name) is not None
    # nothing but the C ABI is exported
    assert {e for e in exported if e.startswith("bitnet")} == set(declared_entry_points())


def test_version_and_strerror(lib):
    assert lib.bitnet_version() >= 100
    for st in (0, -1, -2, -3, -4, -5, -99):
        assert isinstance(lib.bitnet_strerror(st), bytes) and lib.bitnet_strerror(st)


FAKE = 1 << 20  # a 16-byte aligned non-null pointer value; never dereferenced: validation fails first


def _mm(lib, xq=FAKE, s=FAKE, rs=FAKE, wp=FAKE, out=FAKE, acc=None, M=1, N=1, K=128, algo=0):
    return lib.bitnet_i2s_matmul_algo(xq, s, rs, wp, 1.0, out, acc, M, N, K, algo, None)


@pytest.mark.parametrize("kw,status", [
    (dict(xq=None), -1), (dict(s=None), -1), (dict(rs=None), -1), (dict(wp=None), -1), (dict(out=None), -1),
    (dict(K=100), -1), (dict(K=0), -1), (dict(K=-128), -1), (dict(K=128 * 513 * 2), -1),
    (dict(M=0), -1), (dict(N=0), -1), (dict(M=-5), -1), (dict(N=1 << 31), -1),
    (dict(algo=6), -1), (dict(algo=-1), -1), (dict(algo=2, K=65536), -1), (dict(algo=4, K=32768 + 128), -1),
    (dict(algo=5, K=32768 + 128), -1),
    (dict(algo=3, M=64 * 65535 + 1), -1), (dict(algo=3, K=32768 + 128), -1),
    (dict(xq=FAKE + 8), -2), (dict(wp=FAKE + 4), -2), (dict(out=FAKE + 2), -2), (dict(acc=FAKE + 1), -2),
    (dict(s=FAKE + 1), -2), (dict(rs=FAKE + 2), -2),
])
def test_matmul_rejects_bad_arguments_on_host(lib, kw, status):
    assert _mm(lib, **kw) == status


@pytest.mark.parametrize("args,status", [
    ((None, 0, 1, 128, FAKE, FAKE, FAKE), -1),
    ((FAKE, 2, 1, 128, FAKE, FAKE, FAKE), -1),
    ((FAKE, 0, 0, 128, FAKE, FAKE, FAKE), -1),
    ((FAKE, 0, 1, 130, FAKE, FAKE, FAKE), -1),
    ((FAKE + 4, 0, 1, 128, FAKE, FAKE, FAKE), -2),
    ((FAKE, 1, 1, 128, FAKE + 8, FAKE, FAKE), -2),
])
def test_quant_act_rejects_bad_arguments_on_host(lib, args, status):
    assert lib.bitnet_quant_act(*args, None) == status


@pytest.mark.parametrize("args,status", [
    ((None, FAKE, 1, 128, None), -1),
    ((FAKE, None, 1, 128, None), -1),
    ((FAKE, FAKE, 0, 128, None), -1),
    ((FAKE, FAKE, 1, 64, None), -1),
    ((FAKE + 1, FAKE, 1, 128, None), -2),
    ((FAKE, FAKE + 8, 1, 128, None), -2),
    ((FAKE, FAKE, 1, 128, FAKE + 2), -2),
])
def test_pack_rejects_bad_arguments_on_host(lib, args, status):
    assert lib.bitnet_pack_i2s(*args, None) == status


@pytest.mark.parametrize("args,status", [
    # (w, dtype, mode, N, K, wp, w_scale)
    ((None, 0, 0, 1, 128, FAKE, FAKE), -1),
    ((FAKE, 0, 0, 1, 128, None, FAKE), -1),
    ((FAKE, 0, 0, 1, 128, FAKE, None), -1),
    ((FAKE, 2, 0, 1, 128, FAKE, FAKE), -1),
    ((FAKE, 0, 2, 1, 128, FAKE, FAKE), -1),
    ((FAKE, 0, -1, 1, 128, FAKE, FAKE), -1),
    ((FAKE, 0, 0, 0, 128, FAKE, FAKE), -1),
    ((FAKE, 0, 0, 1, 192, FAKE, FAKE), -1),
    ((FAKE, 0, 0, 1, 65536 + 128, FAKE, FAKE), -1),
    ((FAKE, 0, 0, 1 << 30, 65536, FAKE, FAKE), -1),
    ((FAKE + 8, 0, 0, 1, 128, FAKE, FAKE), -2),
    ((FAKE, 1, 1, 1, 128, FAKE + 4, FAKE), -2),
    ((FAKE, 0, 0, 1, 128, FAKE, FAKE + 2), -2),
])
def test_quant_weight_rejects_bad_arguments_on_host(lib, args, status):
    assert lib.bitnet_quant_weight(*args, None) == status


@pytest.mark.parametrize("args,status", [
    # (gate, up, gamma, eps, M, F, xq, s, rowsum, inner_out)
    ((None, FAKE, FAKE, 1e-5, 1, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, None, 1e-5, 1, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, 1e-5, 1, 128, FAKE, None, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, 0.0, 1, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, -1e-5, 1, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, float("inf"), 1, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, float("nan"), 1, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, 1e-5, 0, 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, 1e-5, 1, 192, FAKE, FAKE, FAKE, None), -1),
    ((FAKE, FAKE, FAKE, 1e-5, 1, 32768 + 128, FAKE, FAKE, FAKE, None), -1),
    ((FAKE + 4, FAKE, FAKE, 1e-5, 1, 128, FAKE, FAKE, FAKE, None), -2),
    ((FAKE, FAKE, FAKE + 8, 1e-5, 1, 128, FAKE, FAKE, FAKE, None), -2),
    ((FAKE, FAKE, FAKE, 1e-5, 1, 128, FAKE + 4, FAKE, FAKE, None), -2),
    ((FAKE, FAKE, FAKE, 1e-5, 1, 128, FAKE, FAKE, FAKE, FAKE + 4), -2),
])
def test_ffn_act_quant_rejects_bad_arguments_on_host(lib, args, status):
    assert lib.bitnet_ffn_act_quant(*args, None) == status


def _ffn(lib, x=FAKE, dtype=0, M=1, K=128, F=128, wg=FAKE, wu=FAKE, wd=FAKE, gamma=FAKE, eps=1e-5, go=FAKE,
         uo=FAKE, out=FAKE, xq=None, s=None, rs=None, ws=None, ws_bytes=0):
    return lib.bitnet_w2a8_ffn(x, dtype, M, K, F, wg, 1.0, wu, 1.0, wd, 1.0, gamma, eps, go, uo, out, xq, s, rs, ws,
                               ws_bytes, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), -1), (dict(wd=None), -1), (dict(gamma=None), -1), (dict(uo=None), -1),
    (dict(dtype=2), -1), (dict(M=0), -1), (dict(K=192), -1), (dict(F=64), -1), (dict(F=32768 + 128), -1),
    (dict(eps=0.0), -1), (dict(eps=float("nan")), -1),
    (dict(M=2), -1),                                   # several rows need the quantisation workspace
    (dict(M=1, K=10240 + 128), -1),                    # beyond the two-launch path: workspace again
    (dict(M=2048, K=256, F=256, xq=FAKE, s=FAKE, rs=FAKE, ws=FAKE + 16, ws_bytes=16), -2),  # (unused) workspace misaligned
    (dict(x=FAKE + 8), -2), (dict(wu=FAKE + 4), -2), (dict(go=FAKE + 4), -2), (dict(gamma=FAKE + 4), -2),
    (dict(M=2, xq=FAKE + 4, s=FAKE, rs=FAKE), -2),
])
def test_w2a8_ffn_rejects_bad_arguments_on_host(lib, kw, status):
    assert _ffn(lib, **kw) == status


def test_ffn_workspace_size(lib):
    # the projections take the workspace-free kernels at every size: no workspace is needed
    for M in (1, 64, 2047, 2048, 4096, 1 << 20):
        assert lib.bitnet_w2a8_ffn_workspace_size(M, 2560, 6912) == 0
    assert lib.bitnet_w2a8_ffn_workspace_size(0, 2560, 6912) == -1
    assert lib.bitnet_w2a8_ffn_workspace_size(4096, 2560, 32768 + 128) == -1


def _sweep_desc(**kw):
    d = binding.LinearGroupDesc()
    d.x, d.K, d.count = kw.get("x", FAKE), kw.get("K", 256), kw.get("count", 1)
    d.wp[0], d.w_scale[0], d.N[0], d.out[0] = kw.get("wp", FAKE), 1.0, kw.get("N", 4), kw.get("out", FAKE)
    return d


@pytest.mark.parametrize("kw,dtype,status", [
    (dict(x=None), 0, -1), (dict(count=0), 0, -1), (dict(count=9), 0, -1), (dict(K=192), 0, -1),
    (dict(K=10240 + 128), 0, -1), (dict(N=0), 0, -1), (dict(wp=None), 0, -1), (dict(out=None), 0, -1),
    (dict(), 2, -1),
    (dict(x=FAKE + 8), 0, -2), (dict(wp=FAKE + 4), 0, -2), (dict(out=FAKE + 2), 0, -2),
])
def test_sweep_plan_rejects_bad_tables_on_host(lib, kw, dtype, status):
    descs = (binding.LinearGroupDesc * 2)(_sweep_desc(), _sweep_desc(**kw))
    handle = ctypes.c_void_p(123)
    assert lib.bitnet_sweep_plan_create(ctypes.cast(descs, ctypes.c_void_p), 2, dtype, ctypes.byref(handle)) == status
    assert handle.value is None  # no plan on failure


def test_sweep_plan_null_arguments(lib):
    handle = ctypes.c_void_p()
    descs = (binding.LinearGroupDesc * 1)(_sweep_desc())
    assert lib.bitnet_sweep_plan_create(None, 1, 0, ctypes.byref(handle)) == -1
    assert lib.bitnet_sweep_plan_create(ctypes.cast(descs, ctypes.c_void_p), 0, 0, ctypes.byref(handle)) == -1
    assert lib.bitnet_sweep_plan_create(ctypes.cast(descs, ctypes.c_void_p), 1, 0, None) == -1
    assert lib.bitnet_sweep_plan_run(None, None) == -1
    assert lib.bitnet_sweep_plan_destroy(None) == 0


def test_sweep_plan_struct_layout_matches_header():
    """The ctypes mirror has the C layout: 8-byte x, K, a 4-byte count padded to 8, then the arrays."""
    D = binding.LinearGroupDesc
    assert D.x.offset == 0 and D.K.offset == 8 and D.count.offset == 16 and D.wp.offset == 24
    assert D.w_scale.offset == 24 + 64 and D.N.offset == 24 + 64 + 32 and D.out.offset == 24 + 64 + 32 + 64
    assert ctypes.sizeof(D) == 24 + 64 + 32 + 64 + 64


def test_valid_call_without_gpu_is_unsupported(lib):
    import torch

    if torch.cuda.is_available():
        pytest.skip("a GPU is present; covered by the gpu tests")
    assert _mm(lib) == -4
    assert lib.bitnet_last_device_error() == -4


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(binding, "_lib", None)
    monkeypatch.setattr(binding, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        binding.lib()


def _group(lib, x=FAKE, dtype=0, M=1, K=128, count=1, wp=(FAKE,), ws=(1.0,), N=(1,), out=(FAKE,), acc=None,
           xq=None, s=None, rs=None):
    wp_a = (ctypes.c_void_p * len(wp))(*wp) if wp is not None else None
    out_a = (ctypes.c_void_p * len(out))(*out) if out is not None else None
    acc_a = (ctypes.c_void_p * len(acc))(*acc) if acc is not None else None
    ws_a = (ctypes.c_float * len(ws))(*ws)
    n_a = (ctypes.c_int64 * len(N))(*N)
    return lib.bitnet_w2a8_linear_group(x, dtype, M, K, count, wp_a, ws_a, n_a, out_a, acc_a, xq, s, rs, None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), -1), (dict(dtype=5), -1), (dict(count=0), -1), (dict(count=9), -1), (dict(M=0), -1),
    (dict(K=200), -1), (dict(wp=None), -1), (dict(out=None), -1), (dict(wp=(0,)), -1), (dict(N=(0,)), -1),
    (dict(M=2), -1),                                            # workspace required beyond one launch
    (dict(x=FAKE + 4), -2), (dict(wp=(FAKE + 8,)), -2), (dict(out=(FAKE + 2,)), -2),
    (dict(acc=(FAKE + 1,)), -2), (dict(xq=FAKE + 8), -2),
])
def test_linear_group_rejects_bad_arguments_on_host(lib, kw, status):
    assert _group(lib, **kw) == status


def test_linear_group_ex_rejects_bad_prefetch(lib):
    wp = (ctypes.c_void_p * 1)(FAKE)
    out = (ctypes.c_void_p * 1)(FAKE)
    ws = (ctypes.c_float * 1)(1.0)
    n = (ctypes.c_int64 * 1)(1)
    call = lambda cnt, ptrs, sizes: lib.bitnet_w2a8_linear_group_ex(FAKE, 0, 1, 128, 1, wp, ws, n, out, None, None,
                                                                    None, None, cnt, ptrs, sizes, None)
    P = ctypes.c_void_p * 2
    B = ctypes.c_int64 * 2
    assert call(9, P(FAKE, FAKE), B(16, 16)) == -1
    assert call(-1, P(FAKE, FAKE), B(16, 16)) == -1
    assert call(1, None, B(16, 16)) == -1
    assert call(1, P(0, 0), B(16, 16)) == -1
    assert call(1, P(FAKE, 0), B(-16, 16)) == -1
    assert call(1, P(FAKE + 4, 0), B(16, 16)) == -2


def test_workspace_size_and_ws_validation(lib):
    up = lambda v: (v + 255) // 256 * 256
    for M, N, K in ((2, 3, 128), (4096, 2560, 6912), (1, 1, 32768)):
        assert lib.bitnet_i2s_matmul_workspace_size(M, N, K) == up(M * K * 2) + up(N * K * 2)
    assert lib.bitnet_i2s_matmul_workspace_size(1, 1, 65536) == -1  # beyond the exact-accumulation K
    assert lib.bitnet_i2s_matmul_workspace_size(0, 1, 128) == -1
    need = lib.bitnet_i2s_matmul_workspace_size(1, 1, 128)
    ws = lambda **kw: lib.bitnet_i2s_matmul_ws(kw.get("xq", FAKE), FAKE, FAKE, FAKE, 1.0, FAKE, None, 1, 1, 128,
                                               kw.get("w", FAKE), kw.get("n", need), None)
    assert ws(w=None) == -1
    assert ws(n=need - 1) == -1
    assert ws(w=FAKE + 16) == -2   # the workspace must be 256-byte aligned
    assert ws(xq=FAKE + 8) == -2


@pytest.mark.parametrize("args,status", [
    ((None, 64, 8, FAKE), -1), ((FAKE, 64, 8, None), -1), ((FAKE, 0, 8, FAKE), -1), ((FAKE, 24, 8, FAKE), -1),
    ((FAKE, 16384 + 16, 8, FAKE), -1), ((FAKE, 64, 0, FAKE), -1), ((FAKE, 64, (1 << 20) + 1, FAKE), -1),
    ((FAKE + 8, 64, 8, FAKE), -2), ((FAKE, 64, 8, FAKE + 2), -2),
])
def test_selftest_rejects_bad_arguments_on_host(lib, args, status):
    assert lib.bitnet_selftest_wait_timeout(*args, None) == status
