"""Scalar CPU oracle of the W2A8 ternary matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may
import this package. The product (``ternary_weight_gb300``) never imports it, and it
imports nothing from the product: the only thing the two sides share is the seeded input
generator module ``ternary_weight_gb300.workloads``, which holds no arithmetic of the
method.

The arithmetic lives in ``bitnet_oracle.c`` (plain C11, one IEEE rounding per fp32 op);
this module only builds it with gcc and marshals numpy arrays through ctypes.

Sources are cited by page title and section in ``bitnet_oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "bitnet_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/liboracle.so`` (gcc, no fast-math, no FMA contraction)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "bitnet_oracle.h"))
    ):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    cmd = [
        "gcc", "-std=c11", "-O2", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math",
        "-frounding-math", "-Wall", "-Wextra", "-D_POSIX_C_SOURCE=200809L",
        _SRC, "-o", tmp, "-lm", "-lpthread",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_pack_i2s.argtypes = [P, P, I64, I64]
    lib.oracle_pack_i2s.restype = I64
    lib.oracle_unpack_i2s.argtypes = [P, P, I64, I64]
    lib.oracle_unpack_i2s.restype = ctypes.c_int
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    for name in ("oracle_quant_act_f32", "oracle_quant_act_bf16"):
        fn = getattr(lib, name)
        fn.argtypes = [P, I64, I64, P, P, P]
        fn.restype = ctypes.c_int
    lib.oracle_ternary_matmul.argtypes = [P, P, P, ctypes.c_float, P, P, I64, I64, I64, ctypes.c_int]
    lib.oracle_ternary_matmul.restype = ctypes.c_int
    lib.oracle_raw_code_dot.argtypes = [P, P, P, I64, I64, I64]
    lib.oracle_raw_code_dot.restype = ctypes.c_int
    for fn in (lib.oracle_quant_weight_f32, lib.oracle_quant_weight_bf16):
        fn.argtypes = [P, I64, I64, ctypes.c_int, P, P]
        fn.restype = ctypes.c_int
    lib.oracle_ffn_inner.argtypes = [P, P, P, ctypes.c_float, I64, I64, P]
    lib.oracle_ffn_inner.restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def pack_i2s(w: np.ndarray):
    """Ternary int8 ``w`` (N x K) -> (packed uint8 N x K/4, count of non-ternary entries)."""
    w = np.ascontiguousarray(w, dtype=np.int8)
    N, K = w.shape
    wp = np.empty((N, K // 4), dtype=np.uint8)
    bad = _load().oracle_pack_i2s(_ptr(w), _ptr(wp), N, K)
    if bad < 0:
        raise ValueError("oracle_pack_i2s: bad arguments (K must be a positive multiple of 128)")
    return wp, int(bad)


def unpack_i2s(wp: np.ndarray, K: int) -> np.ndarray:
    """Packed uint8 (N x K/4) -> int8 weights (N x K), each 2-bit code c read as c - 1."""
    wp = np.ascontiguousarray(wp, dtype=np.uint8)
    N = wp.shape[0]
    assert wp.shape[1] * 4 == K
    w = np.empty((N, K), dtype=np.int8)
    if _load().oracle_unpack_i2s(_ptr(wp), _ptr(w), N, K) != 0:
        raise ValueError("oracle_unpack_i2s: bad arguments")
    return w


def bf16_to_f32(bits: int) -> float:
    return float(_load().oracle_bf16_to_f32(int(bits)))


def quant_act(x: np.ndarray, dtype: str = "f32"):
    """Per-token absmax int8 quantisation of M x K rows.

    ``x`` is float32 for ``dtype='f32'`` or uint16 bf16 bit patterns for ``dtype='bf16'``.
    Returns (xq int8 M x K, s float32 M, rowsum int32 M).
    """
    lib = _load()
    if dtype == "f32":
        x = np.ascontiguousarray(x, dtype=np.float32)
        fn = lib.oracle_quant_act_f32
    elif dtype == "bf16":
        x = np.ascontiguousarray(x, dtype=np.uint16)
        fn = lib.oracle_quant_act_bf16
    else:
        raise ValueError(dtype)
    M, K = x.shape
    xq = np.empty((M, K), dtype=np.int8)
    s = np.empty(M, dtype=np.float32)
    rowsum = np.empty(M, dtype=np.int32)
    rc = fn(_ptr(x), M, K, _ptr(xq), _ptr(s), _ptr(rowsum))
    if rc != 0:
        raise RuntimeError("oracle quant_act failed: %d" % rc)
    return xq, s, rowsum


def ternary_matmul(xq: np.ndarray, s: np.ndarray, wp: np.ndarray, w_scale: float,
                   nthreads: int = 1):
    """The matmul by definition. Returns (out float32 M x N, acc int32 M x N)."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    s = np.ascontiguousarray(s, dtype=np.float32)
    wp = np.ascontiguousarray(wp, dtype=np.uint8)
    M, K = xq.shape
    N = wp.shape[0]
    assert wp.shape[1] * 4 == K and s.shape == (M,)
    out = np.empty((M, N), dtype=np.float32)
    acc = np.empty((M, N), dtype=np.int32)
    rc = _load().oracle_ternary_matmul(_ptr(xq), _ptr(s), _ptr(wp), ctypes.c_float(w_scale),
                                       _ptr(out), _ptr(acc), M, N, K, int(nthreads))
    if rc != 0:
        raise RuntimeError("oracle_ternary_matmul failed: %d" % rc)
    return out, acc


def raw_code_dot(xq: np.ndarray, wp: np.ndarray) -> np.ndarray:
    """The pages' raw code dot (codes 0/1/2 multiplied as stored). Returns int32 M x N."""
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    wp = np.ascontiguousarray(wp, dtype=np.uint8)
    M, K = xq.shape
    N = wp.shape[0]
    raw = np.empty((M, N), dtype=np.int32)
    if _load().oracle_raw_code_dot(_ptr(xq), _ptr(wp), _ptr(raw), M, N, K) != 0:
        raise RuntimeError("oracle_raw_code_dot failed")
    return raw


QUANT_WEIGHT_MODES = {"absmean": 0, "sign": 1}


def quant_weight(w: np.ndarray, dtype: str = "f32", mode: str = "absmean"):
    """Weight ternarisation of an N x K matrix (float32, or uint16 bf16 bit patterns).

    Returns (q int8 N x K in {-1, 0, +1}, scale float32): AbsMean (scale = max(mean|w|, 1e-5),
    q = clip(rne(w / scale), -1, 1)) or the sign rule (q = 0 where |w| < 1e-6, else sign(w);
    scale = max|w|).
    """
    lib = _load()
    if dtype == "f32":
        w = np.ascontiguousarray(w, dtype=np.float32)
        fn = lib.oracle_quant_weight_f32
    elif dtype == "bf16":
        w = np.ascontiguousarray(w, dtype=np.uint16)
        fn = lib.oracle_quant_weight_bf16
    else:
        raise ValueError(dtype)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.int8)
    scale = np.empty(1, dtype=np.float32)
    rc = fn(_ptr(w), N, K, QUANT_WEIGHT_MODES[mode], _ptr(q), _ptr(scale))
    if rc != 0:
        raise RuntimeError("oracle quant_weight failed: %d" % rc)
    return q, scale[0]


def ffn_inner(gate: np.ndarray, up: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """FFN inner activation of M x F fp32 gate and up rows: inner = RMSNorm(max(g, 0)^2 * u)
    with per-channel weight gamma (F fp32) and epsilon eps; the sum of squares is the plain
    ascending sum in double, rounded once to fp32. Returns M x F float32."""
    lib = _load()
    gate = np.ascontiguousarray(gate, dtype=np.float32)
    up = np.ascontiguousarray(up, dtype=np.float32)
    gamma = np.ascontiguousarray(gamma, dtype=np.float32)
    if gate.ndim == 1:
        gate, up = gate[None, :], up[None, :]
    M, F = gate.shape
    if up.shape != (M, F) or gamma.shape != (F,):
        raise ValueError("shape mismatch")
    inner = np.empty((M, F), dtype=np.float32)
    rc = lib.oracle_ffn_inner(_ptr(gate), _ptr(up), _ptr(gamma), float(eps), M, F, _ptr(inner))
    if rc != 0:
        raise RuntimeError("oracle ffn_inner failed: %d" % rc)
    return inner


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count() or 1)
