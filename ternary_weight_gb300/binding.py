"""ctypes binding of libbitnet_gb300 (the C ABI in include/bitnet.h).

Argument marshalling only: every step of the computation runs in the library's CUDA
kernels. Tensors are torch CUDA tensors (torch supplies device memory and streams); the
functions pass their data pointers and the current stream to the C entry points and raise
``BitnetError`` on a negative status. There is no CPU fallback: if the shared library is
missing or fails to load, ``lib()`` raises.
"""
from __future__ import annotations

import ctypes
import os

from . import _build

BITNET_OK = 0
BITNET_EINVAL = -1
BITNET_EALIGN = -2
BITNET_ECUDA = -3
BITNET_EUNSUPPORTED = -4
BITNET_ETIMEOUT = -5
BITNET_ERANGE = -6

BITNET_F32 = 0
BITNET_BF16 = 1

ALGO = {"auto": 0, "gemv": 1, "gemm": 2, "smallm": 3, "prefill": 4, "pair": 5}

# every entry point of include/bitnet.h with its ctypes signature
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
SIGNATURES = {
    "bitnet_version": ([], ctypes.c_int),
    "bitnet_strerror": ([ctypes.c_int], ctypes.c_char_p),
    "bitnet_pack_i2s": ([_P, _P, _I64, _I64, _P, _P], ctypes.c_int),
    "bitnet_quant_act": ([_P, ctypes.c_int, _I64, _I64, _P, _P, _P, _P], ctypes.c_int),
    "bitnet_i2s_matmul": ([_P, _P, _P, _P, ctypes.c_float, _P, _P, _I64, _I64, _I64, _P], ctypes.c_int),
    "bitnet_i2s_matmul_algo": (
        [_P, _P, _P, _P, ctypes.c_float, _P, _P, _I64, _I64, _I64, ctypes.c_int, _P], ctypes.c_int),
    "bitnet_w2a8_linear_group": (
        [_P, ctypes.c_int, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "bitnet_w2a8_linear_group_ex": (
        [_P, ctypes.c_int, _I64, _I64, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P, _P, ctypes.c_int, _P, _P, _P],
        ctypes.c_int),
    "bitnet_w2a8_linear": (
        [_P, ctypes.c_int, _I64, _I64, _P, ctypes.c_float, _I64, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "bitnet_i2s_matmul_workspace_size": ([_I64, _I64, _I64], _I64),
    "bitnet_i2s_matmul_ws": (
        [_P, _P, _P, _P, ctypes.c_float, _P, _P, _I64, _I64, _I64, _P, _I64, _P], ctypes.c_int),
    "bitnet_i2s_matmul_noalloc": ([_P, _P, _P, _P, ctypes.c_float, _P, _P, _I64, _I64, _I64, _P], ctypes.c_int),
    "bitnet_last_device_error": ([], ctypes.c_int),
    "bitnet_selftest_wait_timeout": ([_P, _I64, ctypes.c_int32, _P, _P], ctypes.c_int),
    "bitnet_quant_weight": ([_P, ctypes.c_int, ctypes.c_int, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "bitnet_ffn_act_quant": ([_P, _P, _P, ctypes.c_float, _I64, _I64, _P, _P, _P, _P, _P], ctypes.c_int),
    "bitnet_w2a8_ffn_workspace_size": ([_I64, _I64, _I64], _I64),
    "bitnet_sweep_plan_create": ([_P, ctypes.c_int, ctypes.c_int, _P], ctypes.c_int),
    "bitnet_sweep_plan_run": ([_P, _P], ctypes.c_int),
    "bitnet_sweep_plan_destroy": ([_P], ctypes.c_int),
    "bitnet_w2a8_ffn": (
        [_P, ctypes.c_int, _I64, _I64, _I64, _P, ctypes.c_float, _P, ctypes.c_float, _P, ctypes.c_float, _P,
         ctypes.c_float, _P, _P, _P, _P, _P, _P, _P, _I64, _P], ctypes.c_int),
}

_lib = None


class BitnetError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = lib().bitnet_strerror(status).decode() if _lib is not None else str(status)
        super().__init__("%s failed with status %d: %s" % (where, status, msg))
        self.status = status


def lib_path() -> str:
    return _build.LIB_PATH


def lib():
    """Load the CUDA library (built in-tree by ``_build.build()``); raise if it is absent."""
    global _lib
    if _lib is not None:
        return _lib
    path = lib_path()
    if not os.path.exists(path):
        raise RuntimeError(
            "libbitnet_gb300.so is not built (%s); run ternary_weight_gb300._build.build() "
            "or __graft_entry__.build() first -- there is no CPU fallback" % path)
    l = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(l, name)
        fn.argtypes = args
        fn.restype = res
    _lib = l
    return l


def _check(status: int, where: str):
    if status != BITNET_OK:
        raise BitnetError(status, where)


def _stream(stream=None):
    import torch

    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("tensors must be contiguous CUDA tensors")


def pack_i2s(w, out=None, invalid_count=None, stream=None):
    """Ternary int8 weights (N x K, CUDA) -> i2_s packed uint8 (N x K/4)."""
    import torch

    N, K = w.shape
    if out is None:
        out = torch.empty((N, K // 4), dtype=torch.uint8, device=w.device)
    _require_cuda(w, out, invalid_count)
    _check(lib().bitnet_pack_i2s(_ptr(w), _ptr(out), N, K, _ptr(invalid_count), _stream(stream)),
           "bitnet_pack_i2s")
    return out


QUANT_WEIGHT_MODES = {"absmean": 0, "sign": 1}


def quant_weight(w, mode="absmean", out=None, scale=None, stream=None):
    """fp32 or bf16 weights (N x K, CUDA) -> (i2_s packed uint8 N x K/4, fp32 scale tensor of 1)."""
    import torch

    if w.dtype == torch.float32:
        dt = BITNET_F32
    elif w.dtype == torch.bfloat16:
        dt = BITNET_BF16
    else:
        raise ValueError("w must be float32 or bfloat16")
    N, K = w.shape
    out = torch.empty((N, K // 4), dtype=torch.uint8, device=w.device) if out is None else out
    scale = torch.empty(1, dtype=torch.float32, device=w.device) if scale is None else scale
    _require_cuda(w, out, scale)
    _check(lib().bitnet_quant_weight(_ptr(w), dt, QUANT_WEIGHT_MODES[mode], N, K, _ptr(out), _ptr(scale),
                                     _stream(stream)), "bitnet_quant_weight")
    return out, scale


def quant_act(x, xq=None, scale=None, rowsum=None, stream=None):
    """fp32 or bf16 rows (M x K, CUDA) -> (xq int8 M x K, s fp32 M, rowsum int32 M)."""
    import torch

    if x.dtype == torch.float32:
        dt = BITNET_F32
    elif x.dtype == torch.bfloat16:
        dt = BITNET_BF16
    else:
        raise ValueError("x must be float32 or bfloat16")
    M, K = x.shape
    dev = x.device
    xq = torch.empty((M, K), dtype=torch.int8, device=dev) if xq is None else xq
    scale = torch.empty(M, dtype=torch.float32, device=dev) if scale is None else scale
    rowsum = torch.empty(M, dtype=torch.int32, device=dev) if rowsum is None else rowsum
    _require_cuda(x, xq, scale, rowsum)
    _check(lib().bitnet_quant_act(_ptr(x), dt, M, K, _ptr(xq), _ptr(scale), _ptr(rowsum), _stream(stream)),
           "bitnet_quant_act")
    return xq, scale, rowsum


def i2s_matmul(xq, scale, rowsum, wp, w_scale, out=None, acc_out=None, algo="auto", stream=None):
    """W2A8 ternary matmul: returns out (M x N fp32); fills acc_out (M x N int32) if given."""
    import torch

    M, K = xq.shape
    N = wp.shape[0]
    if wp.shape[1] * 4 != K:
        raise ValueError("wp must be N x K/4")
    out = torch.empty((M, N), dtype=torch.float32, device=xq.device) if out is None else out
    _require_cuda(xq, scale, rowsum, wp, out, acc_out)
    _check(lib().bitnet_i2s_matmul_algo(_ptr(xq), _ptr(scale), _ptr(rowsum), _ptr(wp), float(w_scale),
                                        _ptr(out), _ptr(acc_out), M, N, K, ALGO[algo], _stream(stream)),
           "bitnet_i2s_matmul")
    return out


def _act_dtype(x):
    import torch

    if x.dtype == torch.float32:
        return BITNET_F32
    if x.dtype == torch.bfloat16:
        return BITNET_BF16
    raise ValueError("x must be float32 or bfloat16")


def workspace_size(M, N, K) -> int:
    n = lib().bitnet_i2s_matmul_workspace_size(M, N, K)
    if n < 0:
        raise BitnetError(int(n), "bitnet_i2s_matmul_workspace_size")
    return int(n)


def i2s_matmul_ws(xq, scale, rowsum, wp, w_scale, workspace=None, out=None, acc_out=None, stream=None):
    """The prefill path with a device workspace (allocated here from torch if not given)."""
    import torch

    M, K = xq.shape
    N = wp.shape[0]
    if wp.shape[1] * 4 != K:
        raise ValueError("wp must be N x K/4")
    need = workspace_size(M, N, K)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=xq.device)
    out = torch.empty((M, N), dtype=torch.float32, device=xq.device) if out is None else out
    _require_cuda(xq, scale, rowsum, wp, out, acc_out, workspace)
    _check(lib().bitnet_i2s_matmul_ws(_ptr(xq), _ptr(scale), _ptr(rowsum), _ptr(wp), float(w_scale), _ptr(out),
                                      _ptr(acc_out), M, N, K, _ptr(workspace),
                                      workspace.numel() * workspace.element_size(), _stream(stream)),
           "bitnet_i2s_matmul_ws")
    return out


def i2s_matmul_noalloc(xq, scale, rowsum, wp, w_scale, out=None, acc_out=None, stream=None):
    """The prefill matmul without any workspace: for callers that must not allocate device memory.

    The library's own 64 MiB device scratch array stands in for the workspace (problems that
    need more are refused); the output tensor is allocated here only if ``out`` is not given."""
    import torch

    M, K = xq.shape
    N = wp.shape[0]
    if wp.shape[1] * 4 != K:
        raise ValueError("wp must be N x K/4")
    out = torch.empty((M, N), dtype=torch.float32, device=xq.device) if out is None else out
    _require_cuda(xq, scale, rowsum, wp, out, acc_out)
    _check(lib().bitnet_i2s_matmul_noalloc(_ptr(xq), _ptr(scale), _ptr(rowsum), _ptr(wp), float(w_scale), _ptr(out),
                                           _ptr(acc_out), M, N, K, _stream(stream)),
           "bitnet_i2s_matmul_noalloc")
    return out


def linear_group(x, wps, w_scales, outs=None, accs=None, xq=None, scale=None, rowsum=None, prefetch=None,
                 stream=None):
    """Quantise x (M x K fp32/bf16) and multiply it with up to 8 packed projections sharing it.

    One kernel launch when M == 1; xq/scale/rowsum are then optional outputs. ``prefetch`` is
    an optional list of CUDA tensors (e.g. the next group's packed weights) to pull into L2
    while the kernel runs. Returns the list of M x N_l fp32 outputs."""
    import torch

    dt = _act_dtype(x)
    M, K = x.shape
    n = len(wps)
    for w in wps:
        if w.shape[1] * 4 != K:
            raise ValueError("every wp must be N x K/4")
    if outs is None:
        outs = [torch.empty((M, w.shape[0]), dtype=torch.float32, device=x.device) for w in wps]
    _require_cuda(x, xq, scale, rowsum, *wps, *outs, *(accs or []))
    P = ctypes.c_void_p * n
    wp_arr = P(*[w.data_ptr() for w in wps])
    out_arr = P(*[o.data_ptr() for o in outs])
    acc_arr = P(*[(a.data_ptr() if a is not None else None) for a in accs]) if accs is not None else None
    ws_arr = (ctypes.c_float * n)(*[float(v) for v in w_scales])
    n_arr = (ctypes.c_int64 * n)(*[int(w.shape[0]) for w in wps])
    pf = list(prefetch or [])
    pf_ptr = (ctypes.c_void_p * max(1, len(pf)))(*[t.data_ptr() for t in pf])
    pf_bytes = (ctypes.c_int64 * max(1, len(pf)))(*[t.numel() * t.element_size() for t in pf])
    _check(lib().bitnet_w2a8_linear_group_ex(_ptr(x), dt, M, K, n, wp_arr, ws_arr, n_arr, out_arr, acc_arr,
                                             _ptr(xq), _ptr(scale), _ptr(rowsum), len(pf), pf_ptr, pf_bytes,
                                             _stream(stream)),
           "bitnet_w2a8_linear_group")
    return outs


def last_device_error() -> int:
    return lib().bitnet_last_device_error()


def selftest_wait_timeout(src, max_polls, report=None, stream=None):
    """Run the failure-handling self-test: a bounded wait that runs out while a bulk copy of
    ``src`` (a CUDA tensor of 16..16384 bytes) is in flight. Returns the 3-word uint32 report
    (gave up, copy landed, wrapping word sum) as an int32 CUDA tensor."""
    import torch

    report = torch.zeros(3, dtype=torch.int32, device=src.device) if report is None else report
    _require_cuda(src, report)
    _check(lib().bitnet_selftest_wait_timeout(_ptr(src), src.numel() * src.element_size(), int(max_polls),
                                              _ptr(report), _stream(stream)),
           "bitnet_selftest_wait_timeout")
    return report


def linear(x, wp, w_scale, out=None, algo="auto", stream=None):
    """Quantise activation rows and multiply them with packed ternary weights (two launches)."""
    xq, s, rs = quant_act(x, stream=stream)
    return i2s_matmul(xq, s, rs, wp, w_scale, out=out, algo=algo, stream=stream)


def ffn_act_quant(gate, up, gamma, eps, xq=None, scale=None, rowsum=None, inner_out=None, stream=None):
    """FFN inner activation (squared-ReLU gate times up, RMS sub-norm with weight gamma and
    epsilon eps) fused with its per-token quantisation. gate, up: M x F fp32 CUDA tensors;
    gamma: F fp32. Returns (xq int8 M x F, s fp32 M, rowsum int32 M); inner_out (M x F fp32)
    is written when given."""
    import torch

    M, F = gate.shape
    if up.shape != gate.shape or gamma.shape != (F,):
        raise ValueError("gate and up must be M x F, gamma F")
    dev = gate.device
    xq = torch.empty((M, F), dtype=torch.int8, device=dev) if xq is None else xq
    scale = torch.empty(M, dtype=torch.float32, device=dev) if scale is None else scale
    rowsum = torch.empty(M, dtype=torch.int32, device=dev) if rowsum is None else rowsum
    _require_cuda(gate, up, gamma, xq, scale, rowsum, inner_out)
    _check(lib().bitnet_ffn_act_quant(_ptr(gate), _ptr(up), _ptr(gamma), float(eps), M, F, _ptr(xq), _ptr(scale),
                                      _ptr(rowsum), _ptr(inner_out), _stream(stream)),
           "bitnet_ffn_act_quant")
    return xq, scale, rowsum


def ffn_workspace_size(M, K, F) -> int:
    n = lib().bitnet_w2a8_ffn_workspace_size(M, K, F)
    if n < 0:
        raise BitnetError(int(n), "bitnet_w2a8_ffn_workspace_size")
    return int(n)


def w2a8_ffn(x, wp_gate, a_gate, wp_up, a_up, wp_down, a_down, gamma, eps, out=None, gate_out=None, up_out=None,
             xq=None, scale=None, rowsum=None, workspace=None, stream=None):
    """The FFN block: gate/up W2A8 projections of x (M x K fp32/bf16), the squared-ReLU gate
    and RMS sub-norm, then the down W2A8 projection. Returns out (M x K fp32); gate_out and
    up_out (M x F) and, when given, xq/scale/rowsum (the quantised inner rows) are written.
    For M > 1 the workspace buffers are allocated here if not given; ``workspace`` (a uint8
    CUDA tensor of at least ffn_workspace_size bytes) selects the expand-once GEMM path."""
    import torch

    dt = _act_dtype(x)
    M, K = x.shape
    F = wp_gate.shape[0]
    if wp_gate.shape != (F, K // 4) or wp_up.shape != (F, K // 4) or wp_down.shape != (K, F // 4):
        raise ValueError("wp_gate/wp_up must be F x K/4 and wp_down K x F/4")
    dev = x.device
    out = torch.empty((M, K), dtype=torch.float32, device=dev) if out is None else out
    gate_out = torch.empty((M, F), dtype=torch.float32, device=dev) if gate_out is None else gate_out
    up_out = torch.empty((M, F), dtype=torch.float32, device=dev) if up_out is None else up_out
    if M > 1:
        xq = torch.empty((M, max(K, F)), dtype=torch.int8, device=dev) if xq is None else xq
        scale = torch.empty(M, dtype=torch.float32, device=dev) if scale is None else scale
        rowsum = torch.empty(M, dtype=torch.int32, device=dev) if rowsum is None else rowsum
    _require_cuda(x, wp_gate, wp_up, wp_down, gamma, out, gate_out, up_out, xq, scale, rowsum, workspace)
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check(lib().bitnet_w2a8_ffn(_ptr(x), dt, M, K, F, _ptr(wp_gate), float(a_gate), _ptr(wp_up), float(a_up),
                                 _ptr(wp_down), float(a_down), _ptr(gamma), float(eps), _ptr(gate_out),
                                 _ptr(up_out), _ptr(out), _ptr(xq), _ptr(scale), _ptr(rowsum), _ptr(workspace),
                                 ws_bytes, _stream(stream)),
           "bitnet_w2a8_ffn")
    return out


class LinearGroupDesc(ctypes.Structure):
    """ctypes mirror of bitnet_linear_group (include/bitnet.h)."""
    _fields_ = [("x", ctypes.c_void_p), ("K", ctypes.c_int64), ("count", ctypes.c_int),
                ("wp", ctypes.c_void_p * 8), ("w_scale", ctypes.c_float * 8), ("N", ctypes.c_int64 * 8),
                ("out", ctypes.c_void_p * 8)]


class SweepPlan:
    """A persistent sweep over independent projection groups (one kernel launch per run).

    ``groups`` is a list of (x, [(wp, w_scale, out), ...]) with x a 1-D fp32 or bf16 CUDA
    tensor of K values, wp an N x K/4 uint8 tensor and out an N-element fp32 tensor. The
    tensors are bound to the plan (it keeps references to them); run() recomputes every
    group's outputs from the current contents of its x."""

    def __init__(self, groups):
        import torch

        if not groups:
            raise ValueError("at least one group")
        dt = None
        descs = (LinearGroupDesc * len(groups))()
        self._keep = []
        for g, (x, projs) in enumerate(groups):
            d = _act_dtype(x.view(1, -1))
            if dt is None:
                dt = d
            elif d != dt:
                raise ValueError("every group's x must have the same dtype")
            if not 1 <= len(projs) <= 8:
                raise ValueError("1..8 projections per group")
            K = x.numel()
            desc = descs[g]
            desc.x, desc.K, desc.count = x.data_ptr(), K, len(projs)
            for l, (wp, w_scale, out) in enumerate(projs):
                if wp.shape[1] * 4 != K or out.numel() != wp.shape[0] or out.dtype != torch.float32:
                    raise ValueError("wp must be N x K/4 and out N fp32")
                desc.wp[l], desc.w_scale[l], desc.N[l], desc.out[l] = wp.data_ptr(), float(w_scale), wp.shape[0], \
                    out.data_ptr()
            _require_cuda(x, *[t for p in projs for t in (p[0], p[2])])
            self._keep.append((x, projs))
        self._handle = ctypes.c_void_p()
        _check(lib().bitnet_sweep_plan_create(ctypes.cast(descs, ctypes.c_void_p), len(groups), dt,
                                              ctypes.byref(self._handle)),
               "bitnet_sweep_plan_create")

    def run(self, stream=None):
        _check(lib().bitnet_sweep_plan_run(self._handle, _stream(stream)), "bitnet_sweep_plan_run")

    def close(self):
        if getattr(self, "_handle", None) and self._handle.value:
            lib().bitnet_sweep_plan_destroy(self._handle)
            self._handle = ctypes.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
