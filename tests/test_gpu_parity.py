"""GPU parity: the CUDA library (through the C ABI) against the CPU oracle, element by element.

Integers (packed bytes, xq, rowsum, acc) must match bit for bit; the fp32 scale s must match
bit for bit (both sides do one IEEE divide); fp32 outputs must agree within 1e-5 relative
(they are in fact produced by the same IEEE operations in the same order, and the tests
also count exact matches). Inputs come from ternary_weight_gb300.workloads; expected values
come only from oracle/.
"""
import numpy as np
import pytest
import torch

import oracle
from ternary_weight_gb300 import _build, binding, workloads

pytestmark = pytest.mark.gpu

REL_TOL = 1e-5
NT = oracle.default_threads()


@pytest.fixture(scope="module", autouse=True)
def cuda_lib():
    if not torch.cuda.is_available():
        pytest.fail("gpu tests need a CUDA device")
    _build.build()
    binding.lib()
    yield
    assert binding.last_device_error() == 0, "a kernel recorded a device-side error"


def dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t):
    return t.cpu().numpy()


def x_device(x_np, dtype):
    if dtype == "f32":
        return dev(x_np)
    return dev(x_np.view(np.int16)).view(torch.bfloat16)


def assert_out_close(out_gpu, out_ref):
    assert out_gpu.shape == out_ref.shape
    ref = out_ref.astype(np.float64)
    got = out_gpu.astype(np.float64)
    err = np.abs(got - ref)
    bound = REL_TOL * np.abs(ref)
    bad = err > bound
    assert not bad.any(), "fp32 outputs off by more than 1e-5 rel at %d places, max rel %.3g" % (
        bad.sum(), (err / np.maximum(np.abs(ref), 1e-30)).max())


def run_chain(x_np, dtype, w_np, w_scale, algo="auto"):
    """GPU: pack -> quant -> matmul. Oracle: the same on the CPU. Returns both."""
    g_wp = binding.pack_i2s(dev(w_np))
    g_xq, g_s, g_rs = binding.quant_act(x_device(x_np, dtype))
    M, N = x_np.shape[0], w_np.shape[0]
    g_acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    g_out = binding.i2s_matmul(g_xq, g_s, g_rs, g_wp, w_scale, acc_out=g_acc, algo=algo)
    torch.cuda.synchronize()
    o_wp, _ = oracle.pack_i2s(w_np)
    o_xq, o_s, o_rs = oracle.quant_act(x_np, dtype)
    o_out, o_acc = oracle.ternary_matmul(o_xq, o_s, o_wp, w_scale, nthreads=NT)
    return (dict(wp=host(g_wp), xq=host(g_xq), s=host(g_s), rs=host(g_rs), acc=host(g_acc), out=host(g_out)),
            dict(wp=o_wp, xq=o_xq, s=o_s, rs=o_rs, acc=o_acc, out=o_out))


def assert_chain_equal(g, o):
    assert np.array_equal(g["wp"], o["wp"]), "packed bytes differ"
    assert np.array_equal(g["xq"], o["xq"]), "xq differs"
    assert np.array_equal(g["s"].view(np.uint32), o["s"].view(np.uint32)), "scale differs"
    assert np.array_equal(g["rs"], o["rs"]), "rowsum differs"
    assert np.array_equal(g["acc"], o["acc"]), "int32 accumulators differ"
    assert_out_close(g["out"], o["out"])
    assert np.array_equal(g["out"].view(np.uint32), o["out"].view(np.uint32)), "fp32 out not bit-identical"


# ----------------------------------------------------------------------------- pack

@pytest.mark.parametrize("N,K", [(1, 128), (7, 384), (640, 2560), (33, 6912), (5, 8192)])
def test_pack_parity(N, K):
    w = workloads.ternary_weights(N, K, seed=100 + N)
    assert np.array_equal(host(binding.pack_i2s(dev(w))), oracle.pack_i2s(w)[0])


def test_pack_non_ternary_count():
    w = workloads.ternary_weights(9, 256, seed=101)
    w[0, 5], w[3, 200], w[8, 255], w[2, 0] = 5, -7, 127, -128
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    g = binding.pack_i2s(dev(w), invalid_count=cnt)
    o, bad = oracle.pack_i2s(w)
    assert np.array_equal(host(g), o) and int(cnt.item()) == bad == 4


# ----------------------------------------------------------------------------- quant

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("M,K,outlier", [(1, 128, 0.0), (1, 2560, 0.0), (3, 6912, 0.01), (64, 2560, 0.01),
                                         (129, 384, 0.0), (2, 8192, 0.0), (4, 16384, 0.01), (2, 65536, 0.0)])
def test_quant_parity(dtype, M, K, outlier):
    x = workloads.activations(M, K, seed=200 + M + K, dtype=dtype, outlier_p=outlier)
    g = [host(t) for t in binding.quant_act(x_device(x, dtype))]
    o = oracle.quant_act(x, dtype)
    assert np.array_equal(g[0], o[0])
    assert np.array_equal(g[1].view(np.uint32), o[1].view(np.uint32))
    assert np.array_equal(g[2], o[2])


def test_quant_edge_rows():
    K = 256
    x = np.zeros((6, K), np.float32)
    x[1, 7] = 3e-6                          # below the 1e-5 floor
    x[2, :] = 1.0                           # constant row -> all 127
    x[3, :] = -2.5e30                       # huge values
    x[4, ::2], x[4, 1::2] = 127.0, -0.5     # s = 1 exactly: ties at -0.5 -> 0 (even)
    amax = np.array([1090775969], np.uint32).view(np.float32)[0]  # near-tie row (multiply form)
    s = np.float32(np.float32(127.0) / amax)
    x[5, 0] = amax
    x[5, 1:120] = [np.float32((k + 0.5) / float(s)) for k in range(1, 120)]
    g = [host(t) for t in binding.quant_act(dev(x))]
    o = oracle.quant_act(x)
    for a, b in zip(g, o):
        assert np.array_equal(a.view(np.uint32) if a.dtype == np.float32 else a,
                              b.view(np.uint32) if b.dtype == np.float32 else b)


# ----------------------------------------------------------------------------- matmul (full chain)

SMALL_CHAIN = [
    # (M, N, K, dtype) -- several tiles and ragged tails, oracle finishes in seconds
    (1, 1, 128, "f32"), (1, 7, 384, "f32"), (1, 2560, 2560, "f32"), (1, 640, 2560, "f32"),
    (1, 2561, 6912, "bf16"), (2, 300, 8192, "bf16"), (3, 257, 2560, "bf16"), (4, 1000, 6912, "bf16"),
    (7, 129, 1024, "f32"), (16, 700, 2560, "bf16"), (63, 300, 6912, "bf16"), (64, 513, 2560, "bf16"),
]


@pytest.mark.parametrize("M,N,K,dtype", SMALL_CHAIN)
def test_chain_parity_gemv(M, N, K, dtype):
    x = workloads.activations(M, K, seed=300 + M, dtype=dtype, outlier_p=0.01)
    w = workloads.ternary_weights(N, K, seed=301 + N)
    g, o = run_chain(x, dtype, w, workloads.weight_scale(N, K, 302), algo="gemv")
    assert_chain_equal(g, o)


# The few-token tensor-core kernel, forced: every MMA width (16/32/48/64 tokens), ragged N (a
# partial last 128-row tile), K with a half last 256-k stage, K splits over clusters of 1 to 8
# CTAs, M = 1, the decode shapes at M = 4 / 16 / 64, and more than 64 tokens in chunks of 64
# (a ragged last chunk; several chunks with clusters).
SMALLM_CHAIN = [
    (1, 256, 128, "f32"), (2, 300, 2560, "bf16"), (4, 6912, 2560, "bf16"), (8, 1000, 8192, "bf16"),
    (16, 2560, 6912, "bf16"), (17, 700, 384, "f32"), (33, 129, 1024, "bf16"), (48, 2560, 2560, "f32"),
    (63, 513, 10240, "bf16"), (64, 6912, 2560, "bf16"), (64, 2560, 6912, "bf16"), (65, 300, 2560, "bf16"),
    (100, 700, 6912, "f32"), (129, 257, 1024, "bf16"), (200, 513, 2560, "bf16"),
]


@pytest.mark.parametrize("M,N,K,dtype", SMALLM_CHAIN)
def test_chain_parity_smallm(M, N, K, dtype):
    x = workloads.activations(M, K, seed=320 + M, dtype=dtype, outlier_p=0.01)
    w = workloads.ternary_weights(N, K, seed=321 + N)
    g, o = run_chain(x, dtype, w, workloads.weight_scale(N, K, 322), algo="smallm")
    assert_chain_equal(g, o)
    assert binding.last_device_error() == 0


def test_smallm_code3_and_max_magnitude():
    """Bytes with code 3 (weight +2) and activations at +-127 everywhere: the largest exact
    accumulators the kernel can see, through the few-token path."""
    M, N, K = 16, 384, 6912
    xq = np.where(np.arange(M * K).reshape(M, K) % 3 == 0, -127, 127).astype(np.int8)
    s = np.full(M, 1.0, dtype=np.float32)
    rs = xq.astype(np.int64).sum(axis=1).astype(np.int32)
    wp = workloads.random_packed_bytes(N, K, seed=323)
    g_out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    g_acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    binding.i2s_matmul(dev(xq), dev(s), dev(rs), dev(wp), 0.5, out=g_out, acc_out=g_acc, algo="smallm")
    torch.cuda.synchronize()
    o_out, o_acc = oracle.ternary_matmul(xq, s, wp, 0.5, nthreads=NT)
    assert np.array_equal(host(g_acc), o_acc)
    assert np.array_equal(host(g_out).view(np.uint32), o_out.view(np.uint32))


# Large M = 1 matrices, every output compared: 4-40 MB of packed weights take the bulk-copy ring
# kernel (32-lane rows ragged and not, the 8-lane layout, row slices that end inside a tile); above
# 40 MB the persistent register-prefetch GEMV in its many-CTA configuration (four CTAs per SM).
@pytest.mark.parametrize("N,K", [(10000, 8192), (9800, 6912), (9729, 10240), (38920, 2560), (41000, 4096),
                                 (20003, 8448)])
def test_chain_parity_gemv_m1_large(N, K):
    x = workloads.activations(1, K, seed=310 + K, dtype="bf16", outlier_p=0.01)
    w = workloads.ternary_weights(N, K, seed=311 + N)
    g, o = run_chain(x, "bf16", w, workloads.weight_scale(N, K, 312))
    assert_chain_equal(g, o)


GEMM_CHAIN = [
    (1, 256, 128, "f32"), (65, 300, 2560, "bf16"), (127, 257, 384, "bf16"), (128, 256, 2560, "bf16"),
    (129, 513, 1024, "f32"), (200, 1000, 6912, "bf16"), (300, 700, 2560, "bf16"), (256, 640, 8192, "bf16"),
]


@pytest.mark.parametrize("M,N,K,dtype", GEMM_CHAIN)
def test_chain_parity_gemm(M, N, K, dtype):
    x = workloads.activations(M, K, seed=400 + M, dtype=dtype, outlier_p=0.0)
    w = workloads.ternary_weights(N, K, seed=401 + N)
    g, o = run_chain(x, dtype, w, workloads.weight_scale(N, K, 402), algo="gemm")
    assert_chain_equal(g, o)


# The prompt-length kernels, forced: M = 1 and M below one 128-token tile, ragged token tiles
# (129, 300), ragged weight tiles (N not a multiple of 256, N < 128), one 128-k block, K splits over
# clusters of every size the launch picks (1 to 16 CTAs: few tiles and long K), several token
# tiles with splits, the 2B-4T prefill shapes, (2200 rows over 2560) pair tiles that fill one
# whole wave and leave a ragged tail, which the CTA-pair kernel runs as a second, split-K launch,
# both sides of the pair kernel's token-tile switch (128 / 129 rows) with one 128-k block, and the
# longest K (32768) with a ragged pair tile.
PREFILL_CHAIN = [
    (1, 256, 128, "f32"), (5, 77, 2560, "bf16"), (64, 300, 384, "f32"), (127, 257, 1024, "bf16"),
    (128, 6912, 2560, "bf16"), (128, 2560, 6912, "bf16"), (129, 513, 1024, "f32"), (200, 1000, 6912, "bf16"),
    (300, 700, 2560, "bf16"), (256, 640, 8192, "bf16"), (512, 6912, 2560, "bf16"), (130, 100, 32768, "bf16"),
    (640, 2560, 1152, "f32"), (1000, 129, 256, "bf16"), (2200, 2560, 256, "f32"),
    (128, 257, 128, "bf16"), (129, 256, 128, "f32"), (65, 6912, 256, "bf16"), (300, 300, 32768, "bf16"),
]


@pytest.mark.parametrize("algo", ["prefill", "pair"])
@pytest.mark.parametrize("M,N,K,dtype", PREFILL_CHAIN)
def test_chain_parity_prefill(M, N, K, dtype, algo):
    """The prompt-length kernel and its CTA-pair variant, forced."""
    x = workloads.activations(M, K, seed=410 + M, dtype=dtype, outlier_p=0.01)
    w = workloads.ternary_weights(N, K, seed=411 + N)
    g, o = run_chain(x, dtype, w, workloads.weight_scale(N, K, 412), algo=algo)
    assert_chain_equal(g, o)
    assert binding.last_device_error() == 0


def _matmul_only(xq, s, wp, w_scale, algo):
    rs = xq.astype(np.int64).sum(axis=1).astype(np.int32)
    M, N = xq.shape[0], wp.shape[0]
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = binding.i2s_matmul(dev(xq), dev(s), dev(rs), dev(wp), w_scale, acc_out=acc, algo=algo)
    return host(out), host(acc)


@pytest.mark.parametrize("algo", ["gemv", "gemm", "prefill", "pair"])
def test_max_magnitude_accumulators(algo):
    """xq all +-127 against all-(+1) weights: |acc| = 127*K, the largest a ternary row gives."""
    K, N, M = 8192, 260, 3
    xq = np.full((M, K), 127, np.int8)
    xq[1] = -127
    xq[2, ::2] = -127
    wp, _ = oracle.pack_i2s(np.ones((N, K), np.int8))
    s = np.ones(M, np.float32)
    out, acc = _matmul_only(xq, s, wp, 1.0, algo)
    o_out, o_acc = oracle.ternary_matmul(xq, s, wp, 1.0, nthreads=NT)
    assert np.array_equal(acc, o_acc) and acc[0, 0] == 127 * K and acc[1, 0] == -127 * K
    assert np.array_equal(out.view(np.uint32), o_out.view(np.uint32))


@pytest.mark.parametrize("algo", ["gemv", "gemm", "prefill", "pair"])
@pytest.mark.parametrize("M,N,K", [(5, 77, 2560), (130, 300, 1024), (256, 1000, 32768)])
def test_random_bytes_including_code3(algo, M, N, K):
    """Arbitrary packed bytes (code 3 included, read as +2 by the c - 1 rule)."""
    wp = workloads.random_packed_bytes(N, K, seed=500 + M)
    xq = workloads.random_int8(M, K, seed=501 + M)
    s = (np.random.default_rng(502).random(M).astype(np.float32) * 3 + 0.1).astype(np.float32)
    out, acc = _matmul_only(xq, s, wp, 0.0173, algo)
    o_out, o_acc = oracle.ternary_matmul(xq, s, wp, 0.0173, nthreads=NT)
    assert np.array_equal(acc, o_acc)
    assert_out_close(out, o_out)


@pytest.mark.parametrize("M,N,K", [(512, 6912, 2560), (256, 1000, 2560), (130, 300, 1024), (640, 2562, 1152),
                                   (128, 2560, 6912), (512, 2560, 6912)])
@pytest.mark.parametrize("extreme", [False, True])
@pytest.mark.parametrize("algo", ["prefill", "pair"])
def test_prefill_outputs_without_accumulators(M, N, K, extreme, algo):
    """The call a product makes (no int32 accumulators requested) on the prompt-length kernel: the
    finish that runs only there (two values per instruction, the staged tile and its bulk stores
    when the rows are 16-byte aligned, plain stores when N % 4 != 0, split-K sums), and tokens
    whose scale lies outside [2^-100, 2^100] sharing a 32-token chunk with ordinary ones (the
    chunk then takes the IEEE division). Every output bit-identical to the oracle."""
    wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, seed=530 + N))
    xq = workloads.random_int8(M, K, seed=531 + M)
    s = (np.random.default_rng(532 + M).random(M).astype(np.float32) * 3 + 0.1).astype(np.float32)
    if extreme:
        s[3], s[M // 2], s[M - 1] = np.float32(2.0 ** -110), np.float32(2.0 ** 110), np.float32(2.0 ** -101)
    rs = xq.astype(np.int64).sum(axis=1).astype(np.int32)
    out = binding.i2s_matmul(dev(xq), dev(s), dev(rs), dev(wp), 0.0173, algo=algo)
    o_out, _ = oracle.ternary_matmul(xq, s, wp, 0.0173, nthreads=NT)
    got = host(out)
    assert np.array_equal(got.view(np.uint32), o_out.view(np.uint32))
    assert binding.last_device_error() == 0


@pytest.mark.parametrize("M", [1, 2, 3, 63, 64, 65, 127, 128, 129])
def test_gemv_and_gemm_agree(M):
    K, N = 2560, 600
    xq = workloads.random_int8(M, K, seed=600 + M)
    wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, 601))
    s = np.full(M, 1.7, np.float32)
    a = _matmul_only(xq, s, wp, 0.02, "gemv")
    b = _matmul_only(xq, s, wp, 0.02, "gemm")
    assert np.array_equal(a[1], b[1]) and np.array_equal(a[0].view(np.uint32), b[0].view(np.uint32))


def test_misaligned_pointer_is_rejected():
    xq = torch.zeros(2 * 128 + 16, dtype=torch.int8, device="cuda")
    wp = torch.zeros((4, 32), dtype=torch.uint8, device="cuda")
    s = torch.ones(1, device="cuda")
    rs = torch.zeros(1, dtype=torch.int32, device="cuda")
    bad = xq[1:129].view(1, 128)
    with pytest.raises(binding.BitnetError) as e:
        binding.i2s_matmul(bad, s, rs, wp, 1.0)
    assert e.value.status == binding.BITNET_EALIGN


# ----------------------------------------------------------------------------- full-size configs

_ORACLE_FULL = {}


def _oracle_full_size(case):
    """The oracle's pack, quantisation and matmul of a full-size case (every output), computed
    once per case and shared by the kernel paths that are checked on it."""
    if case.name not in _ORACLE_FULL:
        x, w = case.x(), case.weights()
        o_wp, _ = oracle.pack_i2s(w)
        o_xq, o_s, o_rs = oracle.quant_act(x, case.act_dtype)
        o_out, o_acc = oracle.ternary_matmul(o_xq, o_s, o_wp, case.w_scale(), nthreads=NT)
        _ORACLE_FULL.clear()  # keep one case resident at a time
        _ORACLE_FULL[case.name] = dict(wp=o_wp, xq=o_xq, s=o_s, rs=o_rs, out=o_out, acc=o_acc)
    return _ORACLE_FULL[case.name]


def _full_size(case, path="auto"):
    """Full-size GPU run through the C ABI, every element compared with the oracle: packed
    bytes, xq, s, rowsum, the int32 accumulators and the fp32 outputs, bit for bit. ``path`` is
    a kernel choice of bitnet_i2s_matmul_algo or "ws" (bitnet_i2s_matmul_ws)."""
    x, w, ws = case.x(), case.weights(), case.w_scale()
    g_wp = binding.pack_i2s(dev(w))
    g_xq, g_s, g_rs = binding.quant_act(x_device(x, case.act_dtype))
    g_acc = torch.empty((case.M, case.N), dtype=torch.int32, device="cuda")
    if path == "ws":
        g_out = binding.i2s_matmul_ws(g_xq, g_s, g_rs, g_wp, ws, acc_out=g_acc)
    else:
        g_out = binding.i2s_matmul(g_xq, g_s, g_rs, g_wp, ws, acc_out=g_acc, algo=path)
    torch.cuda.synchronize()
    o = _oracle_full_size(case)
    assert np.array_equal(host(g_wp), o["wp"])
    assert np.array_equal(host(g_xq), o["xq"])
    assert np.array_equal(host(g_s).view(np.uint32), o["s"].view(np.uint32))
    assert np.array_equal(host(g_rs), o["rs"])
    assert np.array_equal(host(g_acc), o["acc"])
    out = host(g_out)
    assert_out_close(out, o["out"])
    assert np.array_equal(out.view(np.uint32), o["out"].view(np.uint32))
    assert binding.last_device_error() == 0


@pytest.mark.parametrize("case", [workloads.single_gemv()] + workloads.batched_decode_cases()
                         + workloads.prefill_cases() + workloads.large_cases(), ids=lambda c: c.name)
def test_full_size_configs(case):
    """Every configuration at full size, in the launch configuration the plain call uses."""
    _full_size(case)


FULL_PREFILL_PATHS = [(c, p) for c in workloads.prefill_cases() + workloads.large_cases()[:1]
                      for p in ("smallm", "ws", "prefill")]


@pytest.mark.parametrize("case,path", FULL_PREFILL_PATHS, ids=lambda v: v if isinstance(v, str) else v.name)
def test_full_size_prefill_paths(case, path):
    """The prefill configurations (M = 128, 512 and 4096) through each tensor-core path the
    library offers for them, every element against the oracle."""
    _full_size(case, path)


# ----------------------------------------------------------------------------- fused, grouped linear

@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K,Ns", [(128, [1]), (384, [5, 17]), (2560, [2560, 640, 640]), (2560, [6912, 6912]),
                                  (6912, [2560]), (8192, [3000, 1]), (10240, [300]), (1152, [77]),
                                  (2560, [7, 64, 100, 33, 2, 640, 1, 257])])
def test_linear_group_m1_fused(dtype, K, Ns):
    """One launch: quantisation + up to 8 projections; every output, accumulator and the
    published xq / s / rowsum against the oracle."""
    x = workloads.activations(1, K, seed=800 + K, dtype=dtype, outlier_p=0.01)
    ws = [workloads.ternary_weights(N, K, seed=801 + i) for i, N in enumerate(Ns)]
    scales = [workloads.weight_scale(N, K, seed=830 + i) for i, N in enumerate(Ns)]
    wps = [binding.pack_i2s(dev(w)) for w in ws]
    accs = [torch.empty((1, N), dtype=torch.int32, device="cuda") for N in Ns]
    xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    rs = torch.empty(1, dtype=torch.int32, device="cuda")
    outs = binding.linear_group(x_device(x, dtype), wps, scales, accs=accs, xq=xq, scale=s, rowsum=rs)
    torch.cuda.synchronize()
    o_xq, o_s, o_rs = oracle.quant_act(x, dtype)
    assert np.array_equal(host(xq), o_xq)
    assert np.array_equal(host(s).view(np.uint32), o_s.view(np.uint32))
    assert np.array_equal(host(rs), o_rs)
    for w, sc, out, acc in zip(ws, scales, outs, accs):
        o_out, o_acc = oracle.ternary_matmul(o_xq, o_s, oracle.pack_i2s(w)[0], sc, nthreads=NT)
        assert np.array_equal(host(acc), o_acc)
        assert np.array_equal(host(out).view(np.uint32), o_out.view(np.uint32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_linear_group_m1_rounding_ties(dtype):
    """max|x| = 127 makes s = 1 exactly, so every x = k + 0.5 is a rounding tie: the fused
    quantisation must round each to the even neighbour, as the oracle does."""
    K = 2560
    rng = np.random.default_rng(870)
    halves = (rng.integers(-126, 126, size=K) + 0.5).astype(np.float32)
    ints = rng.integers(-127, 128, size=K).astype(np.float32)
    x = np.where(rng.random(K) < 0.7, halves, ints).astype(np.float32)
    x[17] = 127.0
    x = x.reshape(1, K)
    tie = np.abs(x - np.trunc(x)) == 0.5  # every such value is exact in bf16 too (|x| < 128)
    if dtype == "bf16":
        x = workloads.to_bf16_bits(x)
    ws = [workloads.ternary_weights(N, K, seed=871 + i) for i, N in enumerate([640, 2560])]
    wps = [binding.pack_i2s(dev(w)) for w in ws]
    accs = [torch.empty((1, w.shape[0]), dtype=torch.int32, device="cuda") for w in ws]
    xq = torch.empty((1, K), dtype=torch.int8, device="cuda")
    s = torch.empty(1, dtype=torch.float32, device="cuda")
    rs = torch.empty(1, dtype=torch.int32, device="cuda")
    outs = binding.linear_group(x_device(x, dtype), wps, [0.02, 0.03], accs=accs, xq=xq, scale=s, rowsum=rs)
    torch.cuda.synchronize()
    o_xq, o_s, o_rs = oracle.quant_act(x, dtype)
    assert o_s[0] == 1.0 and tie.sum() > K // 2 and np.all(o_xq[tie] % 2 == 0)  # ties went to even codes
    assert np.array_equal(host(xq), o_xq)
    assert np.array_equal(host(rs), o_rs)
    for w, sc, out, acc in zip(ws, [0.02, 0.03], outs, accs):
        o_out, o_acc = oracle.ternary_matmul(o_xq, o_s, oracle.pack_i2s(w)[0], sc, nthreads=NT)
        assert np.array_equal(host(acc), o_acc)
        assert np.array_equal(host(out).view(np.uint32), o_out.view(np.uint32))


def test_linear_group_m1_without_quant_outputs():
    K, Ns = 2560, [2560, 640]
    x = workloads.activations(1, K, seed=850, dtype="f32")
    ws = [workloads.ternary_weights(N, K, seed=851 + i) for i, N in enumerate(Ns)]
    outs = binding.linear_group(dev(x), [binding.pack_i2s(dev(w)) for w in ws], [0.02, 0.03])
    torch.cuda.synchronize()
    o_xq, o_s, _ = oracle.quant_act(x)
    for w, sc, out in zip(ws, [0.02, 0.03], outs):
        o_out, _ = oracle.ternary_matmul(o_xq, o_s, oracle.pack_i2s(w)[0], sc, nthreads=NT)
        assert_out_close(host(out), o_out)


@pytest.mark.parametrize("M,K", [(3, 2560), (130, 1024), (1, 16384)])
def test_linear_group_two_launch_path(M, K):
    """M > 1 (or K beyond the single-launch kernel): quantisation then one matmul per projection."""
    x = workloads.activations(M, K, seed=860 + M, dtype="bf16")
    Ns = [300, 129]
    ws = [workloads.ternary_weights(N, K, seed=861 + i) for i, N in enumerate(Ns)]
    xq = torch.empty((M, K), dtype=torch.int8, device="cuda")
    s = torch.empty(M, dtype=torch.float32, device="cuda")
    rs = torch.empty(M, dtype=torch.int32, device="cuda")
    accs = [torch.empty((M, N), dtype=torch.int32, device="cuda") for N in Ns]
    outs = binding.linear_group(x_device(x, "bf16"), [binding.pack_i2s(dev(w)) for w in ws], [0.02, 0.03],
                                accs=accs, xq=xq, scale=s, rowsum=rs)
    torch.cuda.synchronize()
    o_xq, o_s, _ = oracle.quant_act(x, "bf16")
    assert np.array_equal(host(xq), o_xq)
    for w, sc, out, acc in zip(ws, [0.02, 0.03], outs, accs):
        o_out, o_acc = oracle.ternary_matmul(o_xq, o_s, oracle.pack_i2s(w)[0], sc, nthreads=NT)
        assert np.array_equal(host(acc), o_acc)
        assert_out_close(host(out), o_out)


def test_linear_group_requires_workspace_beyond_single_launch():
    x = torch.zeros((2, 256), device="cuda")
    wp = torch.zeros((4, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.BitnetError) as e:
        binding.linear_group(x, [wp], [1.0])
    assert e.value.status == binding.BITNET_EINVAL


def test_stack_fused_equals_unfused():
    """The decode stack's fused step and its two-launch step give identical outputs."""
    from ternary_weight_gb300.stack import Group, PackedLinear, TernaryStack

    groups = []
    for gi, (K, Ns) in enumerate([(2560, [2560, 640, 640]), (2560, [2560]), (2560, [6912, 6912]), (6912, [2560])]):
        lins = [PackedLinear.from_ternary("p%d_%d" % (gi, i), dev(workloads.ternary_weights(N, K, 870 + 10 * gi + i)),
                                          0.01 + 0.001 * i) for i, N in enumerate(Ns)]
        groups.append(Group("g%d" % gi, K, lins))
    outs = []
    for fused in (True, False):
        st = TernaryStack(groups, M=1, fused=fused)
        xs = np.concatenate([workloads.activations_f32(1, g.K, 890 + i).ravel() for i, g in enumerate(groups)])
        st.x_all.copy_(torch.from_numpy(xs))
        st.step()
        torch.cuda.synchronize()
        outs.append(host(st.out_all))
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))


def test_linear_group_prefetch_hint_changes_nothing():
    K, Ns = 2560, [6912, 6912]
    x = workloads.activations(1, K, seed=880, dtype="f32")
    wps = [binding.pack_i2s(dev(workloads.ternary_weights(N, K, seed=881 + i))) for i, N in enumerate(Ns)]
    other = [binding.pack_i2s(dev(workloads.ternary_weights(2560, 6912, seed=883)))]
    a = binding.linear_group(dev(x), wps, [0.02, 0.03])
    b = binding.linear_group(dev(x), wps, [0.02, 0.03], prefetch=other + wps)
    torch.cuda.synchronize()
    for u, v in zip(a, b):
        assert np.array_equal(host(u).view(np.uint32), host(v).view(np.uint32))


# ----------------------------------------------------------------------------- prefill with workspace

@pytest.mark.parametrize("M,N,K", [(1, 256, 128), (65, 300, 2560), (128, 256, 2560), (129, 513, 1024),
                                   (200, 1000, 6912), (512, 2560, 6912), (300, 6912, 2560), (256, 640, 8192)])
def test_matmul_ws_parity(M, N, K):
    x = workloads.activations(M, K, seed=900 + M, dtype="bf16")
    w = workloads.ternary_weights(N, K, seed=901 + N)
    ws = workloads.weight_scale(N, K, 902)
    g_wp = binding.pack_i2s(dev(w))
    g_xq, g_s, g_rs = binding.quant_act(x_device(x, "bf16"))
    g_acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    g_out = binding.i2s_matmul_ws(g_xq, g_s, g_rs, g_wp, ws, acc_out=g_acc)
    torch.cuda.synchronize()
    o_xq, o_s, _ = oracle.quant_act(x, "bf16")
    o_out, o_acc = oracle.ternary_matmul(o_xq, o_s, oracle.pack_i2s(w)[0], ws, nthreads=NT)
    assert np.array_equal(host(g_acc), o_acc)
    assert np.array_equal(host(g_out).view(np.uint32), o_out.view(np.uint32))


def test_matmul_ws_random_bytes_and_max_magnitude():
    M, N, K = 130, 300, 8192
    xq = workloads.random_int8(M, K, seed=910)
    xq[0, :] = 127
    xq[1, :] = -127
    wp = workloads.random_packed_bytes(N, K, seed=911)
    wp[0, :] = 0xAA  # all codes 2: acc = 127*K and -127*K in rows 0 and 1
    s = np.full(M, 0.75, np.float32)
    rs = xq.astype(np.int64).sum(axis=1).astype(np.int32)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = binding.i2s_matmul_ws(dev(xq), dev(s), dev(rs), dev(wp), 0.013, acc_out=acc)
    torch.cuda.synchronize()
    o_out, o_acc = oracle.ternary_matmul(xq, s, wp, 0.013, nthreads=NT)
    assert np.array_equal(host(acc), o_acc) and o_acc[0, 0] == 127 * K and o_acc[1, 0] == -127 * K
    assert_out_close(host(out), o_out)


def test_matmul_ws_two_calls_reuse_workspace():
    M, N, K = 256, 512, 2560
    wsbuf = torch.empty(binding.workspace_size(M, N, K), dtype=torch.uint8, device="cuda")
    for seed in (920, 921):
        xq = workloads.random_int8(M, K, seed=seed)
        wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, seed + 5))
        s = np.full(M, 1.25, np.float32)
        rs = xq.astype(np.int64).sum(axis=1).astype(np.int32)
        out = binding.i2s_matmul_ws(dev(xq), dev(s), dev(rs), dev(wp), 0.02, workspace=wsbuf)
        torch.cuda.synchronize()
        o_out, _ = oracle.ternary_matmul(xq, s, wp, 0.02, nthreads=NT)
        assert np.array_equal(host(out).view(np.uint32), o_out.view(np.uint32))


# ----------------------------------------------------------------------------- weight ternarisation

QW_CASES = [
    # (N, K, dtype, mode): one block, ragged N, the 2B-4T shapes, a 100B-class row length
    (1, 128, "f32", "absmean"), (7, 384, "bf16", "absmean"), (640, 2560, "f32", "absmean"),
    (2560, 6912, "bf16", "absmean"), (33, 8192, "f32", "absmean"), (129, 10240, "bf16", "absmean"),
    (300, 2560, "f32", "sign"), (65, 640, "bf16", "sign"), (2560, 2560, "f32", "sign"),
]


def _qw_inputs(N, K, dtype, mode, seed):
    w = (workloads.source_weights_f32(N, K, seed) if mode == "absmean"
         else workloads.near_ternary_weights_f32(N, K, seed))
    return (w, w) if dtype == "f32" else (workloads.to_bf16_bits(w), workloads.to_bf16_bits(w))


@pytest.mark.parametrize("N,K,dtype,mode", QW_CASES)
def test_quant_weight_parity(N, K, dtype, mode):
    """Packed bytes and the scale's bit pattern, against the oracle's ternarisation + pack."""
    w_np, w_dev = _qw_inputs(N, K, dtype, mode, seed=400 + N)
    g_wp, g_s = binding.quant_weight(x_device(w_dev, dtype), mode=mode)
    torch.cuda.synchronize()
    o_q, o_s = oracle.quant_weight(w_np, dtype=dtype, mode=mode)
    assert np.array_equal(host(g_s).view(np.uint32), np.array([o_s], dtype=np.float32).view(np.uint32))
    assert np.array_equal(host(g_wp), oracle.pack_i2s(o_q)[0])
    assert binding.last_device_error() == 0


def test_quant_weight_all_zero_and_ties():
    # all zero: the 1e-5 floor, every code 1 (weight 0)
    g_wp, g_s = binding.quant_weight(torch.zeros((5, 256), dtype=torch.float32, device="cuda"))
    torch.cuda.synchronize()
    assert host(g_s)[0] == np.float32(1e-5) and np.all(host(g_wp) == 0x55)
    # mean |w| = 1 exactly: +-0.5 round to even (0), +-1.5 to +-2 and clip to +-1
    w = np.tile(np.array([0.5, -0.5, 1.5, -1.5], dtype=np.float32), (3, 64))
    g_wp, g_s = binding.quant_weight(dev(w))
    torch.cuda.synchronize()
    o_q, o_s = oracle.quant_weight(w)
    assert o_s == 1.0 and host(g_s)[0] == 1.0
    assert np.array_equal(host(g_wp), oracle.pack_i2s(o_q)[0])


def test_quant_weight_full_exponent_range():
    """Magnitudes from subnormal to just under 2^12: every part of the 128-bit fixed-point sum,
    the floor of values below 2^-74, and codes far from the thresholds."""
    rng = np.random.default_rng(420)
    N, K = 37, 1280
    e = rng.uniform(-149.0, 11.99, size=(N, K))
    w = (np.exp2(e) * rng.choice([-1.0, 1.0], size=(N, K))).astype(np.float32)
    w[0, :4] = [0.0, -0.0, np.float32(2.0 ** -149), np.float32(2.0 ** -74)]
    for dtype in ("f32", "bf16"):
        top = np.float32(4095.9997) if dtype == "f32" else np.float32(4080.0)  # largest in range
        w[0, 4:6] = [top, -top]
        w_dev = w if dtype == "f32" else workloads.to_bf16_bits(w)
        g_wp, g_s = binding.quant_weight(x_device(w_dev, dtype))
        torch.cuda.synchronize()
        o_q, o_s = oracle.quant_weight(w_dev, dtype=dtype)
        assert np.array_equal(host(g_s).view(np.uint32), np.array([o_s], dtype=np.float32).view(np.uint32))
        assert np.array_equal(host(g_wp), oracle.pack_i2s(o_q)[0])
    assert binding.last_device_error() == 0


def _absmean_threshold(scale):
    """Largest fp32 T with T <= scale * (1/2 + 2^-25): rne(fl(w / scale)) is +1 exactly for w > T."""
    from fractions import Fraction
    c = Fraction(float(scale)) * (Fraction(1, 2) + Fraction(1, 2 ** 25))
    t = np.float32(float(c))
    return np.nextafter(t, np.float32(0)) if Fraction(float(t)) > c else t


def test_quant_weight_codes_at_the_rounding_boundary():
    """Weights placed on and next to the +-1/2 rounding boundary of w / scale (the scale is
    iterated to a fixed point so the placed values sit on the boundary of the final scale)."""
    N, K = 16, 512
    w = workloads.source_weights_f32(N, K, 430)
    _, s = oracle.quant_weight(w)
    for _ in range(20):
        t = _absmean_threshold(s)
        edge = np.array([t, np.nextafter(t, np.float32(1)), np.nextafter(t, np.float32(0)), s / 2,
                         np.nextafter(s / 2, np.float32(1))], dtype=np.float32)
        w[:, :5] = edge
        w[:, 5:10] = -edge
        _, s_new = oracle.quant_weight(w)
        if s_new == s:
            break
        s = s_new
    assert s_new == s, "scale did not settle"
    o_q, o_s = oracle.quant_weight(w)
    # the boundary really is exercised: T codes 0, the float above T codes +1
    assert list(o_q[0, :3]) == [0, 1, 0] and list(o_q[0, 5:8]) == [0, -1, 0]
    g_wp, g_s = binding.quant_weight(dev(w))
    torch.cuda.synchronize()
    assert host(g_s)[0] == o_s
    assert np.array_equal(host(g_wp), oracle.pack_i2s(o_q)[0])


@pytest.mark.parametrize("bad", [4096.0, float("inf"), float("nan")])
def test_quant_weight_range_error_is_reported(bad):
    """|w| >= 2^12, inf or NaN under AbsMean: BITNET_ERANGE in the device error word and a NaN
    scale; the word is cleared by the read and the next call is clean."""
    w = workloads.source_weights_f32(9, 256, 440)
    w[4, 100] = np.float32(bad)
    _, g_s = binding.quant_weight(dev(w))
    torch.cuda.synchronize()
    assert np.isnan(host(g_s)[0])
    assert binding.last_device_error() == binding.BITNET_ERANGE
    assert binding.last_device_error() == 0
    w[4, 100] = np.float32(4095.9997)  # the largest magnitude still in range
    g_wp, g_s = binding.quant_weight(dev(w))
    torch.cuda.synchronize()
    o_q, o_s = oracle.quant_weight(w)
    assert host(g_s)[0] == o_s and np.array_equal(host(g_wp), oracle.pack_i2s(o_q)[0])
    assert binding.last_device_error() == 0


def test_quant_weight_then_matmul_chain():
    """fp32 source weights -> ternarise + pack -> matmul with the returned scale, end to end."""
    M, N, K = 3, 700, 2560
    w = workloads.source_weights_f32(N, K, 410)
    x = workloads.activations(M, K, seed=411, dtype="f32")
    g_wp, g_s = binding.quant_weight(dev(w))
    g_xq, g_sx, g_rs = binding.quant_act(dev(x))
    torch.cuda.synchronize()
    scale = float(host(g_s)[0])
    g_out = binding.i2s_matmul(g_xq, g_sx, g_rs, g_wp, scale)
    torch.cuda.synchronize()
    o_q, o_s = oracle.quant_weight(w)
    o_xq, o_sx, _ = oracle.quant_act(x)
    o_out, _ = oracle.ternary_matmul(o_xq, o_sx, oracle.pack_i2s(o_q)[0], float(o_s), nthreads=NT)
    assert scale == o_s
    assert np.array_equal(host(g_out).view(np.uint32), o_out.view(np.uint32))


# ----------------------------------------------------------------------------- FFN block

def _ffn_gamma(F, seed):
    return workloads.rmsnorm_gamma(F, seed)


# The FFN inner row's sum of squares has no order on the page. The oracle takes the plain
# ascending sum in double, rounded once; the kernels add fp32 partials in a fixed order of
# their own, at most F/256 + 8 roundings per term for F <= 32768, so their ss is within
# 136 * 2^-24 = 8.1e-6 relative of the oracle's. That moves c = 1/sqrt(ss/F + eps) by at most
# half as much, and inner = (h * c) * gamma by that plus a few roundings: below 1e-5 relative.
# The codes are decided by inner * s; both factors move by at most 1e-5, so a code may differ
# only where the oracle's product lies within 2e-5 relative of a rounding boundary, and then
# only to the neighbour on the other side.
FFN_REL = 1e-5


def assert_ffn_inner_close(g_inner, o_inner):
    err = np.abs(g_inner.astype(np.float64) - o_inner.astype(np.float64))
    bad = err > FFN_REL * np.abs(o_inner.astype(np.float64))
    assert not bad.any(), "inner off by more than %g rel at %d places" % (FFN_REL, bad.sum())


def assert_quant_of_inner_valid(g_xq, g_s, g_rs, o_inner):
    """The GPU's quantisation of its own inner rows against the oracle's quantisation of the
    oracle's inner rows: s within FFN_REL relative; every code equal to the oracle's, except
    within 2 * FFN_REL of a rounding boundary, where either neighbour is accepted; the row sum
    equal to the sum of the GPU's own codes. Returns the number of codes that differ."""
    o_xq, o_s, _ = oracle.quant_act(o_inner)
    s64, os64 = g_s.astype(np.float64), o_s.astype(np.float64)
    assert np.all(np.abs(s64 - os64) <= FFN_REL * os64), "act scale off by more than %g rel" % FFN_REL
    p = o_inner.astype(np.float64) * os64[:, None]
    w = 2 * FFN_REL * np.abs(p) + 1e-12
    lo = np.clip(np.rint(p - w), -127, 127)
    hi = np.clip(np.rint(p + w), -127, 127)
    g = g_xq.astype(np.float64)
    assert np.all((g == lo) | (g == hi)), "a code differs from the oracle's away from a rounding boundary"
    assert np.array_equal(g_rs, g_xq.astype(np.int64).sum(axis=1).astype(np.int32)), "rowsum is not the sum of xq"
    return int(np.count_nonzero(g_xq != o_xq))


@pytest.mark.parametrize("M,F,eps", [
    (1, 128, 1e-5), (3, 6912, 1e-5), (5, 1152, 0.25), (2, 28672, 1e-5), (7, 32768, 1e-6), (300, 2560, 1e-5),
])
def test_ffn_act_quant_parity(M, F, eps):
    """inner, xq, s and rowsum of the fused sub-norm + quantisation kernel against
    oracle.ffn_inner followed by oracle.quant_act, within the bound stated above."""
    rng = np.random.default_rng(500 + F + M)
    g = (rng.standard_normal((M, F)) * 1.5).astype(np.float32)
    u = rng.standard_normal((M, F)).astype(np.float32)
    gamma = _ffn_gamma(F, 501)
    inner = torch.empty((M, F), dtype=torch.float32, device="cuda")
    g_xq, g_s, g_rs = binding.ffn_act_quant(dev(g), dev(u), dev(gamma), eps, inner_out=inner)
    torch.cuda.synchronize()
    o_inner = oracle.ffn_inner(g, u, gamma, eps)
    assert_ffn_inner_close(host(inner), o_inner)
    assert_quant_of_inner_valid(host(g_xq), host(g_s), host(g_rs), o_inner)


def test_ffn_act_quant_degenerate_rows():
    """All gates non-positive (inner = 0: s at the 1e-5 floor, every code 0), a single positive
    gate (one code at +-127), and a row with huge and tiny h side by side."""
    F = 1024
    g = np.full((3, F), -1.0, np.float32)
    u = np.ones((3, F), np.float32)
    g[1, 77] = 2.0
    rng = np.random.default_rng(510)
    g[2] = rng.standard_normal(F).astype(np.float32)
    g[2, :8] = [1e6, 1e-6, 3e5, -2.0, 7e-8, 1.0, 1e4, 5e-3]
    gamma = _ffn_gamma(F, 511)
    g_xq, g_s, g_rs = binding.ffn_act_quant(dev(g), dev(u), dev(gamma), 1e-5)
    torch.cuda.synchronize()
    o_inner = oracle.ffn_inner(g, u, gamma, 1e-5)
    o_xq, o_s, o_rs = oracle.quant_act(o_inner)
    assert np.all(o_xq[0] == 0) and o_s[0] == np.float32(127.0) / np.float32(1e-5)
    assert abs(int(o_xq[1, 77])) == 127
    gx = host(g_xq)
    assert np.all(gx[0] == 0) and host(g_s)[0] == o_s[0]
    assert abs(int(gx[1, 77])) == 127 and np.count_nonzero(gx[1]) == 1
    assert_quant_of_inner_valid(gx, host(g_s), host(g_rs), o_inner)


def _ffn_oracle_front(x_np, dtype, wg, ag, wu, au, gamma, eps):
    """The FFN block's first half on the CPU: quant_act -> gate/up matmuls -> ffn_inner."""
    xq, s, _ = oracle.quant_act(x_np, dtype)
    gate, _ = oracle.ternary_matmul(xq, s, oracle.pack_i2s(wg)[0], ag, nthreads=NT)
    up, _ = oracle.ternary_matmul(xq, s, oracle.pack_i2s(wu)[0], au, nthreads=NT)
    return gate, up, oracle.ffn_inner(gate, up, gamma, eps)


def check_ffn_block(x_np, dtype, wg, ag, wu, au, wd, ad, gamma, eps, g_gate, g_up, g_xq, g_s, g_rs, g_out):
    """gate/up bit for bit; the quantised inner rows valid against the oracle's inner rows;
    the block output bit for bit equal to the oracle's down projection of the GPU's own codes
    and scales (so the down matmul is checked exactly whatever codes sat on a boundary)."""
    o_gate, o_up, o_inner = _ffn_oracle_front(x_np, dtype, wg, ag, wu, au, gamma, eps)
    assert np.array_equal(g_gate.view(np.uint32), o_gate.view(np.uint32))
    assert np.array_equal(g_up.view(np.uint32), o_up.view(np.uint32))
    assert_quant_of_inner_valid(g_xq, g_s, g_rs, o_inner)
    o_out, _ = oracle.ternary_matmul(g_xq, g_s, oracle.pack_i2s(wd)[0], ad, nthreads=NT)
    assert np.array_equal(g_out.view(np.uint32), o_out.view(np.uint32))


FFN_CASES = [
    # (M, K, F, dtype, workspace): the two-launch path (M = 1, including a row too long for
    # the registers, F = 10240), the few-token path (more than 64 rows in chunks), the
    # prompt-length kernels (from 128 rows; the CTA-pair kernel from 192), and a call that passes
    # a workspace (which the block no longer needs: its size is 0)
    (1, 2560, 6912, "f32", False), (1, 2560, 6912, "bf16", False), (1, 512, 10240, "f32", False),
    (1, 1024, 128, "bf16", False), (2, 2560, 6912, "bf16", False), (17, 640, 1280, "f32", False),
    (65, 2560, 6912, "bf16", False), (130, 1024, 2048, "f32", False), (512, 1024, 2048, "bf16", False),
    (2048, 512, 1024, "bf16", True),
]


def _run_ffn(x_np, dtype, wg, ag, wu, au, wd, ad, gamma, eps, use_ws):
    M, K = x_np.shape
    F = wg.shape[0]
    g_wg, g_wu, g_wd = binding.pack_i2s(dev(wg)), binding.pack_i2s(dev(wu)), binding.pack_i2s(dev(wd))
    gate = torch.empty((M, F), dtype=torch.float32, device="cuda")
    up = torch.empty((M, F), dtype=torch.float32, device="cuda")
    xq = torch.empty((M, max(K, F)), dtype=torch.int8, device="cuda")
    s = torch.empty(M, dtype=torch.float32, device="cuda")
    rs = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = None
    if use_ws:
        ws = torch.empty(binding.ffn_workspace_size(M, K, F), dtype=torch.uint8, device="cuda")
    g_out = binding.w2a8_ffn(x_device(x_np, dtype), g_wg, ag, g_wu, au, g_wd, ad, dev(gamma), eps,
                             gate_out=gate, up_out=up, xq=xq, scale=s, rowsum=rs, workspace=ws)
    torch.cuda.synchronize()
    # the workspace holds the quantised inner rows as a contiguous M x F array at its start
    return (host(gate), host(up), host(xq).reshape(-1)[:M * F].reshape(M, F), host(s), host(rs), host(g_out))


@pytest.mark.parametrize("M,K,F,dtype,use_ws", FFN_CASES)
def test_w2a8_ffn_parity(M, K, F, dtype, use_ws):
    """gate/up outputs and the block output bit for bit, the quantised inner rows valid."""
    seed = 520 + M + F
    x_np = workloads.activations(M, K, seed, dtype)
    wg = workloads.ternary_weights(F, K, seed + 1)
    wu = workloads.ternary_weights(F, K, seed + 2)
    wd = workloads.ternary_weights(K, F, seed + 3)
    ag, au, ad = (workloads.weight_scale(F, K, seed + 4), workloads.weight_scale(F, K, seed + 5),
                  workloads.weight_scale(K, F, seed + 6))
    gamma = _ffn_gamma(F, seed + 7)
    eps = 1e-5
    got = _run_ffn(x_np, dtype, wg, ag, wu, au, wd, ad, gamma, eps, use_ws)
    check_ffn_block(x_np, dtype, wg, ag, wu, au, wd, ad, gamma, eps, *got)
    assert binding.last_device_error() == 0


# ----------------------------------------------------------------------------- persistent sweep

SWEEP_CASES = [
    # (name, dtype, [(K, [N, ...]), ...]) -- mixed K, ragged N, groups split across CTAs and CTAs
    # spanning many groups, the smallest and largest K
    ("mixed", "f32", [(2560, [2560, 640, 640]), (2560, [2560]), (2560, [6912, 6912]), (6912, [2560])]),
    ("ragged", "bf16", [(384, [7]), (128, [1, 3]), (10240, [33]), (1152, [300, 5, 77]), (640, [1000])]),
    ("many_small", "f32", [(256 * (1 + i % 5), [1 + (37 * i) % 53] * (1 + i % 3)) for i in range(150)]),
    ("big_rows", "bf16", [(8192, [28672 // 8]), (10240, [1500])]),
]


@pytest.mark.parametrize("name,dtype,spec", SWEEP_CASES, ids=[c[0] for c in SWEEP_CASES])
def test_sweep_plan_parity(name, dtype, spec):
    """Every group's outputs, bit for bit, against oracle.quant_act + oracle.ternary_matmul."""
    groups, expect = [], []
    for gi, (K, Ns) in enumerate(spec):
        seed = 600 + 10 * gi
        x_np = workloads.activations(1, K, seed, dtype)
        projs, refs = [], []
        xq, s, _ = oracle.quant_act(x_np, dtype)
        for li, N in enumerate(Ns):
            w = workloads.ternary_weights(N, K, seed + 1 + li)
            ws = workloads.weight_scale(N, K, seed + 5 + li)
            out = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
            projs.append((binding.pack_i2s(dev(w)), ws, out))
            o_out, _ = oracle.ternary_matmul(xq, s, oracle.pack_i2s(w)[0], ws, nthreads=NT)
            refs.append(o_out[0])
        groups.append((x_device(x_np, dtype).view(-1), projs))
        expect.append(refs)
    plan = binding.SweepPlan(groups)
    plan.run()
    torch.cuda.synchronize()
    for (x, projs), refs in zip(groups, expect):
        for (_, _, out), ref in zip(projs, refs):
            assert np.array_equal(host(out).view(np.uint32), ref.view(np.uint32))
    # a second run over changed inputs recomputes everything (the plan binds buffers, not values)
    for gi, (x, projs) in enumerate(groups):
        x.copy_(x_device(workloads.activations(1, x.numel(), 900 + gi, dtype), dtype).view(-1))
    plan.run()
    torch.cuda.synchronize()
    for gi, ((x, projs), (K, Ns)) in enumerate(zip(groups, spec)):
        xq, s, _ = oracle.quant_act(workloads.activations(1, K, 900 + gi, dtype), dtype)
        for li, (_, ws, out) in enumerate(projs):
            w = workloads.ternary_weights(Ns[li], K, 600 + 10 * gi + 1 + li)
            ref, _ = oracle.ternary_matmul(xq, s, oracle.pack_i2s(w)[0], ws, nthreads=NT)
            assert np.array_equal(host(out).view(np.uint32), ref[0].view(np.uint32))
    plan.close()
    assert binding.last_device_error() == 0


def test_sweep_plan_full_decode_step_against_oracle():
    """The whole 30-layer 2B-4T decode step (120 groups, 521 MB of packed weights) as one
    persistent plan, every output against oracle.quant_act + oracle.ternary_matmul on the
    step's own seeded inputs (the headline workload)."""
    mats = {n: (N, K) for n, N, K in workloads.LAYER_MATRICES}
    groups, refs = [], []
    for spec in workloads.decode_sweep_specs():
        for gname, names, K in workloads.LAYER_GROUPS:
            x_np = workloads.activations_f32(1, K, spec.act_seeds[gname])
            xq, s, _ = oracle.quant_act(x_np)
            projs = []
            for n in names:
                N = mats[n][0]
                w = workloads.ternary_weights(N, K, spec.weight_seeds[n])
                ws = workloads.weight_scale(N, K, spec.scale_seeds[n])
                out = torch.full((N,), float("nan"), dtype=torch.float32, device="cuda")
                projs.append((binding.pack_i2s(dev(w)), ws, out))
                refs.append(oracle.ternary_matmul(xq, s, oracle.pack_i2s(w)[0], ws, nthreads=NT)[0][0])
            groups.append((dev(x_np).view(-1), projs))
    plan = binding.SweepPlan(groups)
    plan.run()
    torch.cuda.synchronize()
    outs = [p[2] for _, projs in groups for p in projs]
    assert len(outs) == len(refs) == 30 * 7
    for got, ref in zip(outs, refs):
        assert np.array_equal(host(got).view(np.uint32), ref.view(np.uint32))
    plan.close()
    assert binding.last_device_error() == 0


# ----------------------------------------------------------------------------- few token rows

ROWS_CASES = [
    # (M, N, K) through auto dispatch: both sides of the GEMV / few-token crossover (4-5 rows up
    # to K = 10240, 2-3 rows beyond), the 2B-4T shapes, a ragged 32-lane layout (K 6912), the
    # 2-lane layout (K 384), the largest K of the GEMV's staged path, and fewer rows than SMs
    (2, 6912, 2560), (3, 2560, 6912), (4, 640, 2560), (5, 7, 384), (5, 2560, 6912), (8, 2560, 6912),
    (9, 2560, 6912), (11, 6912, 2560), (12, 6912, 2560), (16, 2560, 6912), (16, 300, 10240),
    (13, 1000, 1152), (2, 152, 128), (16, 1, 256), (2, 300, 12288), (3, 300, 12288),
    # two weight rows per lane (walks of 4-5 chunks): both lane layouts, ragged N (a lane's second
    # row past the end), and a ragged 5-chunk walk (K 9216)
    (2, 2560, 6912), (4, 6912, 2560), (4, 1001, 6912), (3, 999, 2560), (2, 300, 10240), (4, 300, 9216),
]


@pytest.mark.parametrize("M,N,K", ROWS_CASES)
def test_few_rows_parity(M, N, K):
    """A few token rows through auto dispatch (dp4a GEMV or the few-token tensor-core kernel):
    int32 accumulators and fp32 outputs bit for bit, on random packed bytes (code 3 included)
    and full-range int8 rows."""
    wp_np = workloads.random_packed_bytes(N, K, 900 + M + N)
    xq_np = workloads.random_int8(M, K, 901 + K)
    s_np = (np.random.default_rng(902).uniform(0.5, 60.0, M)).astype(np.float32)
    rs_np = xq_np.astype(np.int64).sum(axis=1).astype(np.int32)
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = binding.i2s_matmul(dev(xq_np), dev(s_np), dev(rs_np), dev(wp_np), 0.0173, acc_out=acc)
    torch.cuda.synchronize()
    o_out, o_acc = oracle.ternary_matmul(xq_np, s_np, wp_np, 0.0173, nthreads=NT)
    assert np.array_equal(host(acc), o_acc)
    assert np.array_equal(host(out).view(np.uint32), o_out.view(np.uint32))
    assert binding.last_device_error() == 0


# ----------------------------------------------------------------------------- seeded random cases

def _rand_k(rng, hi=10240):
    return int(rng.integers(1, hi // 128 + 1)) * 128


@pytest.mark.parametrize("case", range(24))
def test_random_matmul_shapes(case):
    """Seeded random (M, N, K) through auto dispatch, every kernel the dispatcher can pick, with
    random packed bytes (code 3 included) and full-range int8 rows: bit for bit."""
    rng = np.random.default_rng(7000 + case)
    M = int(rng.choice([1, 2, 3, 5, 8, 9, 12, 15, 17, 31, 48, 64, 65, 100, 129, 200]))
    N = int(rng.integers(1, 3000))
    K = _rand_k(rng, 6912 if M > 64 else 10240)
    wp_np = workloads.random_packed_bytes(N, K, 7100 + case)
    xq_np = workloads.random_int8(M, K, 7200 + case)
    s_np = rng.uniform(0.1, 100.0, M).astype(np.float32)
    rs_np = xq_np.astype(np.int64).sum(axis=1).astype(np.int32)
    ws = float(rng.uniform(0.001, 0.1))
    acc = torch.empty((M, N), dtype=torch.int32, device="cuda")
    out = binding.i2s_matmul(dev(xq_np), dev(s_np), dev(rs_np), dev(wp_np), ws, acc_out=acc)
    torch.cuda.synchronize()
    o_out, o_acc = oracle.ternary_matmul(xq_np, s_np, wp_np, ws, nthreads=NT)
    assert np.array_equal(host(acc), o_acc), (M, N, K)
    assert np.array_equal(host(out).view(np.uint32), o_out.view(np.uint32)), (M, N, K)
    assert binding.last_device_error() == 0


@pytest.mark.parametrize("case", range(6))
def test_random_sweep_plans(case):
    """Seeded random sweep plans (group count, K, projections and rows per group, dtype)."""
    rng = np.random.default_rng(7300 + case)
    dtype = "bf16" if case % 2 else "f32"
    groups, refs = [], []
    for gi in range(int(rng.integers(1, 12))):
        K = _rand_k(rng)
        x_np = workloads.activations(1, K, 7400 + 10 * case + gi, dtype, outlier_p=0.01)
        xq, s, _ = oracle.quant_act(x_np, dtype)
        projs = []
        for li in range(int(rng.integers(1, 9))):
            N = int(rng.integers(1, 1500))
            wp_np = workloads.random_packed_bytes(N, K, 7500 + 100 * case + 10 * gi + li)
            ws = float(rng.uniform(0.001, 0.1))
            projs.append((dev(wp_np), ws, torch.empty(N, dtype=torch.float32, device="cuda")))
            refs.append(oracle.ternary_matmul(xq, s, wp_np, ws, nthreads=NT)[0][0])
        groups.append((x_device(x_np, dtype).view(-1), projs))
    plan = binding.SweepPlan(groups)
    plan.run()
    torch.cuda.synchronize()
    outs = [p[2] for _, projs in groups for p in projs]
    plan.close()
    for got, ref in zip(outs, refs):
        assert np.array_equal(host(got).view(np.uint32), ref.view(np.uint32))
    assert binding.last_device_error() == 0


@pytest.mark.parametrize("case", range(6))
def test_random_ffn_blocks(case):
    """Seeded random FFN blocks (M, K, F, dtype, workspace) against the oracle chain."""
    rng = np.random.default_rng(7600 + case)
    M = int(rng.choice([1, 1, 2, 7, 20, 70]))
    K = _rand_k(rng, 4096)
    F = _rand_k(rng, 8192)
    dtype = "bf16" if case % 2 else "f32"
    x_np = workloads.activations(M, K, 7700 + case, dtype)
    wg, wu = workloads.ternary_weights(F, K, 7710 + case), workloads.ternary_weights(F, K, 7720 + case)
    wd = workloads.ternary_weights(K, F, 7730 + case)
    ag, au, ad = (float(v) for v in rng.uniform(0.005, 0.05, 3))
    gamma = workloads.rmsnorm_gamma(F, 7740 + case)
    use_ws = M > 64 and bool(case % 3)
    got = _run_ffn(x_np, dtype, wg, ag, wu, au, wd, ad, gamma, 1e-5, use_ws)
    check_ffn_block(x_np, dtype, wg, ag, wu, au, wd, ad, gamma, 1e-5, *got)
    assert binding.last_device_error() == 0


@pytest.mark.parametrize("case", range(6))
def test_random_weight_ternarisation(case):
    """Seeded random (N, K, dtype, mode, spread) for bitnet_quant_weight."""
    rng = np.random.default_rng(7800 + case)
    N, K = int(rng.integers(1, 700)), _rand_k(rng)
    dtype, mode = ("bf16" if case % 2 else "f32"), ("sign" if case % 3 == 2 else "absmean")
    w = (workloads.near_ternary_weights_f32(N, K, 7900 + case) if mode == "sign"
         else workloads.source_weights_f32(N, K, 7900 + case, std=float(rng.uniform(0.001, 3.0))))
    w_dev = w if dtype == "f32" else workloads.to_bf16_bits(w)
    g_wp, g_s = binding.quant_weight(x_device(w_dev, dtype), mode=mode)
    torch.cuda.synchronize()
    o_q, o_s = oracle.quant_weight(w_dev, dtype=dtype, mode=mode)
    assert np.array_equal(host(g_s).view(np.uint32), np.array([o_s], dtype=np.float32).view(np.uint32))
    assert np.array_equal(host(g_wp), oracle.pack_i2s(o_q)[0])
    assert binding.last_device_error() == 0
