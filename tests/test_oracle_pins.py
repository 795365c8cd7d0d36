"""Pins of the CPU oracle against what the pages print and what the mathematics fixes.

These run without a GPU. Each test pins one part of the oracle to something other than
the oracle itself: a value printed on a page (tests/golden/, cited there), a library
routine (numpy integer matmul, numpy/torch rounding and bf16 conversion), a closed form,
an invariant, or brute force on tiny inputs. A plausible mistake in the oracle -- a
reversed bit order, a linear instead of 4x32 interleave, a dropped -1, a wrong scale
direction, round-half-away instead of round-half-even -- fails at least one of them.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from conftest import read_golden
from ternary_weight_gb300 import workloads

QK = 128


def _xq(M, K, seed):
    return np.random.default_rng(seed).integers(-127, 128, size=(M, K), dtype=np.int16).astype(np.int8)


# ---------------------------------------------------------------- packing layout

def test_code_map_golden():
    g = read_golden("code_map.txt")
    for v, c in zip(g["value"], g["code"]):
        wp, bad = oracle.pack_i2s(np.full((1, QK), v, dtype=np.int8))
        assert bad == 0
        # every 2-bit field of every byte holds the code
        assert np.all(wp == c * 0b01010101), (v, c, wp[0, :4])
        assert np.all(oracle.unpack_i2s(wp, QK) == v)


def test_byte_example_unpack():
    g = read_golden("byte_example.txt")
    wp = np.full((1, QK // 4), 0x55, dtype=np.uint8)  # every other field: code 1 -> weight 0
    wp[0, 0] = g["packed"][0]
    w = oracle.unpack_i2s(wp, QK)[0]
    assert list(w[g["positions"]]) == g["weights"]
    rest = np.ones(QK, bool)
    rest[g["positions"]] = False
    assert np.all(w[rest] == 0)


@pytest.mark.parametrize("block", [0, 1, 2])
@pytest.mark.parametrize("row", [0, 1])
def test_byte_example_pack(block, row):
    """The byte example, placed in block `block` of row `row`. Every other weight is +1,
    so a linear (4 adjacent weights per byte) layout or a reversed bit order would not
    give the printed byte."""
    g = read_golden("byte_example.txt")
    K, N = 3 * QK, 2
    w = np.ones((N, K), dtype=np.int8)
    for pos, val in zip(g["positions"], g["weights"]):
        w[row, block * QK + pos] = val
    wp, bad = oracle.pack_i2s(w)
    assert bad == 0
    assert wp[row, block * 32] == g["packed"][0]
    other = np.ones_like(wp, dtype=bool)
    other[row, block * 32] = False
    assert np.all(wp[other] == 0xAA)  # all codes 2 (weight +1)


def test_pack_unpack_roundtrip():
    w = workloads.ternary_weights(13, 5 * QK, seed=7)
    wp, bad = oracle.pack_i2s(w)
    assert bad == 0 and wp.shape == (13, 5 * QK // 4)
    assert np.array_equal(oracle.unpack_i2s(wp, 5 * QK), w)


def test_pack_non_ternary_sign_rule():
    w = np.zeros((1, QK), dtype=np.int8)
    w[0, :6] = [5, -7, 127, -128, 1, -1]
    wp, bad = oracle.pack_i2s(w)
    assert bad == 4
    back = oracle.unpack_i2s(wp, QK)[0]
    assert list(back[:6]) == [1, -1, 1, -1, 1, -1]


def test_code3_reads_as_plus_two():
    wp = np.full((1, QK // 4), 0xFF, dtype=np.uint8)
    assert np.all(oracle.unpack_i2s(wp, QK) == 2)


def test_rejects_ragged_k():
    with pytest.raises(ValueError):
        oracle.pack_i2s(np.zeros((1, 100), dtype=np.int8))


# ---------------------------------------------------------------- ternary dot

@pytest.mark.parametrize("positions", [[0, 1, 2, 3], [3, 45, 90, 127], [31, 32, 63, 64]])
def test_worked_example(positions):
    g = read_golden("worked_example.txt")
    xq = np.zeros((1, QK), dtype=np.int8)
    w = np.zeros((1, QK), dtype=np.int8)
    xq[0, positions] = g["x"]
    w[0, positions] = g["w"]
    wp, _ = oracle.pack_i2s(w)
    _, acc = oracle.ternary_matmul(xq, np.ones(1, np.float32), wp, 1.0)
    assert acc[0, 0] == g["dot"][0]
    # the raw code dot multiplies the stored codes: 2*4 + 1*7 + 0*2 + 2*5 = 25 (padding
    # weights are 0 -> code 1, paired with activations 0), and 25 - sum(x) = 25 - 18 = 7
    raw = oracle.raw_code_dot(xq, wp)
    assert raw[0, 0] == 25
    assert raw[0, 0] - int(xq.astype(np.int64).sum()) == g["dot"][0]


@pytest.mark.parametrize("M,N,K,seed", [(1, 1, 128, 1), (3, 5, 256, 2), (4, 8, 384, 3), (2, 7, 128, 4)])
def test_brute_force_against_integer_matmul(M, N, K, seed):
    """Oracle (pack -> unpack -> dot) vs numpy's int64 matmul of the never-packed weights."""
    w = workloads.ternary_weights(N, K, seed)
    xq = _xq(M, K, seed + 100)
    wp, _ = oracle.pack_i2s(w)
    _, acc = oracle.ternary_matmul(xq, np.ones(M, np.float32), wp, 1.0)
    ref = xq.astype(np.int64) @ w.astype(np.int64).T
    assert np.array_equal(acc.astype(np.int64), ref)


def test_one_hot_rows_select_each_activation():
    """Row k of the weight matrix is +e_k, row K+k is -e_k: acc must be +-xq[:, k]."""
    K = 2 * QK
    w = np.concatenate([np.eye(K, dtype=np.int8), -np.eye(K, dtype=np.int8)])
    xq = _xq(3, K, 11)
    wp, _ = oracle.pack_i2s(w)
    _, acc = oracle.ternary_matmul(xq, np.ones(3, np.float32), wp, 1.0)
    assert np.array_equal(acc[:, :K], xq.astype(np.int32))
    assert np.array_equal(acc[:, K:], -xq.astype(np.int32))


def test_constant_weight_rows():
    K = 3 * QK
    xq = _xq(4, K, 12)
    w = np.stack([np.ones(K, np.int8), -np.ones(K, np.int8), np.zeros(K, np.int8)])
    wp, _ = oracle.pack_i2s(w)
    _, acc = oracle.ternary_matmul(xq, np.ones(4, np.float32), wp, 1.0)
    sy = xq.astype(np.int64).sum(axis=1)
    assert np.array_equal(acc[:, 0], sy) and np.array_equal(acc[:, 1], -sy)
    assert np.all(acc[:, 2] == 0)


def test_max_magnitude_accumulator():
    K = 64 * QK  # 8192
    xq = np.full((2, K), 127, dtype=np.int8)
    xq[1] = -127
    w = np.ones((1, K), dtype=np.int8)
    wp, _ = oracle.pack_i2s(w)
    _, acc = oracle.ternary_matmul(xq, np.ones(2, np.float32), wp, 1.0)
    assert acc[0, 0] == 127 * K and acc[1, 0] == -127 * K


@pytest.mark.parametrize("random_bytes", [False, True])
def test_raw_code_identity(random_bytes):
    """sum(code * y) - sum(y) == sum((code - 1) * y): the correction is an identity, for
    ternary codes and (random_bytes) for every 2-bit field, code 3 included."""
    M, N, K = 4, 16, 3 * QK
    xq = _xq(M, K, 13)
    if random_bytes:
        wp = np.random.default_rng(14).integers(0, 256, size=(N, K // 4), dtype=np.uint8)
    else:
        wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, 14))
    raw = oracle.raw_code_dot(xq, wp)
    _, acc = oracle.ternary_matmul(xq, np.ones(M, np.float32), wp, 1.0)
    sy = xq.astype(np.int64).sum(axis=1, keepdims=True)
    assert np.array_equal(raw.astype(np.int64) - sy, acc.astype(np.int64))
    if random_bytes:
        ref = xq.astype(np.int64) @ oracle.unpack_i2s(wp, K).astype(np.int64).T
        assert np.array_equal(acc.astype(np.int64), ref)


def test_threaded_equals_single_thread():
    M, N, K = 3, 37, 2 * QK
    xq = _xq(M, K, 15)
    s = np.array([1.5, 2.0, 0.25], np.float32)
    wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, 16))
    o1, a1 = oracle.ternary_matmul(xq, s, wp, 0.0159, nthreads=1)
    o4, a4 = oracle.ternary_matmul(xq, s, wp, 0.0159, nthreads=4)
    assert np.array_equal(a1, a4) and np.array_equal(o1.view(np.uint32), o4.view(np.uint32))


# ---------------------------------------------------------------- activation quantisation

def test_quant_unit_scale_rounds_half_to_even():
    """amax = 127 makes s = 127/127 = 1 exactly, so q must be numpy's rint (half to even)."""
    K = QK
    x = np.zeros((1, K), np.float32)
    vals = [127.0, 2.5, 3.5, -2.5, -3.5, 0.5, 1.5, -0.5, -1.5, 126.5, -126.5, 0.49999997, 10.0]
    x[0, : len(vals)] = vals
    xq, s, rowsum = oracle.quant_act(x)
    assert s[0] == np.float32(1.0)
    ref = np.rint(x[0].astype(np.float64)).astype(np.int64)
    assert np.array_equal(xq[0].astype(np.int64), ref)
    assert list(xq[0, 1:5]) == [2, 4, -2, -4]  # half-away-from-zero would give 3, 4, -3, -4
    assert rowsum[0] == ref.sum()


@pytest.mark.parametrize("amax,scale", [(254.0, 0.5), (63.5, 2.0), (508.0, 0.25)])
def test_quant_power_of_two_scale(amax, scale):
    """127/amax is a power of two here, so x*s is exact and q = rint(x*s)."""
    rng = np.random.default_rng(17)
    K = 2 * QK
    x = (rng.integers(-4 * int(amax), 4 * int(amax) + 1, size=(1, K)) / 4.0).astype(np.float32)
    x = np.clip(x, -amax, amax)
    x[0, 5] = amax
    xq, s, _ = oracle.quant_act(x)
    assert s[0] == np.float32(scale)
    ref = np.rint(x[0].astype(np.float64) * scale)
    assert np.array_equal(xq[0].astype(np.float64), ref)


def test_quant_zero_and_tiny_rows():
    K = QK
    x = np.zeros((2, K), np.float32)
    x[1, 3] = 2e-6   # below the 1e-5 floor
    x[1, 4] = -5e-6
    xq, s, rowsum = oracle.quant_act(x)
    assert np.all(xq[0] == 0) and rowsum[0] == 0
    # the floor: s = 127 / 1e-5 for both rows (within one ulp of the real quotient)
    for r in range(2):
        assert s[r] == s[0]
        assert abs(float(s[r]) * 1e-5 - 127.0) <= 127.0 * 2.0 ** -23
    assert xq[1, 3] == round(2e-6 * float(s[1])) and xq[1, 4] == round(-5e-6 * float(s[1]))


@pytest.mark.parametrize("outlier_p", [0.0, 0.01])
def test_quant_invariants(outlier_p):
    M, K = 16, 20 * QK
    x = workloads.activations_f32(M, K, seed=18, outlier_p=outlier_p)
    xq, s, rowsum = oracle.quant_act(x)
    q = xq.astype(np.int64)
    assert np.all(np.abs(q) <= 127)                      # -128 never occurs
    assert np.array_equal(q.sum(axis=1), rowsum.astype(np.int64))
    amax = np.abs(x).max(axis=1).astype(np.float64)
    arg = np.abs(x).argmax(axis=1)
    for m in range(M):
        # the largest-magnitude element maps to +-127
        assert q[m, arg[m]] == 127 * np.sign(x[m, arg[m]])
        # s is the inverse of bitnet.rs's alpha_x = amax / 127, to fp32 accuracy
        assert abs(float(s[m]) * amax[m] / 127.0 - 1.0) <= 2.0 ** -23
        # rounding error of the product: at most half a unit plus one fp32 rounding
        err = np.abs(q[m] - x[m].astype(np.float64) * float(s[m]))
        assert err.max() <= 0.5 + 127.0 * 2.0 ** -24
        # monotone in x
        order = np.argsort(x[m], kind="stable")
        assert np.all(np.diff(q[m][order]) >= 0)


def test_bf16_widening_matches_torch_for_every_pattern():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).float().numpy()
    finite = np.isfinite(ref)
    sample = np.flatnonzero(finite)[:: 97]
    for b in sample:
        assert np.float32(oracle.bf16_to_f32(int(bits[b]))).view(np.uint32) == ref[b].view(np.uint32)
    # whole-matrix path: quantising bf16 rows == quantising their exact fp32 widening
    rows = bits[finite].reshape(-1)[: 510 * QK].reshape(510, QK)
    rows_f32 = torch.from_numpy(rows.view(np.int16)).view(torch.bfloat16).float().numpy()
    a = oracle.quant_act(rows, "bf16")
    b = oracle.quant_act(rows_f32, "f32")
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ---------------------------------------------------------------- dequantisation

def test_dequant_unit_scales_is_the_integer():
    K, N = 2 * QK, 9
    x = workloads.activations_f32(2, K, seed=19)
    x[:, 0] = 127.0  # amax = 127 -> s = 1
    xq, s, _ = oracle.quant_act(x)
    assert np.all(s == 1.0)
    wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, 20))
    out, acc = oracle.ternary_matmul(xq, s, wp, 1.0)
    assert np.array_equal(out, acc.astype(np.float32))


def test_dequant_matches_absmax_form():
    """out = acc * alpha_W * alpha_x with alpha_x = amax/127 ("bitnet.rs", "Quantised Forward
    Pass", with its trailing /127 read as the one already inside alpha_x), to a few fp32
    roundings."""
    M, N, K = 5, 33, 4 * QK
    x = workloads.activations_f32(M, K, seed=21, outlier_p=0.01)
    w_scale = workloads.weight_scale(N, K, 22)
    xq, s, _ = oracle.quant_act(x)
    wp, _ = oracle.pack_i2s(workloads.ternary_weights(N, K, 23))
    out, acc = oracle.ternary_matmul(xq, s, wp, w_scale)
    amax = np.abs(x).max(axis=1).astype(np.float64)
    ref = acc.astype(np.float64) * float(np.float32(w_scale)) * (amax / 127.0)[:, None]
    nz = acc != 0
    rel = np.abs(out[nz].astype(np.float64) - ref[nz]) / np.abs(ref[nz])
    assert rel.max() <= 4 * 2.0 ** -24
    assert np.all(out[~nz] == 0.0)


def test_dequant_power_of_two_exact():
    K, N = QK, 4
    x = np.zeros((1, K), np.float32)
    x[0, :4] = [254.0, 100.0, -36.0, 8.0]   # amax = 254 -> s = 0.5
    xq, s, _ = oracle.quant_act(x)
    w = np.zeros((N, K), np.int8)
    w[0, :4] = [1, 1, 0, 0]
    w[1, :4] = [0, -1, 1, 1]
    wp, _ = oracle.pack_i2s(w)
    out, acc = oracle.ternary_matmul(xq, s, wp, 0.25)
    assert list(acc[0]) == [127 + 50, -50 - 18 + 4, 0, 0]
    assert np.array_equal(out[0], acc[0].astype(np.float32) * 2.0 * 0.25)


def test_quant_uses_multiply_form_of_scale():
    """Reading of the two printed scale forms: "BitNet 딥다이브" §4-5 multiplies by
    s = 127 / max|x|, "bitnet.rs" divides by alpha_x = max|x| / 127. They differ in the last
    fp32 ulp, which decides the integer next to a rounding tie. Near-tie inputs are built
    here for one row, and q must follow the multiply form (numpy fp32 multiply + rint)."""
    amax = np.array([1090775969], dtype=np.uint32).view(np.float32)[0]   # 8.245027
    s = np.float32(np.float32(127.0) / amax)
    alpha = np.float32(amax / np.float32(127.0))
    xs, expect, n_differ = [amax], [127.0], 0
    for k in range(1, 120):
        x0 = np.float32((k + 0.5) / float(s))
        for step in range(-3, 4):
            x = x0
            for _ in range(abs(step)):
                x = np.nextafter(x, np.float32(np.sign(step) * np.inf), dtype=np.float32)
            q_mul = np.rint(np.float32(x * s))
            if np.rint(np.float32(x / alpha)) != q_mul:
                n_differ += 1
            xs.append(x)
            expect.append(q_mul)
    assert n_differ >= 10      # the case really separates the two forms
    K = ((len(xs) + QK - 1) // QK) * QK
    row = np.zeros((1, K), np.float32)
    row[0, : len(xs)] = xs
    xq, s_or, _ = oracle.quant_act(row)
    assert s_or[0] == s
    assert np.array_equal(xq[0, : len(xs)].astype(np.float64), np.array(expect))


# ----------------------------------------------------------------------------- weight ternarisation

def test_absmean_page_example():
    """[DeepDive] §6-2: mean|w| = 0.4 and w / 0.4 = [-1.5, -0.5, 0.5, 1.5] as printed; with
    round-half-to-even (numpy's round, the reading taken) the codes are [-1, 0, 0, 1], where
    rounding half away from zero would give [-1, -1, 1, 1]."""
    g = read_golden("absmean_example.txt")
    w = np.array([g["w"]], dtype=np.float32)
    q, scale = oracle.quant_weight(w)
    assert scale == np.float32(g["mean"][0])
    assert np.array_equal(w / np.float32(scale), np.array([g["ratio"]], dtype=np.float32))
    assert q.tolist() == [[-1, 0, 0, 1]]


def test_absmean_rounding_ties_go_to_even():
    # mean|w| = 1 exactly, so w / scale is w: +-0.5 round to 0, +-1.5 to +-2 (clipped to +-1)
    w = np.array([[0.5, -0.5, 1.5, -1.5], [1.0, -1.0, 0.5, 1.5]], dtype=np.float32)
    q, scale = oracle.quant_weight(w)
    assert scale == 1.0
    assert q.tolist() == [[0, 0, 1, -1], [1, -1, 0, 1]]


def test_absmean_all_zero_uses_the_floor():
    q, scale = oracle.quant_weight(np.zeros((3, 256), dtype=np.float32))
    assert scale == np.float32(1e-5) and not q.any()


@pytest.mark.parametrize("c", [0.25, -3.0, 2.0 ** -10, -0.015625])
def test_absmean_constant_matrix(c):
    # N*K = 2^10 copies of |c| sum exactly in fp64, so the mean is |c| and every code is sign(c)
    w = np.full((8, 128), c, dtype=np.float32)
    q, scale = oracle.quant_weight(w)
    assert scale == np.float32(abs(c))
    assert np.all(q == np.sign(c))


@pytest.mark.parametrize("N,K,seed", [(7, 384, 0), (64, 2560, 1), (33, 1000, 2)])
def test_absmean_scale_is_the_correctly_rounded_mean(N, K, seed):
    """The scale is the exact mean rounded to fp32 (checked with an exact rational sum), and it
    is the integer-sum definition recomputed with Python integers:
    S = sum floor(|w| 2^74), mean = fp32(fp64(S) 2^-74 / (N K))."""
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((N, K)) * 0.02).astype(np.float32)
    q, scale = oracle.quant_weight(w)
    absw = [Fraction(float(v)) for v in np.abs(w).ravel()]
    exact = sum(absw) / (N * K)
    assert scale == np.float32(float(exact))
    S = sum(int(a * 2 ** 74) for a in absw)  # int() of a positive Fraction floors
    assert scale == np.float32(float(S) * 2.0 ** -74 / (N * K))
    # and the codes are numpy's round-half-to-even of the fp32 quotient, clipped
    ref = np.clip(np.round(w / np.float32(scale)), -1, 1).astype(np.int8)
    assert np.array_equal(q, ref)


def test_absmean_rejects_weights_outside_the_exact_sum_range():
    w = np.zeros((1, 128), dtype=np.float32)
    w[0, 5] = 4096.0
    with pytest.raises(RuntimeError):
        oracle.quant_weight(w)
    w[0, 5] = np.nextafter(np.float32(4096.0), np.float32(0))  # largest allowed magnitude
    q, scale = oracle.quant_weight(w)
    assert scale == np.float32(float(w[0, 5]) / 128) and q[0, 5] == 1


def test_absmean_bf16_is_the_widened_fp32():
    rng = np.random.default_rng(5)
    wf = (rng.standard_normal((9, 256)) * 0.02).astype(np.float32)
    wb = workloads.to_bf16_bits(wf)
    widened = np.array([[oracle.bf16_to_f32(int(b)) for b in row] for row in wb], dtype=np.float32)
    qb, sb = oracle.quant_weight(wb, dtype="bf16")
    qf, sf = oracle.quant_weight(widened)
    assert sb == sf and np.array_equal(qb, qf)


def test_sign_rule_threshold_and_scale():
    """[DeepDive] §4-2: |w| < 1e-6 codes as 0 (the comparison in double, so 1e-6f itself is
    0), anything else by its sign; the scale kept is max|w|."""
    t = np.float32(1e-6)
    above = np.nextafter(t, np.float32(1), dtype=np.float32)
    w = np.array([[t, -t, above, -above, 0.0, -0.0, 5.0, -7.5]], dtype=np.float32)
    q, scale = oracle.quant_weight(w, mode="sign")
    assert q.tolist() == [[0, 0, 1, -1, 0, 0, 1, -1]]
    assert scale == np.float32(7.5)


# ---------------------------------------------------------------- FFN inner activation

def _ffn_rows(M, F, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((M, F)).astype(np.float32)
    u = rng.standard_normal((M, F)).astype(np.float32)
    gamma = (1.0 + 0.1 * rng.standard_normal(F)).astype(np.float32)
    return g, u, gamma


@pytest.mark.parametrize("eps", [0.0, 1e-5, 0.5])
def test_ffn_inner_matches_fp64_definition(eps):
    """[bitnet.rs] "Forward Pass": inner = RMSNorm(sqrelu(gate) * up), against the same
    formula in float64 (numpy). The oracle rounds h twice, the sum of squares once (it is
    summed in double), then ss / F, + eps, the root, the reciprocal and the two products once
    each: at most 8 * 2^-24 relative in all. A dropped or misplaced term (no square in sqrelu,
    no gamma, eps outside the root, sum instead of mean) is off by far more, and so is a sum
    of squares accumulated in fp32 over the 6912 terms."""
    M, F = 3, 6912
    g, u, gamma = _ffn_rows(M, F, 11)
    got = oracle.ffn_inner(g, u, gamma, eps)
    h = np.maximum(g.astype(np.float64), 0.0) ** 2 * u
    ref = h / np.sqrt(np.mean(h * h, axis=1, keepdims=True) + eps) * gamma
    np.testing.assert_allclose(got, ref, rtol=8 * 2.0 ** -24, atol=1e-30)


def test_ffn_inner_sqrelu_zeroes_non_positive_gates():
    """max(g, 0)^2: negative, -0 and NaN gates give a zero at their position (signed like
    u * gamma, since (0 * 0) * u keeps the sign of u); the rest of the row stays finite."""
    g, u, gamma = _ffn_rows(1, 1024, 12)
    g[0, :4] = [-3.0, -0.0, np.nan, -1e-30]
    inner = oracle.ffn_inner(g, u, gamma, 1e-5)
    assert np.all(inner[0, :4] == 0.0)
    assert np.array_equal(np.signbit(inner[0, :4]), np.signbit(u[0, :4] * gamma[:4]))
    assert np.all(np.isfinite(inner))


def test_ffn_inner_constant_row_normalises_to_gamma():
    """h constant = 12 (g = 2, u = 3): ss = 144 F exactly, mean 144, root 12, so inner is
    gamma * fl(12 * fl(1/12)), within one ulp of gamma; with gamma = 1 every element is ~1."""
    F = 2048
    g = np.full((1, F), 2.0, np.float32)
    u = np.full((1, F), 3.0, np.float32)
    gamma = np.linspace(0.5, 2.0, F).astype(np.float32)
    inner = oracle.ffn_inner(g, u, gamma, 0.0)[0]
    assert np.all(np.abs(inner - gamma) <= np.spacing(gamma) * 1.0)
    ones = oracle.ffn_inner(g, u, np.ones(F, np.float32), 0.0)[0]
    assert np.all(np.abs(ones - 1.0) <= 2.0 ** -23)


def test_ffn_inner_single_spike_is_sqrt_f():
    """One positive gate: h = (a, 0, ...), mean = a^2 / F, so with eps = 0 inner_0 = sqrt(F)
    (to a few ulps) and every other element is 0."""
    F = 4096
    g = np.full((1, F), -1.0, np.float32)
    u = np.ones((1, F), np.float32)
    g[0, 1234] = 1.75
    inner = oracle.ffn_inner(g, u, np.ones(F, np.float32), 0.0)[0]
    assert abs(inner[1234] - 64.0) <= 4 * np.spacing(np.float32(64.0))
    assert np.count_nonzero(inner) == 1


def test_ffn_inner_scale_invariance_exact():
    """With eps = 0 RMSNorm is invariant under scaling h by 2^k, and every fp32 step scales
    exactly, so inner is bit-identical: up * 2^k scales h by 2^k, gate * 2^k by 2^2k."""
    g, u, gamma = _ffn_rows(2, 2560, 13)
    base = oracle.ffn_inner(g, u, gamma, 0.0)
    for k in (-5, 3):
        assert np.array_equal(oracle.ffn_inner(g, u * np.float32(2.0 ** k), gamma, 0.0), base)
        assert np.array_equal(oracle.ffn_inner(g * np.float32(2.0 ** k), u, gamma, 0.0), base)


def test_ffn_inner_all_gates_negative_with_eps():
    """h = 0 everywhere: ss = 0, c = 1/sqrt(eps) finite, inner exactly 0 (no NaN)."""
    g = -np.abs(_ffn_rows(1, 640, 14)[0]) - 1.0
    u = np.ones_like(g)
    inner = oracle.ffn_inner(g, u, np.ones(640, np.float32), 1e-5)
    assert np.all(inner == 0.0)


def test_ffn_inner_rows_are_independent():
    """Each row is normalised by its own sum: a row computed alone equals it in a batch."""
    g, u, gamma = _ffn_rows(4, 1024, 15)
    batch = oracle.ffn_inner(g, u, gamma, 1e-5)
    for m in range(4):
        assert np.array_equal(oracle.ffn_inner(g[m:m + 1], u[m:m + 1], gamma, 1e-5)[0], batch[m])
