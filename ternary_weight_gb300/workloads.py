"""Seeded synthetic inputs and the workload shapes they are drawn for.

This module is the one piece shared by the CUDA path's tests/benchmark and the oracle:
it draws random inputs and holds none of the method's arithmetic (no packing, no
quantisation, no dot products). It imports nothing else from the package.

Shapes follow the BitNet b1.58 2B-4T layer (hidden 2560, FFN 6912, grouped-query
attention with 4 query heads per KV head -> k/v projections of 640 rows), as described in
"bitnet.rs -- BitNet b1.58 Inference Engine in Rust", "Forward Pass", and the 100B-class
GEMV shape K=8192, N=28672.

Recipe (all draws use numpy's PCG64 ``default_rng`` with the seed stated per tensor):
  * ternary weights: iid, P(-1) = 0.3, P(0) = 0.4, P(+1) = 0.3: a uniform 16-bit b gives
    u = floor(10 * b / 65536) in [0, 10) (each u has probability 0.1 to within 1e-4
    relative), then u < 3 -> -1, u < 7 -> 0, else +1;
  * weight scale alpha_W = mean|W_src| of a separately drawn N(0, 0.02) source (a sample
    of min(N*K, 2**20) elements stands for the full matrix; the expectation is
    0.02*sqrt(2/pi) ~= 0.01596);
  * activations: fp32 N(0, 1), or fp32 N(0, 1) rounded to bf16 (round-to-nearest-even),
    optionally with Bernoulli(p) outliers multiplied by 20 before the rounding;
  * FFN sub-norm weight gamma: fp32 1 + 0.1 N(0, 1), epsilon 1e-5;
  * full-precision weights for the ternarisation: fp32 N(0, 0.02^2); for the sign rule,
    ternary weights times 0.0156 with each zero replaced by a magnitude uniform in
    [0.5e-6, 2e-6] of random sign (so about a third of them fall below the 1e-6 threshold).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Tuple

import numpy as np

HIDDEN = 2560
FFN = 6912
KV = 640
N_LAYERS = 30

# The seven ternary projections of one 2B-4T decoder layer: name -> (N, K), grouped by
# the activation row they consume (q/k/v share the attention input, gate/up share the
# FFN input).
LAYER_MATRICES: List[Tuple[str, int, int]] = [
    ("q", HIDDEN, HIDDEN),
    ("k", KV, HIDDEN),
    ("v", KV, HIDDEN),
    ("o", HIDDEN, HIDDEN),
    ("gate", FFN, HIDDEN),
    ("up", FFN, HIDDEN),
    ("down", HIDDEN, FFN),
]
LAYER_GROUPS: List[Tuple[str, List[str], int]] = [
    ("attn_in", ["q", "k", "v"], HIDDEN),
    ("attn_out", ["o"], HIDDEN),
    ("ffn_in", ["gate", "up"], HIDDEN),
    ("ffn_mid", ["down"], FFN),
]

_TERNARY_OF_U = np.array([-1, -1, -1, 0, 0, 0, 0, 1, 1, 1], dtype=np.int8)
# the same map applied to every 16-bit draw b: u = floor(10 * b / 65536)
_TERNARY_OF_B16 = _TERNARY_OF_U[(np.arange(1 << 16, dtype=np.uint32) * 10) >> 16]


def ternary_weights(N: int, K: int, seed: int) -> np.ndarray:
    """N x K int8 ternary matrix, iid P(-1)=P(+1)=0.3, P(0)=0.4."""
    rng = np.random.default_rng(seed)
    b = rng.integers(0, 1 << 16, size=(N, K), dtype=np.uint16)
    return _TERNARY_OF_B16[b]


def weight_scale(N: int, K: int, seed: int) -> float:
    """alpha_W = mean|W_src| of a N(0, 0.02) source matrix (sampled, see module doc)."""
    rng = np.random.default_rng(seed)
    n = int(min(N * K, 1 << 20))
    src = rng.normal(0.0, 0.02, size=n)
    return float(np.float32(np.mean(np.abs(src))))


def source_weights_f32(N: int, K: int, seed: int, std: float = 0.02) -> np.ndarray:
    """N x K fp32 full-precision weights ~ N(0, std^2): the input of the weight ternarisation."""
    rng = np.random.default_rng(seed)
    return (rng.standard_normal(size=(N, K), dtype=np.float32) * np.float32(std)).astype(np.float32)


def near_ternary_weights_f32(N: int, K: int, seed: int, a: float = 0.0156) -> np.ndarray:
    """N x K fp32 weights that are already ternary up to noise, for the sign rule: values
    +-a, and zeros replaced by magnitudes spread across 1e-6 (half below, half above)."""
    rng = np.random.default_rng(seed)
    t = ternary_weights(N, K, seed).astype(np.float32) * np.float32(a)
    tiny = (rng.uniform(0.5e-6, 2e-6, size=(N, K)) * rng.choice([-1.0, 1.0], size=(N, K))).astype(np.float32)
    return np.where(t == 0, tiny, t).astype(np.float32)


def rmsnorm_gamma(F: int, seed: int) -> np.ndarray:
    """F fp32 per-channel weights of an RMSNorm (the FFN sub-norm): 1 + 0.1 N(0, 1)."""
    rng = np.random.default_rng(seed)
    return (1.0 + 0.1 * rng.standard_normal(F)).astype(np.float32)


FFN_EPS = 1e-5  # the sub-norm's epsilon in the FFN workloads (the pages print none)


def activations_f32(M: int, K: int, seed: int, outlier_p: float = 0.0) -> np.ndarray:
    """M x K fp32 N(0,1) rows, optional Bernoulli(outlier_p) x20 outliers."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal(size=(M, K), dtype=np.float32)
    if outlier_p > 0.0:
        hit = rng.random(size=(M, K)) < outlier_p
        x = np.where(hit, x * np.float32(20.0), x).astype(np.float32)
    return x


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """fp32 -> bf16 (round-to-nearest-even, via torch's CPU cast) as uint16 bit patterns."""
    import torch

    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16).copy()


def activations(M: int, K: int, seed: int, dtype: str, outlier_p: float = 0.0) -> np.ndarray:
    """fp32 array for dtype='f32', uint16 bf16 patterns for dtype='bf16'."""
    x = activations_f32(M, K, seed, outlier_p)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return to_bf16_bits(x)
    raise ValueError(dtype)


@dataclass(frozen=True)
class MatmulCase:
    """One matmul problem: activations M x K (dtype), ternary weights N x K."""
    name: str
    M: int
    N: int
    K: int
    act_dtype: str = "f32"
    outlier_p: float = 0.0
    seed: int = 0          # activations use seed, weights seed+1, weight scale seed+2

    def weights(self) -> np.ndarray:
        return ternary_weights(self.N, self.K, self.seed + 1)

    def w_scale(self) -> float:
        return weight_scale(self.N, self.K, self.seed + 2)

    def x(self) -> np.ndarray:
        return activations(self.M, self.K, self.seed, self.act_dtype, self.outlier_p)


def single_gemv() -> MatmulCase:
    """One W2A8 GEMV, M=1, K=N=2560, fp32 activations, seed 0."""
    return MatmulCase("gemv_2560x2560_m1", 1, HIDDEN, HIDDEN, "f32", 0.0, 0)


def batched_decode_cases() -> List[MatmulCase]:
    """Batched decode GEMVs M in {1,4,16,64} on the FFN shapes, bf16 with 1% x20 outliers."""
    out = []
    for i, M in enumerate((1, 4, 16, 64)):
        for j, (K, N) in enumerate(((HIDDEN, FFN), (FFN, HIDDEN))):
            out.append(MatmulCase("decode_m%d_k%d_n%d" % (M, K, N), M, N, K, "bf16", 0.01,
                                  3000 + 10 * (2 * i + j)))
    return out


def prefill_cases() -> List[MatmulCase]:
    """Prefill GEMMs M in {128,512} on the FFN shapes, bf16 N(0,1)."""
    out = []
    for i, M in enumerate((128, 512)):
        for j, (K, N) in enumerate(((HIDDEN, FFN), (FFN, HIDDEN))):
            out.append(MatmulCase("prefill_m%d_k%d_n%d" % (M, K, N), M, N, K, "bf16", 0.0,
                                  4000 + 10 * (2 * i + j)))
    return out


def large_cases() -> List[MatmulCase]:
    """Prefill M=4096 (K=6912, N=2560) and the 100B-class GEMV M=1 (K=8192, N=28672)."""
    return [
        MatmulCase("prefill_m4096_k6912_n2560", 4096, HIDDEN, FFN, "bf16", 0.0, 5000),
        MatmulCase("gemv_100b_k8192_n28672", 1, 28672, 8192, "bf16", 0.0, 5010),
    ]


@dataclass
class DecodeLayerSpec:
    """Seeds for one layer of the 30-layer decode sweep (fp32 activations, M=1)."""
    layer: int
    weight_seeds: dict = field(default_factory=dict)
    scale_seeds: dict = field(default_factory=dict)
    act_seeds: dict = field(default_factory=dict)


def decode_sweep_specs(n_layers: int = N_LAYERS) -> List[DecodeLayerSpec]:
    """Seed plan of the 2B-4T decode sweep: seed = 2000 + 100*layer + tensor index."""
    specs = []
    for l in range(n_layers):
        spec = DecodeLayerSpec(l)
        for t, (name, _, _) in enumerate(LAYER_MATRICES):
            spec.weight_seeds[name] = 2000 + 100 * l + t
            spec.scale_seeds[name] = 2000 + 100 * l + 20 + t
        for t, (gname, _, _) in enumerate(LAYER_GROUPS):
            spec.act_seeds[gname] = 2000 + 100 * l + 50 + t
        specs.append(spec)
    return specs


def decode_sweep_weight_bytes(n_layers: int = N_LAYERS) -> int:
    """Packed i2_s bytes of the sweep (2 bits per weight)."""
    return n_layers * sum(N * K // 4 for _, N, K in LAYER_MATRICES)


def random_packed_bytes(N: int, K: int, seed: int) -> np.ndarray:
    """N x K/4 uniformly random bytes: every 2-bit field, the unused code 3 included, with
    probability 1/4 each. Used for adversarial parity cases (the layout is irrelevant to it)."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, 256, size=(N, K // 4), dtype=np.uint8)


def random_int8(M: int, K: int, seed: int, lo: int = -127, hi: int = 127) -> np.ndarray:
    """M x K uniformly random int8 in [lo, hi]."""
    rng = np.random.default_rng(seed)
    return rng.integers(lo, hi + 1, size=(M, K), dtype=np.int16).astype(np.int8)
