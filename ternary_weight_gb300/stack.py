"""Resident ternary projections run as one CUDA graph.

A decode step of a BitNet b1.58 model applies, layer after layer, groups of ternary
projections that share one activation row (q/k/v on the attention input, o on the attention
output, gate/up on the FFN input, down on the FFN middle). ``TernaryStack`` keeps every
projection's i2_s packed weights resident in HBM and runs, per group, the activation
quantisation and one GEMV per projection -- all through the C ABI, by default as one fused
launch per group -- in a fixed order. The whole sequence is captured once into a CUDA graph, so a step is one graph
launch. Activations enter through one contiguous input buffer and results leave through
one contiguous output buffer, so a host round trip is one copy each way.

Everything the step computes runs in the library's kernels; torch only owns the buffers,
the stream and the graph.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Sequence

import torch

from . import binding


@dataclass
class PackedLinear:
    """One ternary projection: i2_s packed weights (N x K/4 uint8, resident) and alpha_W."""
    name: str
    wp: torch.Tensor
    w_scale: float
    N: int
    K: int

    @classmethod
    def from_ternary(cls, name: str, w_int8: torch.Tensor, w_scale: float, stream=None) -> "PackedLinear":
        N, K = w_int8.shape
        wp = binding.pack_i2s(w_int8, stream=stream)
        return cls(name, wp, float(w_scale), N, K)

    def weight_bytes(self) -> int:
        return self.N * self.K // 4


@dataclass
class Group:
    """Projections that consume the same activation row(s)."""
    name: str
    K: int
    linears: List[PackedLinear]


class TernaryStack:
    """Groups of ternary projections executed in order, as one CUDA graph per step."""

    def __init__(self, groups: Sequence[Group], M: int = 1, act_dtype=torch.float32, device="cuda",
                 algo: str = "auto", fused: bool = True, prefetch_next: bool = False):
        self.groups = list(groups)
        self.fused = fused
        self.prefetch_next = prefetch_next
        self.M = M
        self.act_dtype = act_dtype
        self.device = torch.device(device)
        self.algo = algo
        esz = torch.tensor([], dtype=act_dtype).element_size()
        # one contiguous input buffer (activations of every group, in order)
        self.in_elems = sum(M * g.K for g in self.groups)
        self.x_all = torch.zeros(self.in_elems, dtype=act_dtype, device=self.device)
        # one contiguous output buffer (every projection's M x N fp32 result, in order)
        self.out_elems = sum(M * l.N for g in self.groups for l in g.linears)
        self.out_all = torch.zeros(self.out_elems, dtype=torch.float32, device=self.device)
        self.x, self.xq, self.s, self.rs, self.out = [], [], [], [], []
        xo = oo = 0
        for g in self.groups:
            assert all(l.K == g.K for l in g.linears)
            self.x.append(self.x_all[xo:xo + M * g.K].view(M, g.K))
            xo += M * g.K
            self.xq.append(torch.empty((M, g.K), dtype=torch.int8, device=self.device))
            self.s.append(torch.empty(M, dtype=torch.float32, device=self.device))
            self.rs.append(torch.empty(M, dtype=torch.int32, device=self.device))
            outs = []
            for l in g.linears:
                outs.append(self.out_all[oo:oo + M * l.N].view(M, l.N))
                oo += M * l.N
            self.out.append(outs)
        self.act_bytes_in = self.in_elems * esz
        self.graph = None

    # ---- accounting ----
    def launches_per_step(self) -> int:
        if self.fused and self.M == 1:
            return len(self.groups)
        return sum(1 + len(g.linears) for g in self.groups)

    def gemv_launches_per_step(self) -> int:
        return sum(len(g.linears) for g in self.groups)

    def gemv_bytes_per_step(self) -> int:
        """Algorithmic bytes of the matmuls: packed weights (2 bits/weight), int8 activations,
        scale and row sum, fp32 outputs."""
        M = self.M
        return sum(l.weight_bytes() + M * l.K + 8 * M + 4 * M * l.N for g in self.groups for l in g.linears)

    def quant_bytes_per_step(self) -> int:
        esz = torch.tensor([], dtype=self.act_dtype).element_size()
        return sum(self.M * g.K * (esz + 1) + 8 * self.M for g in self.groups)

    def bytes_per_step(self) -> int:
        return self.gemv_bytes_per_step() + self.quant_bytes_per_step()

    # ---- execution ----
    def run(self, stream=None, gemv_only: bool = False):
        """Enqueue one step (quantise each group's row, then its GEMVs) on the stream.

        fused (default): one bitnet_w2a8_linear_group call per group -- quantisation and every
        projection of the group in a single kernel when M == 1 -- which also pulls the next
        group's packed weights into L2 while it runs (prefetch_next; the last group prefetches
        the first, for the next step). Otherwise (or with gemv_only, which leaves out the
        quantisation) one quantisation launch per group and one bitnet_i2s_matmul launch per
        projection."""
        for gi, g in enumerate(self.groups):
            if self.fused and not gemv_only:
                single = self.M == 1
                nxt = self.groups[(gi + 1) % len(self.groups)]
                binding.linear_group(self.x[gi], [l.wp for l in g.linears], [l.w_scale for l in g.linears],
                                     outs=self.out[gi], xq=None if single else self.xq[gi],
                                     scale=None if single else self.s[gi], rowsum=None if single else self.rs[gi],
                                     prefetch=[l.wp for l in nxt.linears] if self.prefetch_next else None,
                                     stream=stream)
                continue
            if not gemv_only:
                binding.quant_act(self.x[gi], self.xq[gi], self.s[gi], self.rs[gi], stream=stream)
            for li, l in enumerate(g.linears):
                binding.i2s_matmul(self.xq[gi], self.s[gi], self.rs[gi], l.wp, l.w_scale,
                                   out=self.out[gi][li], algo=self.algo, stream=stream)

    def capture(self, gemv_only: bool = False) -> torch.cuda.CUDAGraph:
        """Capture one step into a CUDA graph (after one eager run that warms everything up)."""
        s = torch.cuda.Stream(device=self.device)
        s.wait_stream(torch.cuda.current_stream(self.device))
        with torch.cuda.stream(s):
            self.run(stream=s, gemv_only=gemv_only)
        torch.cuda.current_stream(self.device).wait_stream(s)
        torch.cuda.synchronize(self.device)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            self.run(gemv_only=gemv_only)
        if not gemv_only:
            self.graph = g
        return g

    def step(self):
        """One graph launch of the captured step on the current stream."""
        if self.graph is None:
            self.capture()
        self.graph.replay()
