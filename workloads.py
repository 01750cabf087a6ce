"""Seeded synthetic workloads for the attention forward pass.

This module holds only shapes, seeds and random-number draws: none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the oracle's
checks take their inputs from here, so the two sides always see the same
16-bit tensors.

Recipe: Q, K, V are drawn in that order from one ``torch.Generator`` seeded
with ``1000 + config_index`` as float32 standard normals of shape [B,H,N,d],
then rounded to nearest-even into the workload's 16-bit type.  The
"peaky" workload multiplies Q and K by 2 after rounding (exact in bf16/fp16).
Row samples for large workloads come from a second generator seeded with
``2000 + config_index``.
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int            # 1-based position in the workload list
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "fp16" or "bf16"
    causal: bool
    qk_mult: float = 1.0  # Q and K multiplied by this after rounding
    splitkv: bool = False  # run through the split-KV entry point (automatic count)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.float16 if self.dtype == "fp16" else torch.bfloat16

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs of the metric: 4*B*H*N^2*d, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V; write O (16-bit) and LSE (fp32)."""
        bh_n = self.B * self.H * self.N
        return 4 * bh_n * self.d * 2 + bh_n * 4

    def describe(self) -> str:
        mask = "causal" if self.causal else "full"
        extra = f", Q,K x{self.qk_mult:g}" if self.qk_mult != 1.0 else ""
        extra += ", split-KV" if self.splitkv else ""
        return (f"B={self.B} H={self.H} N={self.N} d={self.d} {self.dtype} "
                f"{mask}{extra}")


WORKLOADS = [
    Workload(1, "tiny_fp16_d64", 1, 2, 256, 64, "fp16", False),
    Workload(2, "bf16_d128_n2048", 4, 16, 2048, 128, "bf16", False),
    Workload(3, "bf16_d128_n8192_causal", 2, 16, 8192, 128, "bf16", True),
    Workload(4, "bf16_d256_n4096_peaky", 4, 8, 4096, 256, "bf16", False, 2.0),
    Workload(5, "bf16_d128_n32768_causal", 1, 32, 32768, 128, "bf16", True),
    # one long causal sequence with a single head: 128 query-tile pairs
    # cannot fill the SMs on their own (the split-KV case)
    Workload(6, "bf16_d128_n32768_h1_causal_splitkv", 1, 1, 32768, 128, "bf16", True,
             splitkv=True),
]


def workload(index: int) -> Workload:
    return WORKLOADS[index - 1]


def make_qkv(wl: Workload, seed: int | None = None):
    """CPU tensors q, k, v in the workload's dtype, drawn as the recipe says."""
    g = torch.Generator().manual_seed(1000 + wl.index if seed is None else seed)
    shape = (wl.B, wl.H, wl.N, wl.d)
    out = []
    for _ in range(3):
        out.append(torch.randn(shape, generator=g, dtype=torch.float32)
                   .to(wl.torch_dtype))
    q, k, v = out
    if wl.qk_mult != 1.0:
        q = q * wl.qk_mult
        k = k * wl.qk_mult
    return q, k, v


def make_random_qkv(B: int, H: int, N: int, d: int, dtype, seed: int,
                    qk_mult: float = 1.0):
    """Same recipe for an ad-hoc shape (parity and edge-case tests)."""
    wl = Workload(0, "adhoc", B, H, N, d,
                  "fp16" if dtype == torch.float16 else "bf16", False, qk_mult)
    return make_qkv(wl, seed=seed)


def sample_rows(wl: Workload, count: int = 512, seed: int | None = None):
    """Seeded (b, h, i) triples: ``count`` random ones plus fixed boundary rows.

    The fixed rows are 0, 1, 127, 128 and N-1 of head (0,0) and of the last
    head, and, for causal workloads, the first and last rows of every
    128-row query tile boundary up to 1024.
    """
    g = torch.Generator().manual_seed(2000 + wl.index if seed is None else seed)
    b = torch.randint(0, wl.B, (count,), generator=g)
    h = torch.randint(0, wl.H, (count,), generator=g)
    i = torch.randint(0, wl.N, (count,), generator=g)
    rows = set(zip(b.tolist(), h.tolist(), i.tolist()))
    fixed = {0, 1, 127, 128, wl.N - 1}
    if wl.causal:
        for t in range(128, min(wl.N, 1025), 128):
            fixed.update({t - 1, t})
    for (bb, hh) in ((0, 0), (wl.B - 1, wl.H - 1)):
        for r in fixed:
            if 0 <= r < wl.N:
                rows.add((bb, hh, r))
    return sorted(rows)
