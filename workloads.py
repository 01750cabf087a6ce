"""Seeded synthetic workloads for the attention forward pass.

This module holds only shapes, seeds and random-number draws: none of the
attention arithmetic.  Both the CUDA path's tests/benchmark and the oracle's
checks take their inputs from here, so the two sides always see the same
16-bit tensors.

Recipe: Q, K, V are drawn in that order from one ``torch.Generator`` seeded
with ``1000 + config_index`` as float32 standard normals of shape [B,H,N,d],
then rounded to nearest-even into the workload's 16-bit type (or to FP8
E4M3, saturating, for the fp8 workload).  The "peaky" workload multiplies Q
and K by 2 after rounding (exact in bf16/fp16).
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
    dtype: str            # "fp16", "bf16" or "fp8" (E4M3 inputs, bf16 output)
    causal: bool
    qk_mult: float = 1.0  # Q and K multiplied by this after rounding
    splitkv: bool = False  # run through the split-KV entry point (automatic count)
    varlen: bool = False   # B sequences of seeded lengths in [N/16, N], packed along rows
    # decode against a cache: B sequences of n_q query rows each, packed
    # [B*n_q, H, d], attending to N cached keys each (packed [B*N, H_kv, d]),
    # masks bottom-right aligned (fa_fwd_varlen_qk); 0 otherwise
    n_q: int = 0
    H_kv: int = 0

    def seqlens(self) -> list[int]:
        """Lengths of the packed sequences (varlen workloads): B integers drawn
        uniformly from [max(1, N/16), N] by a generator seeded with
        3000 + index."""
        if not self.varlen:
            return [self.N] * self.B
        g = torch.Generator().manual_seed(3000 + self.index)
        return torch.randint(max(1, self.N // 16), self.N + 1, (self.B,), generator=g).tolist()

    def cu_seqlens(self) -> list[int]:
        out = [0]
        for n in self.seqlens():
            out.append(out[-1] + n)
        return out

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return {"fp16": torch.float16, "bf16": torch.bfloat16,
                "fp8": torch.float8_e4m3fn}[self.dtype]

    @property
    def decode(self) -> bool:
        return self.n_q > 0

    @property
    def kv_heads(self) -> int:
        return self.H_kv if self.H_kv > 0 else self.H

    @property
    def flops(self) -> float:
        """Algorithmic FLOPs of the metric: 4*H*d*sum_b n_b^2 (4*B*H*N^2*d for
        equal lengths), halved when causal.  Decode workloads count 4*H*d per
        admissible (query, key) pair: n_q * N without a mask, and
        n_q * (N - n_q) + n_q (n_q + 1) / 2 per sequence under the
        bottom-right causal mask."""
        if self.decode:
            nq, nk = float(self.n_q), float(self.N)
            pairs = nq * (nk - nq) + nq * (nq + 1) / 2 if self.causal else nq * nk
            return 4.0 * self.H * self.d * self.B * pairs
        f = 4.0 * self.H * self.d * sum(float(n) * n for n in self.seqlens())
        return f / 2 if self.causal else f

    @property
    def hbm_bytes(self) -> int:
        """Algorithmic HBM bytes: read Q, K, V; write O (16-bit) and LSE (fp32)."""
        if self.decode:
            q_rows = self.B * self.n_q * self.H
            kv_rows = self.B * self.N * self.kv_heads
            return q_rows * self.d * 2 * 2 + 2 * kv_rows * self.d * 2 + q_rows * 4
        rows = self.H * sum(self.seqlens())
        in_bytes = 1 if self.dtype == "fp8" else 2
        return 3 * rows * self.d * in_bytes + rows * self.d * 2 + rows * 4

    def describe(self) -> str:
        mask = "causal" if self.causal else "full"
        if self.decode:
            return (f"{self.B} sequences of {self.n_q} query rows against {self.N} cached keys, "
                    f"H={self.H} H_kv={self.kv_heads} d={self.d} {self.dtype} {mask} "
                    f"(bottom-right)")
        extra = f", Q,K x{self.qk_mult:g}" if self.qk_mult != 1.0 else ""
        extra += ", split-KV" if self.splitkv else ""
        if self.varlen:
            return (f"{self.B} sequences of {min(self.seqlens())}..{max(self.seqlens())} rows "
                    f"(total {sum(self.seqlens())}) packed, H={self.H} d={self.d} "
                    f"{self.dtype} {mask}{extra}")
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
    # 16 causal sequences of 256..4096 rows packed along the rows (a
    # variable-length training batch)
    Workload(7, "bf16_d128_varlen16_causal", 16, 16, 4096, 128, "bf16", True, varlen=True),
    # the headline shape with FP8 E4M3 inputs (descale factors 1)
    Workload(8, "fp8_d128_n2048", 4, 16, 2048, 128, "fp8", False),
    # decode-shaped: 32 sequences of 32 query rows against 8192 cached keys,
    # 8 query heads per K/V head (fa_fwd_varlen_qk)
    Workload(9, "bf16_d128_decode_q32_k8192_gqa8", 32, 32, 8192, 128, "bf16", True,
             n_q=32, H_kv=4),
]


def workload(index: int) -> Workload:
    return WORKLOADS[index - 1]


def make_qkv(wl: Workload, seed: int | None = None):
    """CPU tensors q, k, v in the workload's dtype, drawn as the recipe says
    ([B, H, N, d]; packed [total, H, d] for varlen workloads; for decode
    workloads q [B*n_q, H, d] and k, v [B*N, H_kv, d])."""
    g = torch.Generator().manual_seed(1000 + wl.index if seed is None else seed)
    if wl.decode:
        shapes = [(wl.B * wl.n_q, wl.H, wl.d)] + [(wl.B * wl.N, wl.kv_heads, wl.d)] * 2
    else:
        shape = (sum(wl.seqlens()), wl.H, wl.d) if wl.varlen else (wl.B, wl.H, wl.N, wl.d)
        shapes = [shape] * 3
    out = []
    for shape in shapes:
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
    lens = wl.seqlens()
    b = torch.randint(0, wl.B, (count,), generator=g)
    h = torch.randint(0, wl.H, (count,), generator=g)
    i = torch.randint(0, wl.N, (count,), generator=g)
    # rows of a shorter sequence are folded into its length
    rows = set((bb, hh, ii % lens[bb]) for bb, hh, ii in zip(b.tolist(), h.tolist(), i.tolist()))
    for (bb, hh) in ((0, 0), (wl.B - 1, wl.H - 1)):
        n = lens[bb]
        fixed = {0, 1, 127, 128, n - 1}
        if wl.causal:
            for t in range(128, min(n, 1025), 128):
                fixed.update({t - 1, t})
        for r in fixed:
            if 0 <= r < n:
                rows.add((bb, hh, r))
    return sorted(rows)
