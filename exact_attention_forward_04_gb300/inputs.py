"""Seeded synthetic inputs for the attention forward pass.

This module only draws random numbers and names workload shapes. It holds no
attention arithmetic, so both the float64 oracle (``oracle/``) and the CUDA
path can consume exactly the same bf16 tensors without sharing any code.

Recipe (one generator per workload):
  * ``torch.Generator().manual_seed(seed)`` on the CPU;
  * draw ``q``, ``k``, ``v`` in that order, each as
    ``torch.randn(B, H, N, d, dtype=float32, generator=g) * sigma``;
  * round each to bf16 (round-to-nearest-even, torch's ``.to``).

The five named workloads are the shapes the attention forward is measured and
checked on: a 128-token single head, two d=128 long-sequence shapes with and
without a causal mask, a 32K-token causal head set, and a d=64 batch whose
Q and K are drawn with sigma=3 so that most softmax rows are dominated by a few
keys ("peaky" rows).
"""
from __future__ import annotations

import dataclasses
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    sigma_q: float = 1.0
    sigma_k: float = 1.0
    sigma_v: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> float:
        """Metric FLOPs: 4*B*H*N^2*d, halved under the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2.0 if self.causal else f

    def describe(self) -> str:
        m = "causal" if self.causal else "full"
        return f"B={self.B},H={self.H},N={self.N},d={self.d},{m}"


WORKLOADS = (
    Workload("tiny_b1h1n128d64", 1, 1, 128, 64, False, seed=0),
    Workload("b4h16n2048d128", 4, 16, 2048, 128, False, seed=1),
    Workload("b2h32n8192d128_causal", 2, 32, 8192, 128, True, seed=2),
    Workload("b1h32n32768d128_causal", 1, 32, 32768, 128, True, seed=3),
    Workload("b16h32n1024d64_peaky", 16, 32, 1024, 64, False, seed=4,
             sigma_q=3.0, sigma_k=3.0),
)

# Few heads with a long sequence: too few 256-row query tiles to occupy the
# GPU, the case the split key/value forward is for.
SPLITKV_WORKLOADS = (
    Workload("b1h1n8192d128", 1, 1, 8192, 128, False, seed=5),
    Workload("b1h2n16384d128_causal", 1, 2, 16384, 128, True, seed=6),
)

BY_NAME = {w.name: w for w in WORKLOADS + SPLITKV_WORKLOADS}


def make_qkv(B: int, H: int, N: int, d: int, seed: int,
             sigma_q: float = 1.0, sigma_k: float = 1.0, sigma_v: float = 1.0):
    """Return CPU bf16 tensors q, k, v of shape [B, H, N, d], contiguous."""
    g = torch.Generator().manual_seed(int(seed))
    out = []
    for sigma in (sigma_q, sigma_k, sigma_v):
        x = torch.randn(B, H, N, d, dtype=torch.float32, generator=g)
        if sigma != 1.0:
            x.mul_(sigma)
        out.append(x.to(torch.bfloat16).contiguous())
    return tuple(out)


def make_qkv_on_device(B: int, H: int, N: int, d: int, seed: int, device, heads_per_draw: int = 256):
    """Seeded q, k, v drawn directly on ``device`` for shapes too large to
    draw on the host quickly: a ``torch.Generator(device)`` seeded with
    ``seed`` draws q, then k, then v, each in slices of ``heads_per_draw``
    (batch*head) slices of N(0, 1) fp32 rounded to bf16.  Returns device bf16
    tensors [B, H, N, d]; copy slices to the host for the oracle."""
    g = torch.Generator(device=device).manual_seed(int(seed))
    out = []
    for _ in range(3):
        x = torch.empty(B * H, N, d, dtype=torch.bfloat16, device=device)
        for h0 in range(0, B * H, heads_per_draw):
            h1 = min(B * H, h0 + heads_per_draw)
            x[h0:h1] = torch.randn(h1 - h0, N, d, dtype=torch.float32, device=device, generator=g)
        out.append(x.view(B, H, N, d))
    return tuple(out)


def make_workload(w: Workload):
    return make_qkv(w.B, w.H, w.N, w.d, w.seed, w.sigma_q, w.sigma_k, w.sigma_v)


def make_e4m3_codes(B: int, H: int, N: int, d: int, seed: int, max_exp_field: int = 9,
                    n_tensors: int = 3):
    """Random 8-bit codes (CPU uint8 [B, H, N, d], ``n_tensors`` of them) laid
    out as sign (bit 7), exponent field (bits 6..3) and mantissa (bits 2..0):
    sign and mantissa uniform, exponent field uniform in [0, max_exp_field].
    With max_exp_field <= 14 no code is the NaN pattern.  Plus one random
    positive factor per (batch, head) and tensor, uniform in [2^-8, 2^-4)."""
    g = torch.Generator().manual_seed(int(seed))
    codes, factors = [], []
    for _ in range(n_tensors):
        s = torch.randint(0, 2, (B, H, N, d), generator=g, dtype=torch.int32)
        e = torch.randint(0, max_exp_field + 1, (B, H, N, d), generator=g, dtype=torch.int32)
        m = torch.randint(0, 8, (B, H, N, d), generator=g, dtype=torch.int32)
        codes.append(((s << 7) | (e << 3) | m).to(torch.uint8))
        u = torch.rand(B, H, generator=g, dtype=torch.float32)
        factors.append((2.0 ** (-8 + 4 * u)).to(torch.float32))
    return codes, factors
