"""Seeded synthetic inputs shared by the tests, the bench and the oracle checks.

This module only draws random tensors; it holds none of the attention
arithmetic. Q, K, V and dO are standard normal draws rounded to the io dtype;
the optional bias is fp32 with standard deviation 0.5. Each tensor has its own
CPU generator seed (Q 1, K 2, V 3, dO 4, bias 5, each plus ``seed_base``), so a
tensor does not change when another one's shape does.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}


@dataclass(frozen=True)
class Shape:
    B: int
    H: int
    S_q: int
    S_kv: int
    D_qk: int
    D_v: int
    H_kv: int = 0  # K/V heads (grouped-query attention); 0 means H

    @property
    def kv_heads(self) -> int:
        return self.H_kv if self.H_kv else self.H


def _randn(shape, seed: int, device="cpu") -> torch.Tensor:
    if str(device).startswith("cuda"):
        g = torch.Generator(device=device).manual_seed(seed)
    else:
        g = torch.Generator().manual_seed(seed)
    return torch.randn(*shape, generator=g, dtype=torch.float32, device=device)


def make_inputs(shape: Shape, dtype: str = "bf16", with_bias: bool = False,
                seed_base: int = 0, device="cpu") -> dict:
    """q, do [B, H, S_q, D] and k, v [B, H_kv, S_kv, D] in the io dtype, and bias
    fp32 [1, H, S_q, S_kv] or None."""
    t = DTYPES[dtype]
    s = shape
    out = {
        "q": _randn((s.B, s.H, s.S_q, s.D_qk), 1 + seed_base, device).to(t),
        "k": _randn((s.B, s.kv_heads, s.S_kv, s.D_qk), 2 + seed_base, device).to(t),
        "v": _randn((s.B, s.kv_heads, s.S_kv, s.D_v), 3 + seed_base, device).to(t),
        "do": _randn((s.B, s.H, s.S_q, s.D_v), 4 + seed_base, device).to(t),
        "bias": None,
    }
    if with_bias:
        out["bias"] = 0.5 * _randn((1, s.H, s.S_q, s.S_kv), 5 + seed_base, device)
    return out


def packed_lengths(n: int, lo: int, hi: int, seed: int) -> list[int]:
    """n sequence lengths drawn uniformly from [lo, hi] by a seeded generator."""
    g = torch.Generator().manual_seed(seed)
    return [int(x) for x in torch.randint(lo, hi + 1, (n,), generator=g)]


def seqstarts(lengths) -> list[int]:
    """Row offsets of packed sequences: 0, then the running sums of the lengths."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return out


def make_packed_inputs(H: int, total_q: int, total_k: int, D_qk: int, D_v: int,
                       dtype: str = "bf16", H_kv: int = 0, seed_base: int = 0,
                       device="cpu") -> dict:
    """Packed-sequence tensors: q, do [H, total_q, D] and k, v [H_kv, total_k, D]
    (the batch-mode draws of one batch entry with total rows)."""
    x = make_inputs(Shape(1, H, total_q, total_k, D_qk, D_v, H_kv), dtype, seed_base=seed_base,
                    device=device)
    return {n: x[n][0] for n in ("q", "k", "v", "do")}
