"""fp64 oracle of attention over packed variable-length sequences.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle``: only ``tests/``,
``__graft_entry__.smoke()`` and ``bench.py``'s ``cpu_baseline`` / reference
legs may import it.

CK tile fmha_bwd_kernel.hpp has a group mode: the kernel arguments carry
seqstart_q_ptr / seqstart_k_ptr, and for batch entry i the Q / dO / LSE
pointers move to row seqstart_q[i] and the K / V / dK / dV pointers to row
seqstart_k[i], with seqlen_q / seqlen_k taken as the differences of
consecutive starts. Each sequence is thus an attention problem of its own on
its rows, and that is what this module computes, by handing each sequence's
rows to the batch-mode oracle (``sdpa_oracle``) as a problem with B = 1.

Layout (the batch-mode BHSD with the batch folded into the rows): q, do
[H, total_q, D], k, v [H_kv, total_k, D], lse [H, total_q].

Readings where the pages are silent:

* The causal mask is top-left within each sequence (local key j visible to
  local query i iff j <= i), as in batch mode; windows and the bottom-right
  alignment likewise use each sequence's own lengths.
* A query row whose sequence has no key gets O = 0, LSE = -inf and dQ = 0;
  a key whose sequence has no query gets dK = dV = 0 (the batch-mode rule for
  a row that sees no key, and an empty sum).
* Dropout: sequence i draws the bits of batch entry i of a
  [B, H, max_seqlen_q, max_seqlen_k] batch-mode problem, local row and
  column for row and column (``Problem.drop_frame``).
* No bias with packed sequences.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import sdpa_oracle as so


@dataclass(frozen=True)
class Packed:
    """Sizes and scalar parameters of one packed-sequence call."""

    seqstart_q: tuple
    seqstart_k: tuple
    H: int
    D_qk: int
    D_v: int
    scale: float
    is_causal: bool = False
    dropout_p: float = 0.0
    seed: int = 0
    offset: int = 0
    H_kv: int = 0
    max_seqlen_q: int = 0  # 0: the longest sequence
    max_seqlen_k: int = 0
    window: tuple | None = None  # as in sdpa_oracle.Problem, per sequence
    bottom_right: bool = False
    alibi_slopes: tuple | None = None  # [B][H], sequence i taking row i

    @property
    def B(self) -> int:
        return len(self.seqstart_q) - 1

    @property
    def kv_heads(self) -> int:
        return self.H_kv if self.H_kv else self.H

    def lens(self, i: int) -> tuple[int, int]:
        return (self.seqstart_q[i + 1] - self.seqstart_q[i], self.seqstart_k[i + 1] - self.seqstart_k[i])

    def frame(self) -> tuple[int, int]:
        mq = self.max_seqlen_q or max(self.lens(i)[0] for i in range(self.B))
        mk = self.max_seqlen_k or max(self.lens(i)[1] for i in range(self.B))
        return mq, mk

    def sequence(self, i: int) -> so.Problem:
        """Sequence i as a batch-mode problem with one batch entry."""
        lq, lk = self.lens(i)
        mq, mk = self.frame()
        return so.Problem(1, self.H, lq, lk, self.D_qk, self.D_v, self.scale, self.is_causal,
                          self.dropout_p, self.seed, self.offset, self.H_kv, self.window,
                          self.bottom_right, drop_frame=(self.B, mq, mk, i),
                          alibi_slopes=None if self.alibi_slopes is None else (self.alibi_slopes[i],))


def _rows(x, a: int, b: int):
    """Rows a..b-1 of a packed [heads, total, D] tensor as a [1, heads, n, D] array."""
    return so._f64(x)[:, a:b][None]


def forward(pk: Packed, q, k, v):
    """O [H, total_q, D_v] and LSE [H, total_q]."""
    total_q = pk.seqstart_q[-1]
    o = np.zeros((pk.H, total_q, pk.D_v))
    lse = np.full((pk.H, total_q), -np.inf)
    for i in range(pk.B):
        qa, qb = pk.seqstart_q[i], pk.seqstart_q[i + 1]
        ka, kb = pk.seqstart_k[i], pk.seqstart_k[i + 1]
        if qb == qa or kb == ka:
            continue  # no query, or no key: O = 0 and LSE = -inf
        oi, li = so.forward(pk.sequence(i), _rows(q, qa, qb), _rows(k, ka, kb), _rows(v, ka, kb))
        o[:, qa:qb] = oi[0]
        lse[:, qa:qb] = li[0]
    return o, lse


def backward(pk: Packed, q, k, v, do):
    """dQ [H, total_q, D_qk], dK [H_kv, total_k, D_qk], dV [H_kv, total_k, D_v]."""
    total_q, total_k = pk.seqstart_q[-1], pk.seqstart_k[-1]
    dq = np.zeros((pk.H, total_q, pk.D_qk))
    dk = np.zeros((pk.kv_heads, total_k, pk.D_qk))
    dv = np.zeros((pk.kv_heads, total_k, pk.D_v))
    for i in range(pk.B):
        qa, qb = pk.seqstart_q[i], pk.seqstart_q[i + 1]
        ka, kb = pk.seqstart_k[i], pk.seqstart_k[i + 1]
        if qb == qa or kb == ka:
            continue  # an empty side: every gradient of the sequence is 0
        g = so.backward(pk.sequence(i), _rows(q, qa, qb), _rows(k, ka, kb), _rows(v, ka, kb),
                        _rows(do, qa, qb))
        dq[:, qa:qb] = g[0][0]
        dk[:, ka:kb] = g[1][0]
        dv[:, ka:kb] = g[2][0]
    return dq, dk, dv
