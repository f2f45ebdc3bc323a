"""GPU parity of the packed variable-length path (sdpa_fwd_varlen /
sdpa_bwd_varlen) against the packed-sequence oracle, element by element, and
its bitwise agreement with batch mode when every sequence has the same length.

Cases cover ragged lengths with tails inside a tile, cross-attention lengths,
grouped and single K/V heads, dropout with max lengths above the real ones,
sequences without queries or without keys, d 64 / 128 / 192, bf16 and fp16,
through both backwards (the default fused one, whose fp32 dQ accumulator spans
the packed rows, and the deterministic one).
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import pytest
import torch

import oracle
from oracle import varlen as ovl
from parity_util import assert_close, assert_lse
from scaled_dot_product_06_gb300 import (sdpa_bwd, sdpa_bwd_varlen, sdpa_device_error, sdpa_fwd,
                                         sdpa_fwd_varlen)
from scaled_dot_product_06_gb300.inputs import make_packed_inputs, packed_lengths, seqstarts

pytestmark = pytest.mark.gpu


@dataclass(frozen=True)
class VCase:
    H: int
    lq: tuple
    lk: tuple
    D_qk: int
    D_v: int
    dtype: str = "bf16"
    causal: bool = False
    p: float = 0.0
    H_kv: int = 0
    max_q: int = 0  # 0: the longest query length
    max_k: int = 0
    seed: int = 0x55
    offset: int = 3

    @property
    def sc(self):
        return 1.0 / np.sqrt(self.D_qk)

    @property
    def maxes(self):
        return self.max_q or max(self.lq), self.max_k or max(self.lk)

    def packed(self):
        mq, mk = self.maxes
        return ovl.Packed(tuple(seqstarts(self.lq)), tuple(seqstarts(self.lk)), self.H, self.D_qk,
                          self.D_v, self.sc, self.causal, self.p, self.seed, self.offset, self.H_kv,
                          mq, mk)


def run_varlen(c: VCase, x: dict, deterministic=False):
    dev = "cuda"
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    sq = torch.tensor(seqstarts(c.lq), dtype=torch.int32, device=dev)
    sk = torch.tensor(seqstarts(c.lk), dtype=torch.int32, device=dev)
    mq, mk = c.maxes
    kw = dict(scale=c.sc, is_causal=c.causal, dropout_p=c.p, seed=c.seed, offset=c.offset)
    o, lse = sdpa_fwd_varlen(q, k, v, sq, sk, mq, mk, **kw)
    dq, dk, dv = sdpa_bwd_varlen(q, k, v, o, do, lse, sq, sk, mq, mk, deterministic=deterministic,
                                 **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0, "a kernel wait ran out"
    return o, lse, dq, dk, dv


CASES = [
    VCase(2, (130, 1, 300, 77, 256), (130, 1, 300, 77, 256), 128, 128, causal=True),
    VCase(4, (64, 200, 129), (100, 50, 384), 64, 64, dtype="fp16", H_kv=2),
    VCase(2, (256, 130, 5), (256, 130, 8), 192, 128, causal=True, p=0.1),
    VCase(4, (128, 384, 200), (128, 384, 200), 128, 128, causal=True, H_kv=1),
    VCase(2, (50, 0, 70, 33), (0, 40, 90, 33), 64, 64, causal=True),
    VCase(3, (100, 60), (92, 140), 128, 128, p=0.2, max_q=512, max_k=512),
]


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("c", CASES, ids=lambda c: f"H{c.H}kv{c.H_kv}-d{c.D_qk}-{c.dtype}"
                         f"{'-causal' if c.causal else ''}{'-p' + str(c.p) if c.p else ''}-"
                         f"{len(c.lq)}seq")
def test_varlen_matches_oracle(c, deterministic):
    pk = c.packed()
    x = make_packed_inputs(c.H, sum(c.lq), sum(c.lk), c.D_qk, c.D_v, c.dtype, c.H_kv)
    o, lse, dq, dk, dv = run_varlen(c, x, deterministic)
    o_ref, lse_ref = ovl.forward(pk, x["q"], x["k"], x["v"])
    assert_close("o", o, o_ref)
    assert_lse(lse, lse_ref)
    dq_ref, dk_ref, dv_ref = ovl.backward(pk, x["q"], x["k"], x["v"], x["do"])
    assert_close("dq", dq, dq_ref)
    assert_close("dk", dk, dk_ref)
    assert_close("dv", dv, dv_ref)


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused", "deterministic"])
@pytest.mark.parametrize("p", [0.0, 0.15])
def test_uniform_lengths_bitwise_equal_batch_mode(p, deterministic):
    """Equal lengths: the packed path computes exactly the batch-mode numbers
    (same tiles, same accumulation order, same dropout bits); the fused
    backward's dQ within fp32 summation order (its reductions add in arrival
    order)."""
    B, H, S, D = 3, 4, 384, 128
    c = VCase(H, (S,) * B, (S,) * B, D, D, causal=True, p=p)
    x = make_packed_inputs(H, B * S, B * S, D, D)
    o, lse, dq, dk, dv = run_varlen(c, x, deterministic)
    to_b = lambda t: t.reshape(t.shape[0], B, S, t.shape[-1]).transpose(0, 1).contiguous().cuda()
    kw = dict(scale=c.sc, is_causal=True, dropout_p=p, seed=c.seed, offset=c.offset)
    qb, kb, vb, dob = (to_b(x[n]) for n in ("q", "k", "v", "do"))
    ob, lseb = sdpa_fwd(qb, kb, vb, **kw)
    dqb, dkb, dvb, _ = sdpa_bwd(qb, kb, vb, ob, dob, lseb, deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    from_b = lambda t: t.transpose(0, 1).reshape(t.shape[1], B * S, t.shape[-1])
    assert torch.equal(from_b(ob), o)
    assert torch.equal(lseb.transpose(0, 1).reshape(H, B * S), lse)
    if deterministic:
        assert torch.equal(from_b(dqb), dq)
    else:
        assert_close("dq packed vs batch", dq, from_b(dqb).double().cpu().numpy(), rel=1e-2)
    assert torch.equal(from_b(dkb), dk)
    assert torch.equal(from_b(dvb), dv)


def test_packed_h32_d128_causal_16_sequences_sampled():
    """The packed-sequence workload the benchmark times (16 sequences of
    512..8192 tokens, 32 heads, d 128, causal), through the fused and the
    deterministic backward: two sequences checked on sampled rows and key
    columns of one head, the others through the key-sum invariants (dK sums to
    0 over each sequence's keys, dV to the sequence's query-sum of dO)."""
    lens = tuple(packed_lengths(16, 512, 8192, seed=2024))
    c = VCase(32, lens, lens, 128, 128, causal=True)
    pk = c.packed()
    x = make_packed_inputs(32, sum(lens), sum(lens), 128, 128)
    runs = {"fused": run_varlen(c, x), "deterministic": run_varlen(c, x, deterministic=True)}
    rng = np.random.default_rng(9)
    for i, h in ((int(np.argmax(lens)), 5), (3, 30)):
        pr = pk.sequence(i)
        a, b = pk.seqstart_q[i], pk.seqstart_q[i + 1]
        n = b - a
        xs = {m: x[m][:, a:b][None] for m in ("q", "k", "v", "do")}
        rows = np.unique(np.concatenate([np.arange(min(n, 40)), np.arange(max(0, n - 40), n),
                                         rng.integers(0, n, 40)]))
        cols = np.unique(np.concatenate([np.arange(min(n, 24)), np.arange(max(0, n - 24), n),
                                         rng.integers(0, n, 24)]))
        o_ref, lse_ref = oracle.forward_head(pr, 0, h, xs["q"], xs["k"], xs["v"], rows=rows)
        dq_r, dk_c, dv_c, _ = oracle.backward_head(pr, 0, h, xs["q"], xs["k"], xs["v"], xs["do"],
                                                   rows=rows, cols=cols, row_chunk=2048)
        for tag, (o, lse, dq, dk, dv) in runs.items():
            r_t, c_t = (torch.as_tensor(a + r, device=o.device) for r in (rows, cols))
            assert_close(f"o seq {i}", o[h][r_t], o_ref)
            assert_lse(lse[h][r_t], lse_ref)
            assert_close(f"dq seq {i} ({tag})", dq[h][r_t], dq_r)
            assert_close(f"dk seq {i} ({tag})", dk[h][c_t], dk_c)
            assert_close(f"dv seq {i} ({tag})", dv[h][c_t], dv_c)
    starts = pk.seqstart_q
    for tag, (o, lse, dq, dk, dv) in runs.items():
        for i in range(16):
            a, b = starts[i], starts[i + 1]
            dk64 = dk[:, a:b].double()
            rel = dk64.sum(dim=1).abs().max().item() / dk64.abs().sum(dim=1).max().item()
            assert rel < 2e-2, f"{tag}, sequence {i}: key-sum of dK is not ~0 (relative {rel:.3e})"
            assert_close(f"sum_j dV seq {i} ({tag})", dv[:, a:b].double().sum(dim=1).cpu(),
                         x["do"][:, a:b].double().sum(dim=1).numpy(), rel=3e-2)
    # the two backwards agree on every element, within the bf16 rounding of
    # the outputs
    f, d = runs["fused"], runs["deterministic"]
    for name, k in (("dq", 2), ("dk", 3), ("dv", 4)):
        diff = (f[k].float() - d[k].float()).abs().max().item()
        top = d[k].float().abs().max().item()
        assert diff <= 1e-2 * top, f"{name}: fused vs deterministic max|diff| {diff:.3e} (max {top:.3e})"


def test_packed_dropout_bits_drawn_beforehand_give_the_same_bits():
    """Packed: the mask of the padded [b, h, max_q, max_k] frame, passed in,
    gives the bits of the drawing path."""
    from scaled_dot_product_06_gb300 import sdpa_dropout_mask
    c = VCase(2, (100, 60), (92, 140), 128, 128, p=0.2, max_q=512, max_k=512)
    x = make_packed_inputs(c.H, sum(c.lq), sum(c.lk), c.D_qk, c.D_v, c.dtype)
    a = run_varlen(c, x)
    dev = "cuda"
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    sq = torch.tensor(seqstarts(c.lq), dtype=torch.int32, device=dev)
    sk = torch.tensor(seqstarts(c.lk), dtype=torch.int32, device=dev)
    mq, mk = c.maxes
    mask = sdpa_dropout_mask(len(c.lq), c.H, mq, mk, c.p, c.seed, c.offset)
    kw = dict(scale=c.sc, is_causal=c.causal, dropout_p=c.p, seed=c.seed, offset=c.offset,
              dropout_mask=mask)
    o, lse = sdpa_fwd_varlen(q, k, v, sq, sk, mq, mk, **kw)
    dq, dk, dv = sdpa_bwd_varlen(q, k, v, o, do, lse, sq, sk, mq, mk, **kw)
    torch.cuda.synchronize()
    for name, x1, x2 in zip(("o", "lse", "dq", "dk", "dv"), a, (o, lse, dq, dk, dv)):
        if name == "dq":  # the fused backward's reductions add in arrival order
            assert_close("dq drawn vs given bits", x2, x1.double().cpu().numpy(), rel=1e-2)
        else:
            assert torch.equal(x1, x2), name
    # the deterministic backward: every result bitwise
    a = run_varlen(c, x, deterministic=True)
    dq, dk, dv = sdpa_bwd_varlen(q, k, v, o, do, lse, sq, sk, mq, mk, deterministic=True, **kw)
    torch.cuda.synchronize()
    for x1, x2 in zip(a, (o, lse, dq, dk, dv)):
        assert torch.equal(x1, x2)


def test_statistics_only_workspace_runs_the_deterministic_backward():
    """A caller's workspace of sdpa_bwd_varlen_workspace_size(b, h, total_q)
    bytes (the row statistics alone, no room for the fused backward's dQ
    accumulator) runs the deterministic backward: its bits, exactly."""
    from scaled_dot_product_06_gb300 import sdpa_bwd_varlen_workspace_size
    c = VCase(4, (130, 1, 300, 77), (130, 1, 300, 77), 128, 128, causal=True)
    x = make_packed_inputs(c.H, sum(c.lq), sum(c.lk), c.D_qk, c.D_v, c.dtype)
    det = run_varlen(c, x, deterministic=True)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    sq = torch.tensor(seqstarts(c.lq), dtype=torch.int32, device="cuda")
    mq, mk = c.maxes
    small = sdpa_bwd_varlen_workspace_size(len(c.lq), c.H, sum(c.lq))
    full = sdpa_bwd_varlen_workspace_size(len(c.lq), c.H, sum(c.lq), c.D_qk)
    assert small < full
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    dq, dk, dv = sdpa_bwd_varlen(q, k, v, det[0], do, det[1], sq, sq, mq, mk, scale=c.sc,
                                 is_causal=True, workspace=ws)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    for name, a, b in zip(("dq", "dk", "dv"), (dq, dk, dv), det[2:]):
        assert torch.equal(a, b), name
