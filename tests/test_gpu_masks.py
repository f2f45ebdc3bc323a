"""GPU parity of the mask variants (local windows, bottom-right alignment)
against the oracle, element by element, in batch and packed mode; and the
equalities that make the window path the causal / unmasked path when it
should be (bitwise).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from oracle import varlen as ovl
from parity_util import assert_close, assert_lse
from scaled_dot_product_06_gb300 import (sdpa_bwd, sdpa_bwd_varlen, sdpa_device_error, sdpa_fwd,
                                         sdpa_fwd_varlen)
from scaled_dot_product_06_gb300.inputs import Shape, make_inputs, make_packed_inputs, seqstarts

pytestmark = pytest.mark.gpu

SEED, OFFSET = 0x77, 5

# (B, H, H_kv, S_q, S_kv, D_qk, D_v, dtype, window, bottom_right, p, bias)
CASES = [
    (1, 2, 2, 640, 640, 128, 128, "bf16", (100, 0), False, 0.0, False),   # sliding window
    (1, 4, 2, 300, 700, 64, 64, "fp16", (-1, 0), True, 0.0, False),       # bottom-right causal
    (1, 2, 2, 700, 300, 128, 128, "bf16", (-1, 0), True, 0.0, False),     # rows without keys
    (1, 2, 2, 400, 520, 192, 128, "bf16", (64, 200), False, 0.1, False),  # two sides, dropout
    (1, 2, 1, 384, 384, 64, 64, "bf16", (1, 0), False, 0.0, False),       # two keys per row
    (2, 2, 2, 512, 512, 128, 128, "bf16", (256, 32), False, 0.0, True),   # window and bias
    (1, 2, 2, 333, 1000, 128, 128, "bf16", (130, 130), True, 0.0, False), # ragged, bottom-right
    # one key tile: query tiles without keys keep the accumulator path (dQ = 0
    # there); a window every query tile meets takes the direct dQ write
    (1, 2, 2, 300, 100, 128, 128, "bf16", (-1, 0), True, 0.0, False),     # bottom-right, s_kv < 128
    (1, 2, 2, 260, 128, 64, 64, "bf16", (40, 0), False, 0.0, False),      # late rows see no key
    (1, 2, 2, 200, 128, 64, 64, "bf16", (300, 0), False, 0.0, True),      # wide window, bias
]


def case_id(c):
    B, H, H_kv, S_q, S_kv, D_qk, D_v, dt, win, br, p, bias = c
    return (f"b{B}h{H}kv{H_kv}-{S_q}x{S_kv}-d{D_qk}-{dt}-w{win[0]}_{win[1]}"
            f"{'-br' if br else ''}{'-p' + str(p) if p else ''}{'-bias' if bias else ''}")


@pytest.mark.parametrize("c", CASES, ids=case_id)
def test_window_matches_oracle(c):
    B, H, H_kv, S_q, S_kv, D_qk, D_v, dt, win, br, p, with_bias = c
    shp = Shape(B, H, S_q, S_kv, D_qk, D_v, H_kv)
    x = make_inputs(shp, dt, with_bias=with_bias)
    scale = 1.0 / np.sqrt(D_qk)
    pr = oracle.Problem(B, H, S_q, S_kv, D_qk, D_v, scale, False, p, SEED, OFFSET, H_kv, win, br)
    dev = "cuda"
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    bias = None if x["bias"] is None else x["bias"].to(dev)
    kw = dict(scale=scale, dropout_p=p, seed=SEED, offset=OFFSET, bias=bias, window=win,
              bottom_right=br)
    o, lse = sdpa_fwd(q, k, v, **kw)
    o_ref, lse_ref = oracle.forward(pr, x["q"], x["k"], x["v"], x["bias"])
    assert_close("o", o, o_ref)
    assert_lse(lse, lse_ref)
    dq_r, dk_r, dv_r, db_r = oracle.backward(pr, x["q"], x["k"], x["v"], x["do"], x["bias"])
    for det in (False, True):  # the default (fused) and the deterministic backward
        dq, dk, dv, dbias = sdpa_bwd(q, k, v, o, do, lse, deterministic=det, **kw)
        torch.cuda.synchronize()
        assert sdpa_device_error() == 0
        assert_close(f"dq det={det}", dq, dq_r)
        assert_close(f"dk det={det}", dk, dk_r)
        assert_close(f"dv det={det}", dv, dv_r)
        if with_bias:
            assert_close(f"dbias det={det}", dbias, db_r)


@pytest.mark.parametrize("scale", [-0.1, 0.0])
def test_window_with_negative_or_zero_scale(scale):
    """A window under a negative scale (raw scores, row max from their
    minimum, masked keys at +inf before scaling) and under a zero scale (the
    kernel that scales first)."""
    B, H, S_q, S_kv, D = 1, 2, 384, 520, 128
    win, br = (100, 20), True
    x = make_inputs(Shape(B, H, S_q, S_kv, D, D), "bf16")
    pr = oracle.Problem(B, H, S_q, S_kv, D, D, scale, False, window=win, bottom_right=br)
    q, k, v, do = (x[n].to("cuda") for n in ("q", "k", "v", "do"))
    kw = dict(scale=scale, window=win, bottom_right=br)
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv, _ = sdpa_bwd(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    o_ref, lse_ref = oracle.forward(pr, x["q"], x["k"], x["v"])
    assert_close("o", o, o_ref)
    assert_lse(lse, lse_ref)
    dq_r, dk_r, dv_r, _ = oracle.backward(pr, x["q"], x["k"], x["v"], x["do"])
    assert_close("dq", dq, dq_r)
    assert_close("dk", dk, dk_r)
    assert_close("dv", dv, dv_r)


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused", "deterministic"])
def test_packed_window_bottom_right_matches_oracle(deterministic):
    lq, lk = (100, 300, 7, 256), (200, 150, 64, 256)
    H, H_kv, D = 4, 2, 128
    win, br = (50, 10), True
    scale = 1.0 / np.sqrt(D)
    pk = ovl.Packed(tuple(seqstarts(lq)), tuple(seqstarts(lk)), H, D, D, scale, False, H_kv=H_kv,
                    window=win, bottom_right=br)
    x = make_packed_inputs(H, sum(lq), sum(lk), D, D, "bf16", H_kv)
    dev = "cuda"
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    sq = torch.tensor(seqstarts(lq), dtype=torch.int32, device=dev)
    sk = torch.tensor(seqstarts(lk), dtype=torch.int32, device=dev)
    kw = dict(scale=scale, window=win, bottom_right=br)
    o, lse = sdpa_fwd_varlen(q, k, v, sq, sk, max(lq), max(lk), **kw)
    dq, dk, dv = sdpa_bwd_varlen(q, k, v, o, do, lse, sq, sk, max(lq), max(lk),
                                 deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    o_ref, lse_ref = ovl.forward(pk, x["q"], x["k"], x["v"])
    assert_close("o", o, o_ref)
    assert_lse(lse, lse_ref)
    dq_r, dk_r, dv_r = ovl.backward(pk, x["q"], x["k"], x["v"], x["do"])
    assert_close("dq", dq, dq_r)
    assert_close("dk", dk, dk_r)
    assert_close("dv", dv, dv_r)


@pytest.mark.parametrize("causal", [False, True])
def test_window_path_equals_plain_path_bitwise(causal):
    """Windows that admit the same pairs give the same bits as the plain
    causal / unmasked calls: (-1, 0) and windows past the problem's size (the
    plain kernels), and (S-1, 0) / (S-1, S-1), which the kernels compiled for
    general windows run."""
    B, H, S, D = 1, 4, 700, 128
    x = make_inputs(Shape(B, H, S, S, D, D), "bf16", device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o_a, lse_a = sdpa_fwd(q, k, v, is_causal=causal)
    wins = [(-1, 0), (S - 1, 0)] if causal else [(5000, 5000), (S - 1, S - 1)]
    # every gradient of the deterministic backward; dK and dV of the default
    # one (its dQ sums fp32 reductions in arrival order)
    for det in (True, False):
        g_a = sdpa_bwd(q, k, v, o_a, do, lse_a, is_causal=causal, deterministic=det)
        for win in wins:
            o_b, lse_b = sdpa_fwd(q, k, v, window=win, bottom_right=False)
            g_b = sdpa_bwd(q, k, v, o_b, do, lse_b, window=win, bottom_right=False,
                           deterministic=det)
            torch.cuda.synchronize()
            assert torch.equal(o_a, o_b) and torch.equal(lse_a, lse_b), win
            for a, b in zip(g_a[0 if det else 1:3], g_b[0 if det else 1:3]):
                assert torch.equal(a, b), (win, det)


def test_diagonal_window_is_exact():
    """Window (0, 0): each row sees its own key alone, so P = 1 there. Then
    O = V and dV = dO exactly (one product with 1.0, nothing else added), and
    dS = dP - D = 0 in exact arithmetic: dQ and dK are only the difference of
    two fp32 sums of the same 64 products in different orders, bounded by
    ~2 * 64 * 2^-24 * sum|dO_d V_d| (< 1e-3 here, times scale * |K| < 1)."""
    B, H, S, D = 1, 2, 384, 64
    x = make_inputs(Shape(B, H, S, S, D, D), "bf16", device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse = sdpa_fwd(q, k, v, window=(0, 0))
    dq, dk, dv, _ = sdpa_bwd(q, k, v, o, do, lse, window=(0, 0))
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    assert torch.equal(o, v)
    assert torch.equal(dv, do)
    ref_lse = (q.double() * k.double()).sum(-1) / np.sqrt(D)
    assert (lse.double() - ref_lse).abs().max().item() < 1e-3
    assert dq.abs().max().item() < 1e-3 and dk.abs().max().item() < 1e-3


def alibi_slopes(H):
    """The geometric ALiBi slopes 2^(-8 (h + 1) / H)."""
    return [2.0 ** (-8.0 * (h + 1) / H) for h in range(H)]


# (B, H, H_kv, S_q, S_kv, D, dtype, window, bottom_right, p, per_batch)
ALIBI_CASES = [
    (1, 4, 2, 300, 520, 64, "bf16", None, False, 0.0, False),      # unmasked: bottom-right
    (2, 4, 4, 384, 384, 128, "fp16", (-1, 0), False, 0.0, True),   # causal, slopes per batch
    (1, 2, 2, 333, 700, 128, "bf16", (200, 0), True, 0.1, False),  # window, bottom-right, dropout
]


@pytest.mark.parametrize("c", ALIBI_CASES, ids=lambda c: f"b{c[0]}h{c[1]}-{c[3]}x{c[4]}-d{c[5]}-"
                         f"w{c[7]}{'-br' if c[8] else ''}{'-p' if c[9] else ''}")
def test_alibi_matches_oracle(c):
    B, H, H_kv, S_q, S_kv, D, dt, win, br, p, per_batch = c
    x = make_inputs(Shape(B, H, S_q, S_kv, D, D, H_kv), dt)
    sl = np.array([[s * (1.0 + 0.5 * b) for s in alibi_slopes(H)] for b in range(B)]
                  if per_batch else [alibi_slopes(H)] * B, dtype=np.float32)
    slopes_t = torch.tensor(sl if per_batch else sl[0], device="cuda")
    scale = 1.0 / np.sqrt(D)
    pr = oracle.Problem(B, H, S_q, S_kv, D, D, scale, False, p, SEED, OFFSET, H_kv, win, br,
                        alibi_slopes=tuple(tuple(float(v) for v in row) for row in sl))
    q, k, v, do = (x[n].to("cuda") for n in ("q", "k", "v", "do"))
    kw = dict(scale=scale, dropout_p=p, seed=SEED, offset=OFFSET, window=win, bottom_right=br,
              alibi_slopes=slopes_t)
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv, _ = sdpa_bwd(q, k, v, o, do, lse, **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    o_ref, lse_ref = oracle.forward(pr, x["q"], x["k"], x["v"])
    assert_close("o", o, o_ref)
    assert_lse(lse, lse_ref)
    dq_r, dk_r, dv_r, _ = oracle.backward(pr, x["q"], x["k"], x["v"], x["do"])
    assert_close("dq", dq, dq_r)
    assert_close("dk", dk, dk_r)
    assert_close("dv", dv, dv_r)


@pytest.mark.parametrize("deterministic", [False, True], ids=["fused", "deterministic"])
def test_packed_alibi_causal_matches_oracle(deterministic):
    lq = lk = (130, 257, 64)
    H, D = 4, 128
    sl = np.array([[s * (i + 1) for s in alibi_slopes(H)] for i in range(3)], dtype=np.float32)
    scale = 1.0 / np.sqrt(D)
    pk = ovl.Packed(tuple(seqstarts(lq)), tuple(seqstarts(lk)), H, D, D, scale, True,
                    alibi_slopes=tuple(tuple(float(v) for v in row) for row in sl))
    x = make_packed_inputs(H, sum(lq), sum(lk), D, D, "bf16")
    q, k, v, do = (x[n].to("cuda") for n in ("q", "k", "v", "do"))
    st = torch.tensor(seqstarts(lq), dtype=torch.int32, device="cuda")
    kw = dict(scale=scale, is_causal=True, alibi_slopes=torch.tensor(sl, device="cuda"))
    o, lse = sdpa_fwd_varlen(q, k, v, st, st, max(lq), max(lk), **kw)
    dq, dk, dv = sdpa_bwd_varlen(q, k, v, o, do, lse, st, st, max(lq), max(lk),
                                 deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    o_ref, lse_ref = ovl.forward(pk, x["q"], x["k"], x["v"])
    assert_close("o", o, o_ref)
    assert_lse(lse, lse_ref)
    dq_r, dk_r, dv_r = ovl.backward(pk, x["q"], x["k"], x["v"], x["do"])
    assert_close("dq", dq, dq_r)
    assert_close("dk", dk, dk_r)
    assert_close("dv", dv, dv_r)
