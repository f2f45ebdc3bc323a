"""Pins of the oracle's ALiBi reading to facts outside it.

* Zero slopes are no ALiBi.
* Under a causal mask every visible key has j <= i + off, so the penalty
  -m |j - i - off| equals m j - m (i + off): a bias that depends on the key
  alone plus a constant per row, which the softmax cancels. O and every
  gradient then equal those of the oracle's (separately pinned) bias path with
  Bias_ij = m j, and LSE moves by exactly -m (i + off).
* Without a mask the penalty is -m times the distance of the key from the
  query's aligned position: PyTorch float64 attention with that distance
  taken from torch.cdist (|x_i - y_j| of 1-D positions), plus autograd.
* With a bottom-right window the penalty is aligned bottom-right; with a
  top-left one, top-left (the mask decides, as CK's make_alibi_from_lr_mask
  takes the mask type).
"""
import numpy as np
import pytest
import torch

from oracle import Problem, backward, forward, varlen

RNG = np.random.default_rng(99)


def rand(*shape):
    return RNG.standard_normal(shape)


def tensors(pr):
    return (rand(pr.B, pr.H, pr.S_q, pr.D_qk), rand(pr.B, pr.kv_heads, pr.S_kv, pr.D_qk),
            rand(pr.B, pr.kv_heads, pr.S_kv, pr.D_v), rand(pr.B, pr.H, pr.S_q, pr.D_v))


SLOPES = ((0.5, 0.125, 0.03125), (0.25, 0.0625, 0.7))  # [B=2][H=3]


def test_zero_slopes_are_no_alibi():
    base = dict(B=2, H=3, S_q=6, S_kv=9, D_qk=4, D_v=3, scale=0.5, is_causal=True)
    pr0 = Problem(**base)
    pr1 = Problem(**base, alibi_slopes=((0.0,) * 3,) * 2)
    q, k, v, do = tensors(pr0)
    np.testing.assert_array_equal(forward(pr0, q, k, v)[0], forward(pr1, q, k, v)[0])
    for a, b in zip(backward(pr0, q, k, v, do)[:3], backward(pr1, q, k, v, do)[:3]):
        np.testing.assert_array_equal(a, b)


@pytest.mark.parametrize("S_q,S_kv,br", [(7, 7, False), (5, 9, True), (8, 11, False)])
def test_causal_alibi_is_a_key_bias_plus_a_row_constant(S_q, S_kv, br):
    B, H = 2, 3
    pr = Problem(B, H, S_q, S_kv, 4, 3, 0.5, True, bottom_right=br, alibi_slopes=SLOPES)
    pr_b = Problem(B, H, S_q, S_kv, 4, 3, 0.5, True, bottom_right=br)
    q, k, v, do = tensors(pr)
    off = S_kv - S_q if br else 0
    m = np.array(SLOPES)                                   # [B, H]
    j = np.arange(S_kv)
    i = np.arange(S_q)
    o, lse = forward(pr, q, k, v)
    dq, dk, dv, _ = backward(pr, q, k, v, do)
    # the bias path takes one [1, H, S_q, S_kv] tensor for every batch entry,
    # so each entry is compared with a bias built from its own slopes
    for b in range(B):
        bias = np.broadcast_to(m[b][:, None, None] * j[None, None, :], (H, S_q, S_kv))[None].copy()
        o_b, lse_b = forward(pr_b, q, k, v, bias)
        dq_b, dk_b, dv_b, _ = backward(pr_b, q, k, v, do, bias)
        np.testing.assert_allclose(o[b], o_b[b], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[b], lse_b[b] - m[b][:, None] * (i[None, :] + off),
                                   rtol=1e-12, atol=1e-12)
        for a, c in ((dq, dq_b), (dk, dk_b), (dv, dv_b)):
            np.testing.assert_allclose(a[b], c[b], rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("S_q,S_kv", [(6, 6), (5, 9), (9, 4)])
def test_unmasked_alibi_matches_torch_cdist(S_q, S_kv):
    B, H = 2, 3
    pr = Problem(B, H, S_q, S_kv, 4, 3, 0.5, False, alibi_slopes=SLOPES)
    q, k, v, do = tensors(pr)
    off = S_kv - S_q  # no mask: bottom-right
    pos_q = torch.arange(S_q, dtype=torch.float64)[:, None] + off
    pos_k = torch.arange(S_kv, dtype=torch.float64)[:, None]
    dist = torch.cdist(pos_q, pos_k, p=1.0)                   # |i + off - j|
    mask = -torch.tensor(SLOPES, dtype=torch.float64)[:, :, None, None] * dist
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=0.5)
    to.backward(torch.tensor(do))
    o, _ = forward(pr, q, k, v)
    dq, dk, dv, _ = backward(pr, q, k, v, do)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("br", [False, True])
def test_windowed_alibi_follows_the_mask_alignment(br):
    B, H, S_q, S_kv = 2, 3, 7, 12
    win = (3, 2)
    pr = Problem(B, H, S_q, S_kv, 4, 3, 0.5, False, window=win, bottom_right=br,
                 alibi_slopes=SLOPES)
    q, k, v, do = tensors(pr)
    off = S_kv - S_q if br else 0
    pos_q = torch.arange(S_q, dtype=torch.float64)[:, None] + off
    pos_k = torch.arange(S_kv, dtype=torch.float64)[:, None]
    band = np.tril(np.triu(np.ones((S_q, S_kv), dtype=bool), k=off - win[0]), k=off + win[1])
    mask = -torch.tensor(SLOPES, dtype=torch.float64)[:, :, None, None] * torch.cdist(pos_q, pos_k, p=1.0)
    mask = mask.masked_fill(~torch.tensor(band), float("-inf"))
    to = torch.nn.functional.scaled_dot_product_attention(torch.tensor(q), torch.tensor(k),
                                                          torch.tensor(v), attn_mask=mask, scale=0.5)
    np.testing.assert_allclose(forward(pr, q, k, v)[0], to.numpy(), rtol=1e-12, atol=1e-13)


def test_packed_alibi_takes_each_sequence_row():
    lq, lk = [4, 6], [5, 6]
    slopes = ((0.3, 0.1), (0.05, 0.9))
    sq = (0, 4, 10)
    sk = (0, 5, 11)
    pk = varlen.Packed(sq, sk, 2, 4, 3, 0.5, True, alibi_slopes=slopes)
    q, k, v = rand(2, 10, 4), rand(2, 11, 4), rand(2, 11, 3)
    o, _ = varlen.forward(pk, q, k, v)
    for i in range(2):
        pr = Problem(1, 2, lq[i], lk[i], 4, 3, 0.5, True, alibi_slopes=(slopes[i],))
        o_i, _ = forward(pr, q[:, sq[i]:sq[i + 1]][None], k[:, sk[i]:sk[i + 1]][None],
                         v[:, sk[i]:sk[i + 1]][None])
        np.testing.assert_array_equal(o[:, sq[i]:sq[i + 1]], o_i[0])
