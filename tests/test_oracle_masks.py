"""Pins of the oracle's mask variants (local windows, bottom-right alignment)
to facts outside it.

* Bottom-right causal: PyTorch's own lower-right causal bias
  (torch.nn.attention.bias.causal_lower_right) with its float64 attention and
  autograd.
* Windows: the band numpy's triu / tril draw with their diagonal offsets
  (the diagonal through (0, off), off = S_kv - S_q for bottom-right), used as
  a boolean mask of PyTorch's float64 attention and autograd.
* Locality: with a window, V rows outside row i's window cannot change O_i,
  and the ones inside do.
* Special cases: window (-1, 0) is causal; windows wider than the problem are
  no mask; bottom-right equals top-left when S_q = S_kv.
"""
import numpy as np
import pytest
import torch
from torch.nn.attention.bias import causal_lower_right

from oracle import Problem, backward, forward, varlen

RNG = np.random.default_rng(4321)


def rand(*shape):
    return RNG.standard_normal(shape)


def tensors(pr):
    return (rand(pr.B, pr.H, pr.S_q, pr.D_qk), rand(pr.B, pr.kv_heads, pr.S_kv, pr.D_qk),
            rand(pr.B, pr.kv_heads, pr.S_kv, pr.D_v), rand(pr.B, pr.H, pr.S_q, pr.D_v))


def torch_reference(pr, q, k, v, do, mask):
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask, scale=pr.scale,
                                                         enable_gqa=True)
    o.backward(torch.tensor(do))
    return o.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


def assert_matches(pr, q, k, v, do, mask):
    o_t, dq_t, dk_t, dv_t = torch_reference(pr, q, k, v, do, mask)
    o, _ = forward(pr, q, k, v)
    dq, dk, dv, _ = backward(pr, q, k, v, do)
    np.testing.assert_allclose(o, o_t, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, dq_t, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, dk_t, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, dv_t, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("S_q,S_kv", [(5, 9), (7, 7), (1, 6)])
def test_bottom_right_causal_matches_torch_lower_right(S_q, S_kv):
    pr = Problem(2, 2, S_q, S_kv, 4, 3, 0.6, True, bottom_right=True)
    q, k, v, do = tensors(pr)
    assert_matches(pr, q, k, v, do, causal_lower_right(S_q, S_kv))


def band(S_q, S_kv, left, right, bottom_right):
    """Boolean band from numpy's triu / tril offsets (True = visible)."""
    off = S_kv - S_q if bottom_right else 0
    m = np.ones((S_q, S_kv), dtype=bool)
    if left >= 0:
        m = np.triu(m, k=off - left)
    if right >= 0:
        m = np.tril(m, k=off + right)
    return torch.tensor(m)


@pytest.mark.parametrize("S_q,S_kv,left,right,br,H_kv", [
    (9, 9, 3, 0, False, 2),     # sliding window, causal side
    (8, 12, 2, 1, True, 2),     # both sides, bottom-right
    (10, 7, -1, 2, False, 1),   # unbounded left, two keys right
    (6, 11, 4, -1, True, 2),    # unbounded right
    (12, 12, 0, 0, False, 2),   # the diagonal alone
])
def test_window_matches_torch_with_numpy_band(S_q, S_kv, left, right, br, H_kv):
    pr = Problem(2, 2, S_q, S_kv, 4, 3, 0.45, False, H_kv=H_kv, window=(left, right),
                 bottom_right=br)
    q, k, v, do = tensors(pr)
    mask = band(S_q, S_kv, left, right, br)
    assert bool(mask.any(dim=1).all()), "torch gives NaN on rows without keys: pick sizes without"
    assert_matches(pr, q, k, v, do, mask)


def test_window_locality():
    pr = Problem(1, 1, 16, 16, 4, 3, 0.5, False, window=(3, 1))
    q, k, v, _ = tensors(pr)
    o, _ = forward(pr, q, k, v)
    i = 9  # window: keys 6 .. 10
    v_out = v.copy()
    v_out[0, 0, [0, 5, 11, 15]] += 10.0
    o_out, _ = forward(pr, q, k, v_out)
    np.testing.assert_array_equal(o_out[0, 0, i], o[0, 0, i])
    v_in = v.copy()
    v_in[0, 0, 6] += 10.0
    o_in, _ = forward(pr, q, k, v_in)
    assert np.abs(o_in[0, 0, i] - o[0, 0, i]).max() > 1e-3


def test_special_cases():
    base = dict(B=1, H=2, S_q=7, S_kv=10, D_qk=4, D_v=3, scale=0.5)
    pr_c = Problem(**base, is_causal=True)
    q, k, v, do = tensors(pr_c)
    same = [(Problem(**base, is_causal=False, window=(-1, 0)), pr_c),
            (Problem(**base, window=(20, 20)), Problem(**base)),
            (Problem(**base, window=(-1, -1), bottom_right=True), Problem(**base))]
    for a, b in same:
        np.testing.assert_array_equal(forward(a, q, k, v)[0], forward(b, q, k, v)[0])
        np.testing.assert_array_equal(backward(a, q, k, v, do)[1], backward(b, q, k, v, do)[1])
    sq = dict(base, S_kv=7)
    pr_a = Problem(**sq, is_causal=True, window=(2, 0))
    pr_b = Problem(**sq, is_causal=True, window=(2, 0), bottom_right=True)
    q, k, v, do = tensors(pr_a)
    np.testing.assert_array_equal(forward(pr_a, q, k, v)[0], forward(pr_b, q, k, v)[0])


def test_rows_without_keys_bottom_right():
    """Bottom-right causal with S_q > S_kv: the first S_q - S_kv rows see no
    key: O = 0, LSE = -inf, no gradient (the rule for a row without keys)."""
    pr = Problem(1, 2, 9, 5, 4, 3, 0.5, True, bottom_right=True)
    q, k, v, do = tensors(pr)
    o, lse = forward(pr, q, k, v)
    dq, _, _, _ = backward(pr, q, k, v, do)
    np.testing.assert_array_equal(o[:, :, :4], 0.0)
    assert np.all(np.isneginf(lse[:, :, :4]))
    np.testing.assert_array_equal(dq[:, :, :4], 0.0)
    # the remaining rows are PyTorch's lower-right causal attention
    o_t, dq_t, dk_t, dv_t = torch_reference(
        Problem(1, 2, 5, 5, 4, 3, 0.5, True), q[:, :, 4:], k, v, do[:, :, 4:],
        causal_lower_right(5, 5))
    np.testing.assert_allclose(o[:, :, 4:], o_t, rtol=1e-12, atol=1e-13)
    _, dk, dv, _ = backward(pr, q, k, v, do)
    np.testing.assert_allclose(dk, dk_t, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, dv_t, rtol=1e-11, atol=1e-12)


def test_packed_window_bottom_right_matches_torch_blocks():
    """Packed sequences with a bottom-right window: each sequence's block of the
    mask is its own numpy band (lengths of the sequence, not of the packing)."""
    lq, lk = [5, 3, 8], [9, 6, 8]
    sq = tuple(np.concatenate([[0], np.cumsum(lq)]).tolist())
    sk = tuple(np.concatenate([[0], np.cumsum(lk)]).tolist())
    pk = varlen.Packed(sq, sk, 2, 4, 3, 0.5, False, window=(2, 1), bottom_right=True)
    q, k = rand(2, sq[-1], 4), rand(2, sk[-1], 4)
    v, do = rand(2, sk[-1], 3), rand(2, sq[-1], 3)
    m = torch.zeros(sq[-1], sk[-1], dtype=torch.bool)
    for i in range(3):
        m[sq[i]:sq[i + 1], sk[i]:sk[i + 1]] = band(lq[i], lk[i], 2, 1, True)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq[None], tk[None], tv[None], attn_mask=m,
                                                          scale=0.5)[0]
    to.backward(torch.tensor(do))
    o, _ = varlen.forward(pk, q, k, v)
    dq, dk, dv = varlen.backward(pk, q, k, v, do)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)
