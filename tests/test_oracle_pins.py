"""Pins of the fp64 oracle to facts that do not come from the oracle itself.

Closed forms, invariants of the softmax Jacobian, central finite differences of
loss = <dO, O>, PyTorch's own float64 attention and autograd as an independent
library routine, and statistics of the dropout mask. Each test is chosen so
that a plausible slip in the oracle (a dropped scale, a transposed operand, a
wrong sign in dS, a missing 1/(1-p), log2 instead of ln) fails at least one.
"""
import math

import numpy as np
import pytest
import torch

from oracle import Problem, backward, backward_head, forward, forward_head, philox

RNG = np.random.default_rng(1234)


def rand(*shape, scale=1.0):
    return RNG.standard_normal(shape) * scale


def problem(B=1, H=1, S_q=5, S_kv=7, D_qk=4, D_v=3, scale=0.5, causal=False, p=0.0,
            seed=11, offset=3):
    return Problem(B, H, S_q, S_kv, D_qk, D_v, scale, causal, p, seed, offset)


def tensors(pr, bias=False):
    q = rand(pr.B, pr.H, pr.S_q, pr.D_qk)
    k = rand(pr.B, pr.H, pr.S_kv, pr.D_qk)
    v = rand(pr.B, pr.H, pr.S_kv, pr.D_v)
    do = rand(pr.B, pr.H, pr.S_q, pr.D_v)
    b = rand(1, pr.H, pr.S_q, pr.S_kv, scale=0.5) if bias else None
    return q, k, v, do, b


# ------------------------------------------------------------------ closed forms
@pytest.mark.parametrize("p", [0.0, 0.3])
def test_single_key_returns_v(p):
    pr = problem(S_q=6, S_kv=1, p=p)
    q, k, v, _, bias = tensors(pr, bias=True)
    o, lse = forward(pr, q, k, v, bias)
    keep = philox.keep_mask(1, 1, 6, 1, p, pr.seed, pr.offset, 0, 0)
    z = keep[:, 0] / (1 - p)
    np.testing.assert_allclose(o[0, 0], z[:, None] * v[0, 0, 0][None, :], rtol=1e-13, atol=1e-13)
    # one visible key: the logsumexp is that key's score
    s0 = pr.scale * q[0, 0] @ k[0, 0, 0] + bias[0, 0, :, 0]
    np.testing.assert_allclose(lse[0, 0], s0, rtol=1e-13)


def test_identity_values_expose_probabilities():
    # with V = I the output rows are the softmax rows themselves
    for causal in (False, True):
        pr = problem(S_q=6, S_kv=6, D_v=6, causal=causal)
        q, k, _, _, bias = tensors(pr, bias=True)
        v = np.eye(6)[None, None]
        o, _ = forward(pr, q, k, v, bias)
        P = o[0, 0]
        assert (P >= 0).all()
        np.testing.assert_allclose(P.sum(axis=1), 1.0, rtol=1e-14)
        if causal:
            assert np.all(P[np.triu_indices(6, 1)] == 0.0)


def test_first_causal_row_is_first_value():
    pr = problem(S_q=8, S_kv=8, causal=True)
    q, k, v, _, bias = tensors(pr, bias=True)
    o, lse = forward(pr, q, k, v, bias)
    np.testing.assert_allclose(o[0, 0, 0], v[0, 0, 0], rtol=1e-14)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_queries_average_visible_values(causal):
    pr = problem(S_q=7, S_kv=7, causal=causal, scale=0.7)
    _, k, v, _, _ = tensors(pr)
    q = np.zeros((1, 1, 7, pr.D_qk))
    o, lse = forward(pr, q, k, v)
    for i in range(7):
        n = i + 1 if causal else 7
        assert lse[0, 0, i] == pytest.approx(math.log(n), rel=1e-14)  # natural log
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n].mean(axis=0), rtol=1e-13, atol=1e-15)


@pytest.mark.parametrize("causal", [False, True])
def test_zero_scale_averages_visible_values(causal):
    """scale = 0 with nonzero queries: every visible key weighs 1/n, so
    O_i is the mean of the visible V rows, LSE_i = ln n, dQ = dK = 0 (both
    carry the factor scale) and dV_j sums dO_i / n_i over the rows i that
    see key j."""
    pr = problem(S_q=6, S_kv=9, causal=causal, scale=0.0)
    q, k, v, do, _ = tensors(pr)
    o, lse = forward(pr, q, k, v)
    dq, dk, dv, _ = backward(pr, q, k, v, do)
    n = [min(i + 1, 9) if causal else 9 for i in range(6)]
    for i in range(6):
        assert lse[0, 0, i] == pytest.approx(math.log(n[i]), rel=1e-14)
        np.testing.assert_allclose(o[0, 0, i], v[0, 0, :n[i]].mean(axis=0), rtol=1e-13, atol=1e-15)
    assert np.all(dq == 0.0) and np.all(dk == 0.0)
    want = np.zeros((9, pr.D_v))
    for i in range(6):
        want[:n[i]] += do[0, 0, i] / n[i]
    np.testing.assert_allclose(dv[0, 0], want, rtol=1e-13, atol=1e-15)


def test_fully_masked_row_is_zero():
    pr = problem(S_q=4, S_kv=5)
    q, k, v, do, bias = tensors(pr, bias=True)
    bias[0, 0, 2, :] = -np.inf
    o, lse = forward(pr, q, k, v, bias)
    assert lse[0, 0, 2] == -np.inf and np.all(o[0, 0, 2] == 0.0)
    dq, dk, dv, dbias = backward(pr, q, k, v, do, bias)
    assert np.all(dq[0, 0, 2] == 0.0) and np.all(dbias[0, 0, 2] == 0.0)


def test_zero_output_gradient_gives_zero_gradients():
    pr = problem(B=2, H=2, causal=True, p=0.2)
    q, k, v, _, bias = tensors(pr, bias=True)
    do = np.zeros((2, 2, pr.S_q, pr.D_v))
    for g in backward(pr, q, k, v, do, bias):
        assert np.all(g == 0.0)


# ------------------------------------------------------------------ invariants
@pytest.mark.parametrize("causal", [False, True])
def test_softmax_jacobian_invariants(causal):
    pr = problem(B=2, H=2, S_q=6, S_kv=9, causal=causal)
    q, k, v, do, bias = tensors(pr, bias=True)
    dq, dk, dv, dbias = backward(pr, q, k, v, do, bias)
    # each row of dS sums to zero, so do the rows of dBias and the key-sum of dK
    np.testing.assert_allclose(dbias.sum(axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(dk.sum(axis=2), 0.0, atol=1e-12)
    # P rows sum to one, so the key-sum of dV is the query-sum of dO
    np.testing.assert_allclose(dv.sum(axis=2), do.sum(axis=2), rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ finite differences
def loss(pr, q, k, v, do, bias):
    o, _ = forward(pr, q, k, v, bias)
    return float((o * do).sum())


@pytest.mark.parametrize("shape,causal,p,use_bias", [
    ((1, 1, 5, 7, 4, 3), False, 0.0, True),
    ((1, 1, 5, 7, 4, 3), True, 0.0, False),
    ((1, 2, 8, 8, 4, 4), True, 0.0, True),
    ((1, 2, 8, 8, 4, 4), False, 0.25, True),
    ((2, 1, 6, 4, 3, 5), True, 0.4, False),
])
def test_central_finite_differences(shape, causal, p, use_bias):
    B, H, S_q, S_kv, D_qk, D_v = shape
    pr = Problem(B, H, S_q, S_kv, D_qk, D_v, 0.6, causal, p, 77, 5)
    q, k, v, do, bias = tensors(pr, bias=use_bias)
    dq, dk, dv, dbias = backward(pr, q, k, v, do, bias)
    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv), ("bias", bias, dbias)):
        if x is None:
            continue
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            x0 = x[idx]
            x[idx] = x0 + eps
            lp = loss(pr, q, k, v, do, bias)
            x[idx] = x0 - eps
            lm = loss(pr, q, k, v, do, bias)
            x[idx] = x0
            num[idx] = (lp - lm) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-6, atol=1e-8, err_msg=name)


# ------------------------------------------------------------------ library cross-check
@pytest.mark.parametrize("causal,use_bias", [(False, False), (True, False), (False, True),
                                             (True, True)])
def test_matches_torch_float64_attention_and_autograd(causal, use_bias):
    """PyTorch's CPU scaled_dot_product_attention in float64 is an independent
    implementation of the same definition when dropout is off."""
    pr = problem(B=2, H=3, S_q=9, S_kv=13, D_qk=8, D_v=6, scale=0.3, causal=causal)
    q, k, v, do, bias = tensors(pr, bias=use_bias)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = None
    if use_bias or causal:
        m = torch.zeros(pr.S_q, pr.S_kv, dtype=torch.float64)
        if causal:
            m = m.masked_fill(torch.ones(pr.S_q, pr.S_kv, dtype=torch.bool).triu(1), float("-inf"))
        tb = torch.tensor(bias, requires_grad=True) if use_bias else None
        mask = m + (tb if use_bias else 0)
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                          scale=pr.scale)
    to.backward(torch.tensor(do))
    o, lse = forward(pr, q, k, v, bias)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    s = torch.tensor(q) @ torch.tensor(k).transpose(-1, -2) * pr.scale
    if mask is not None:
        s = s + mask.detach()
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-13)
    dq, dk, dv, dbias = backward(pr, q, k, v, do, bias)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)
    if use_bias:
        np.testing.assert_allclose(dbias, tb.grad.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_negative_scale_matches_torch_float64(causal):
    """A negative scale (the softmax then favours the smallest products):
    PyTorch's float64 attention with the same scale, and autograd."""
    pr = problem(B=1, H=2, S_q=7, S_kv=10, D_qk=5, D_v=4, scale=-0.4, causal=causal)
    q, k, v, do, _ = tensors(pr)
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal,
                                                          scale=pr.scale)
    to.backward(torch.tensor(do))
    o, _ = forward(pr, q, k, v)
    dq, dk, dv, _ = backward(pr, q, k, v, do)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


# ------------------------------------------------------------------ sampled slices
def test_row_and_column_sampling_agree_with_full():
    pr = problem(B=2, H=2, S_q=33, S_kv=40, D_qk=8, D_v=4, causal=True, p=0.15)
    q, k, v, do, bias = tensors(pr, bias=True)
    o, lse = forward(pr, q, k, v, bias)
    dq, dk, dv, _ = backward(pr, q, k, v, do, bias)
    rows = np.array([0, 5, 17, 32])
    cols = np.array([1, 2, 30, 39])
    o_r, lse_r = forward_head(pr, 1, 1, q, k, v, bias, rows=rows)
    np.testing.assert_allclose(o_r, o[1, 1, rows], rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(lse_r, lse[1, 1, rows], rtol=1e-13)
    dq_r, dk_c, dv_c, _ = backward_head(pr, 1, 1, q, k, v, do, bias, rows=rows, cols=cols,
                                        row_chunk=7)
    np.testing.assert_allclose(dq_r, dq[1, 1, rows], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dk_c, dk[1, 1, cols], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dv_c, dv[1, 1, cols], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ dropout statistics
def test_dropout_is_unbiased():
    """Averaged over seeds, the dropout output converges to the dropout-free
    output: checks the 1/(1-p) rescale and that the row sums are pre-dropout."""
    pr0 = problem(S_q=4, S_kv=6, D_v=2, p=0.0)
    q, k, v, _, _ = tensors(pr0)
    o_ref, lse_ref = forward(pr0, q, k, v)
    n = 600
    acc = np.zeros_like(o_ref)
    for s in range(n):
        pr = Problem(1, 1, 4, 6, 4, 2, pr0.scale, False, 0.3, seed=1000 + s, offset=0)
        o, lse = forward(pr, q, k, v)
        np.testing.assert_array_equal(lse, lse_ref)
        acc += o
    mean = acc / n
    # per-element std of one draw is at most sqrt(p/(1-p)) * sqrt(sum P^2 v^2) <= ~0.65*max|v|
    tol = 5 * math.sqrt(0.3 / 0.7) * np.abs(v).max() / math.sqrt(n)
    assert np.abs(mean - o_ref).max() < tol


def test_keep_fraction_binomial():
    p = 0.1
    keep = philox.keep_mask(2, 2, 64, 256, p, 0x1234, 0, 1, 1)
    n = keep.size
    frac = keep.mean()
    assert abs(frac - (1 - p)) < 5 * math.sqrt(p * (1 - p) / n)


def test_drop_threshold_values():
    assert philox.drop_threshold(0.0) == 0
    assert philox.drop_threshold(0.1) == 429496729
    assert philox.drop_threshold(0.5) == 2 ** 31
    with pytest.raises(ValueError):
        philox.drop_threshold(1.0)


def test_packed_words_match_mask():
    B, H, S_q, S_kv, p = 1, 2, 3, 12, 0.4
    words = philox.packed_mask_words(B, H, S_q, S_kv, p, 99, 7)
    bits = np.unpackbits(words.view(np.uint8), bitorder="little")[: B * H * S_q * S_kv]
    full = np.stack([philox.keep_mask(B, H, S_q, S_kv, p, 99, 7, 0, h) for h in range(H)])
    np.testing.assert_array_equal(bits.astype(bool), full.reshape(-1))


# ------------------------------------------------------------------ grouped K/V heads
def _gqa_problem(H, H_kv, causal, p=0.0):
    return Problem(2, H, 9, 13, 8, 6, 0.3, causal, p, 7, 5, H_kv)


@pytest.mark.parametrize("H,H_kv,causal,use_bias", [(4, 2, False, False), (6, 2, True, True),
                                                    (4, 1, True, False)])
def test_grouped_heads_match_torch_enable_gqa(H, H_kv, causal, use_bias):
    """PyTorch's CPU scaled_dot_product_attention with enable_gqa (float64) is an
    independent implementation of the grouped-head mapping: forward, LSE and
    autograd gradients (dK, dV summed over each group by autograd)."""
    pr = _gqa_problem(H, H_kv, causal)
    q, do = rand(pr.B, H, pr.S_q, pr.D_qk), rand(pr.B, H, pr.S_q, pr.D_v)
    k, v = rand(pr.B, H_kv, pr.S_kv, pr.D_qk), rand(pr.B, H_kv, pr.S_kv, pr.D_v)
    bias = rand(1, H, pr.S_q, pr.S_kv, scale=0.5) if use_bias else None
    tq, tk, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = None
    if use_bias or causal:
        m = torch.zeros(pr.S_q, pr.S_kv, dtype=torch.float64)
        if causal:
            m = m.masked_fill(torch.ones(pr.S_q, pr.S_kv, dtype=torch.bool).triu(1), float("-inf"))
        tb = torch.tensor(bias, requires_grad=True) if use_bias else None
        mask = m + (tb if use_bias else 0)
    to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                          scale=pr.scale, enable_gqa=True)
    to.backward(torch.tensor(do))
    o, lse = forward(pr, q, k, v, bias)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    dq, dk, dv, dbias = backward(pr, q, k, v, do, bias)
    assert dk.shape == k.shape and dv.shape == v.shape
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)
    if use_bias:
        np.testing.assert_allclose(dbias, tb.grad.numpy(), rtol=1e-11, atol=1e-12)


def test_grouped_heads_equal_repeated_kv_with_dropout():
    """With dropout (which torch cannot reproduce), grouped heads equal the
    ungrouped problem on K/V repeated over each group, with dK / dV summed over
    the group: the dropout bits depend on the query head only."""
    H, H_kv = 6, 3
    g = H // H_kv
    pr = _gqa_problem(H, H_kv, True, p=0.25)
    full = Problem(pr.B, H, pr.S_q, pr.S_kv, pr.D_qk, pr.D_v, pr.scale, True, 0.25, 7, 5)
    q, do = rand(pr.B, H, pr.S_q, pr.D_qk), rand(pr.B, H, pr.S_q, pr.D_v)
    k, v = rand(pr.B, H_kv, pr.S_kv, pr.D_qk), rand(pr.B, H_kv, pr.S_kv, pr.D_v)
    kr, vr = np.repeat(k, g, axis=1), np.repeat(v, g, axis=1)
    o, lse = forward(pr, q, k, v)
    o_f, lse_f = forward(full, q, kr, vr)
    np.testing.assert_array_equal(o, o_f)
    np.testing.assert_array_equal(lse, lse_f)
    dq, dk, dv, _ = backward(pr, q, k, v, do)
    dq_f, dk_f, dv_f, _ = backward(full, q, kr, vr, do)
    np.testing.assert_array_equal(dq, dq_f)
    np.testing.assert_allclose(dk, dk_f.reshape(pr.B, H_kv, g, pr.S_kv, pr.D_qk).sum(axis=2), rtol=1e-13, atol=1e-14)
    np.testing.assert_allclose(dv, dv_f.reshape(pr.B, H_kv, g, pr.S_kv, pr.D_v).sum(axis=2), rtol=1e-13, atol=1e-14)
