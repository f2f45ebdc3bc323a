"""Pins of the packed-sequence oracle (oracle.varlen) to facts outside it.

* PyTorch's float64 scaled_dot_product_attention and autograd, called once
  over all packed rows with a block-diagonal mask (a key is visible only to
  queries of its own sequence, causal top-left within the sequence): an
  independent implementation of the per-sequence rule, so a leak across
  sequences or a causal mask taken on packed instead of local indices fails.
* With dropout (which torch cannot reproduce): the batch-mode oracle on the
  sequences zero-padded to the longest lengths, with a -inf bias on the padded
  keys, gives the same result on the real rows. That is the reading of the
  dropout bits (sequence i draws batch entry i of the padded problem) stated
  through a different path of the oracle (bias and padding, not slicing).
* Empty sequences: the values the reading fixes (O = 0, LSE = -inf, zero
  gradients) and no effect on the other sequences.
"""
import numpy as np
import pytest
import torch

from oracle import Problem, backward, forward, varlen

RNG = np.random.default_rng(77)


def rand(*shape):
    return RNG.standard_normal(shape)


def starts(lens):
    return tuple(int(x) for x in np.concatenate([[0], np.cumsum(lens)]))


def packed_tensors(pk):
    tq, tk = pk.seqstart_q[-1], pk.seqstart_k[-1]
    return (rand(pk.H, tq, pk.D_qk), rand(pk.kv_heads, tk, pk.D_qk), rand(pk.kv_heads, tk, pk.D_v),
            rand(pk.H, tq, pk.D_v))


def block_mask(pk):
    """Additive [total_q, total_k] mask: 0 where visible, -inf elsewhere."""
    tq, tk = pk.seqstart_q[-1], pk.seqstart_k[-1]
    m = np.full((tq, tk), -np.inf)
    for i in range(pk.B):
        qa, qb = pk.seqstart_q[i], pk.seqstart_q[i + 1]
        ka, kb = pk.seqstart_k[i], pk.seqstart_k[i + 1]
        vis = np.ones((qb - qa, kb - ka), dtype=bool)
        if pk.is_causal:
            vis = np.tril(vis)
        m[qa:qb, ka:kb] = np.where(vis, 0.0, -np.inf)
    return torch.tensor(m)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("H,H_kv,lq,lk", [
    (2, 2, [5, 1, 9, 4], [5, 1, 9, 4]),     # self-attention lengths
    (4, 2, [3, 7, 6], [8, 2, 11]),         # cross lengths, grouped K/V heads
    (3, 1, [6, 6], [4, 9]),                # one K/V head
])
def test_packed_matches_torch_block_diagonal(causal, H, H_kv, lq, lk):
    pk = varlen.Packed(starts(lq), starts(lk), H, 4, 3, 0.7, causal, H_kv=H_kv)
    q, k, v, do = packed_tensors(pk)
    tq, tk_, tv = (torch.tensor(a, requires_grad=True) for a in (q, k, v))
    mask = block_mask(pk)
    to = torch.nn.functional.scaled_dot_product_attention(tq[None], tk_[None], tv[None],
                                                          attn_mask=mask, scale=pk.scale,
                                                          enable_gqa=True)[0]
    to.backward(torch.tensor(do))
    o, lse = varlen.forward(pk, q, k, v)
    np.testing.assert_allclose(o, to.detach().numpy(), rtol=1e-12, atol=1e-13)
    # LSE: torch's logsumexp over the same masked scores
    kr = np.repeat(k, H // H_kv, axis=0)
    s = pk.scale * torch.einsum("hqd,hkd->hqk", torch.tensor(q), torch.tensor(kr)) + mask
    np.testing.assert_allclose(lse, torch.logsumexp(s, dim=-1).numpy(), rtol=1e-12, atol=1e-12)
    dq, dk, dv = varlen.backward(pk, q, k, v, do)
    np.testing.assert_allclose(dq, tq.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dk, tk_.grad.numpy(), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad.numpy(), rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_dropout_equals_padded_batch(causal):
    """Sequences zero-padded to (max_q, max_k) in batch mode with a -inf bias on
    the padded keys: same O, LSE, dQ, dK, dV on the real rows, dropout bits
    included (padded query rows carry dO = 0, so they add nothing to dK, dV)."""
    H, lq, lk = 2, [5, 3, 8], [6, 8, 4]
    mq, mk = 9, 8  # at least the longest lengths, max_k a multiple of 4
    pk = varlen.Packed(starts(lq), starts(lk), H, 4, 3, 0.6, causal, 0.3, 21, 4,
                       max_seqlen_q=mq, max_seqlen_k=mk)
    q, k, v, do = packed_tensors(pk)
    B = pk.B
    qp, dop = np.zeros((B, H, mq, 4)), np.zeros((B, H, mq, 3))
    kp, vp = np.zeros((B, H, mk, 4)), np.zeros((B, H, mk, 3))
    for i in range(B):
        qa, ka = pk.seqstart_q[i], pk.seqstart_k[i]
        qp[i, :, :lq[i]], dop[i, :, :lq[i]] = q[:, qa:qa + lq[i]], do[:, qa:qa + lq[i]]
        kp[i, :, :lk[i]], vp[i, :, :lk[i]] = k[:, ka:ka + lk[i]], v[:, ka:ka + lk[i]]
    o, lse = varlen.forward(pk, q, k, v)
    dq, dk, dv = varlen.backward(pk, q, k, v, do)
    pr = Problem(B, H, mq, mk, 4, 3, 0.6, causal, 0.3, 21, 4)
    for i in range(B):
        # the bias is shared by the batch entries, so each entry is checked with
        # a bias that masks its own padded keys
        bias = np.zeros((1, H, mq, mk))
        bias[..., lk[i]:] = -np.inf
        o_p, lse_p = forward(pr, qp, kp, vp, bias)
        dq_p, dk_p, dv_p, _ = backward(pr, qp, kp, vp, dop, bias)
        qa, ka = pk.seqstart_q[i], pk.seqstart_k[i]
        rq, rk = slice(qa, qa + lq[i]), slice(ka, ka + lk[i])
        np.testing.assert_allclose(o[:, rq], o_p[i, :, :lq[i]], rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse[:, rq], lse_p[i, :, :lq[i]], rtol=1e-12)
        np.testing.assert_allclose(dq[:, rq], dq_p[i, :, :lq[i]], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dk[:, rk], dk_p[i, :, :lk[i]], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(dv[:, rk], dv_p[i, :, :lk[i]], rtol=1e-11, atol=1e-12)


def test_uniform_lengths_equal_batch_mode_with_dropout():
    """Equal lengths and max lengths: the packed problem is the batch problem
    with the batch moved into the rows, dropout bits and all."""
    B, H, S, D = 3, 2, 8, 4
    pk = varlen.Packed(starts([S] * B), starts([S] * B), H, D, D, 0.5, True, 0.25, 9, 2)
    q, k, v, do = packed_tensors(pk)
    to_b = lambda x: x.reshape(x.shape[0], B, S, x.shape[-1]).transpose(1, 0, 2, 3)
    pr = Problem(B, H, S, S, D, D, 0.5, True, 0.25, 9, 2)
    o_b, lse_b = forward(pr, to_b(q), to_b(k), to_b(v))
    dq_b, dk_b, dv_b, _ = backward(pr, to_b(q), to_b(k), to_b(v), to_b(do))
    o, lse = varlen.forward(pk, q, k, v)
    dq, dk, dv = varlen.backward(pk, q, k, v, do)
    np.testing.assert_array_equal(to_b(o), o_b)
    np.testing.assert_array_equal(lse.reshape(H, B, S).transpose(1, 0, 2), lse_b)
    np.testing.assert_array_equal(to_b(dq), dq_b)
    np.testing.assert_array_equal(to_b(dk), dk_b)
    np.testing.assert_array_equal(to_b(dv), dv_b)


def test_empty_sequences():
    """A sequence without keys: O = 0, LSE = -inf, dQ = 0; without queries:
    dK = dV = 0; the other sequences are those of the call without them."""
    lq, lk = [4, 3, 0, 5], [6, 0, 2, 7]
    pk = varlen.Packed(starts(lq), starts(lk), 2, 4, 3, 0.5, True)
    q, k, v, do = packed_tensors(pk)
    o, lse = varlen.forward(pk, q, k, v)
    dq, dk, dv = varlen.backward(pk, q, k, v, do)
    np.testing.assert_array_equal(o[:, 4:7], 0.0)
    assert np.all(np.isneginf(lse[:, 4:7]))
    np.testing.assert_array_equal(dq[:, 4:7], 0.0)
    np.testing.assert_array_equal(dk[:, 6:8], 0.0)
    np.testing.assert_array_equal(dv[:, 6:8], 0.0)
    # sequences 0 and 3 alone
    keep_q = np.r_[0:4, 7:12]
    keep_k = np.r_[0:6, 8:15]
    pk2 = varlen.Packed(starts([4, 5]), starts([6, 7]), 2, 4, 3, 0.5, True)
    o2, lse2 = varlen.forward(pk2, q[:, keep_q], k[:, keep_k], v[:, keep_k])
    dq2, dk2, dv2 = varlen.backward(pk2, q[:, keep_q], k[:, keep_k], v[:, keep_k], do[:, keep_q])
    np.testing.assert_array_equal(o[:, keep_q], o2)
    np.testing.assert_array_equal(lse[:, keep_q], lse2)
    np.testing.assert_array_equal(dq[:, keep_q], dq2)
    np.testing.assert_array_equal(dk[:, keep_k], dk2)
    np.testing.assert_array_equal(dv[:, keep_k], dv2)
