"""GPU parity at the five workloads' full sizes, in the launch configuration
bench.py times (whole-problem sdpa_fwd + sdpa_bwd calls).

The oracle cannot materialise every head at these sizes in seconds, so each
check compares sampled outputs it computes one by one (whole (b, h) slices,
or sampled query rows and key columns of one head), plus invariants that hold
at any size: with no dropout every row of dS sums to zero, so the key-sum of
dK vanishes and the key-sum of dV equals the query-sum of dO.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import philox
from parity_util import Case, assert_close, assert_lse, run_gpu
from scaled_dot_product_06_gb300 import sdpa_dropout_mask
from scaled_dot_product_06_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


def slice_check(case, x, outs, b, h):
    o, lse, dq, dk, dv, _ = outs
    pr = case.problem()
    o_ref, lse_ref = oracle.forward_head(pr, b, h, x["q"], x["k"], x["v"], x["bias"])
    assert_close(f"o[{b},{h}]", o[b, h], o_ref)
    assert_lse(lse[b, h], lse_ref)
    dq_r, dk_r, dv_r, ds = oracle.backward_head(pr, b, h, x["q"], x["k"], x["v"], x["do"],
                                                x["bias"])
    assert_close(f"dq[{b},{h}]", dq[b, h], dq_r)
    assert_close(f"dk[{b},{h}]", dk[b, h], dk_r)
    assert_close(f"dv[{b},{h}]", dv[b, h], dv_r)
    return ds


def key_sum_invariants(case, outs, x):
    """No dropout: sum over keys of dK is 0 and of dV equals sum over queries of dO."""
    _, _, _, dk, dv, _ = outs
    dk64 = dk.double()
    rel = dk64.sum(dim=2).abs().max().item() / dk64.abs().sum(dim=2).max().item()
    assert rel < 2e-2, f"key-sum of dK is not ~0 (relative {rel:.3e})"
    dv_sum = dv.double().sum(dim=2).cpu().numpy()
    do_sum = x["do"].double().sum(dim=2).numpy()
    assert_close("sum_j dV", torch.from_numpy(dv_sum), do_sum, rel=3e-2)


def test_small_configuration_every_element():
    from parity_util import check_full
    check_full(Case(1, 2, 128, 128, 64, 64, scale=0.125))


def test_b4h16_s2048_d128_causal():
    case = Case(4, 16, 2048, 2048, 128, 128, causal=True)
    x = make_inputs(case.shape, case.dtype)
    outs = run_gpu(case, x)
    for b, h in ((0, 0), (3, 15), (2, 7)):
        slice_check(case, x, outs, b, h)
    key_sum_invariants(case, outs, x)


def test_b2h16_s4096_d192x128_causal_bias():
    case = Case(2, 16, 4096, 4096, 192, 128, causal=True, bias=True)
    x = make_inputs(case.shape, case.dtype, with_bias=True)
    outs = run_gpu(case, x)
    dbias = outs[5]
    for h in (0, 11):  # dBias sums over the batch, so sample whole heads
        ds_sum = 0.0
        for b in range(case.B):
            ds_sum = ds_sum + slice_check(case, x, outs, b, h)
        assert_close(f"dbias[{h}]", dbias[0, h], ds_sum)
    key_sum_invariants(case, outs, x)


def same_bits_with_keep_bits(case, x, outs):
    """The kernels' own Philox draws at this size give exactly the bits of
    sdpa_dropout_mask: the forward and backward run again with the mask passed
    in (the kernels then read it) and must agree bit for bit (O, LSE, dK, dV;
    dQ in the deterministic backward, whose sums have a fixed order)."""
    from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_fwd
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    kw = dict(scale=case.sc, is_causal=case.causal, dropout_p=case.p, seed=case.seed,
              offset=case.offset)
    mask = sdpa_dropout_mask(case.B, case.H, case.S_q, case.S_kv, case.p, case.seed, case.offset)
    o, lse = sdpa_fwd(q, k, v, dropout_mask=mask, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o, outs[0]) and torch.equal(lse, outs[1])
    _, dk, dv, _ = sdpa_bwd(q, k, v, o, do, lse, dropout_mask=mask, **kw)
    torch.cuda.synchronize()
    assert torch.equal(dk, outs[3]) and torch.equal(dv, outs[4])
    del dk, dv
    det_a = sdpa_bwd(q, k, v, o, do, lse, deterministic=True, **kw)
    det_b = sdpa_bwd(q, k, v, o, do, lse, dropout_mask=mask, deterministic=True, **kw)
    torch.cuda.synchronize()
    for a, b in zip(det_a[:3], det_b[:3]):
        assert torch.equal(a, b)


def test_b8h16_s1024x2048_d64_fp16_dropout():
    case = Case(8, 16, 1024, 2048, 64, 64, dtype="fp16", p=0.1)
    x = make_inputs(case.shape, case.dtype)
    outs = run_gpu(case, x)
    for b, h in ((0, 0), (7, 15), (3, 9)):
        slice_check(case, x, outs, b, h)
    same_bits_with_keep_bits(case, x, outs)
    # keep bits of the sampled slices, bit-exact
    bits = sdpa_dropout_mask(case.B, case.H, case.S_q, case.S_kv, case.p, case.seed,
                             case.offset).cpu().numpy().view(np.uint32)
    flat = np.unpackbits(bits.view(np.uint8), bitorder="little")
    per_head = case.S_q * case.S_kv
    for b, h in ((0, 0), (7, 15), (5, 2)):
        start = (b * case.H + h) * per_head
        got = flat[start:start + per_head].reshape(case.S_q, case.S_kv).astype(bool)
        want = philox.keep_mask(case.B, case.H, case.S_q, case.S_kv, case.p, case.seed,
                                case.offset, b, h)
        np.testing.assert_array_equal(got, want)


def test_b1h32_s16384_d128_causal_sampled():
    case = Case(1, 32, 16384, 16384, 128, 128, causal=True)
    x = make_inputs(case.shape, case.dtype)
    o, lse, dq, dk, dv, _ = outs = run_gpu(case, x)
    pr = case.problem()
    rng = np.random.default_rng(3)
    h = 17
    rows = np.unique(np.concatenate([np.arange(0, 130), np.arange(16384 - 130, 16384),
                                     rng.integers(0, 16384, 120)]))
    cols = np.unique(np.concatenate([np.arange(0, 66), np.arange(16384 - 66, 16384),
                                     rng.integers(0, 16384, 60)]))
    r_t, c_t = torch.as_tensor(rows, device=o.device), torch.as_tensor(cols, device=o.device)
    o_ref, lse_ref = oracle.forward_head(pr, 0, h, x["q"], x["k"], x["v"], rows=rows)
    assert_close("o rows", o[0, h][r_t], o_ref)
    assert_lse(lse[0, h][r_t], lse_ref)
    dq_r, dk_c, dv_c, _ = oracle.backward_head(pr, 0, h, x["q"], x["k"], x["v"], x["do"],
                                               rows=rows, cols=cols, row_chunk=2048)
    assert_close("dq rows", dq[0, h][r_t], dq_r)
    assert_close("dk cols", dk[0, h][c_t], dk_c)
    assert_close("dv cols", dv[0, h][c_t], dv_c)
    key_sum_invariants(case, outs, x)


def test_b1h32kv4_s16384_d128_causal_gqa_sampled():
    """Grouped-query attention at the long-context size (32 query heads on 4 K/V
    heads): sampled rows of one query head, sampled key columns of one K/V head
    (the oracle summed over its 8 query heads), and the key-sum invariants."""
    case = Case(1, 32, 16384, 16384, 128, 128, causal=True, H_kv=4)
    x = make_inputs(case.shape, case.dtype)
    o, lse, dq, dk, dv, _ = outs = run_gpu(case, x)
    assert dk.shape == (1, 4, 16384, 128) and dv.shape == (1, 4, 16384, 128)
    pr = case.problem()
    rng = np.random.default_rng(5)
    h, hk = 21, 2   # query head 21 reads K/V head 2
    rows = np.unique(np.concatenate([np.arange(0, 64), np.arange(16384 - 64, 16384),
                                     rng.integers(0, 16384, 64)]))
    cols = np.unique(np.concatenate([np.arange(0, 32), np.arange(16384 - 32, 16384),
                                     rng.integers(0, 16384, 32)]))
    r_t, c_t = torch.as_tensor(rows, device=o.device), torch.as_tensor(cols, device=o.device)
    o_ref, lse_ref = oracle.forward_head(pr, 0, h, x["q"], x["k"], x["v"], rows=rows)
    assert_close("o rows", o[0, h][r_t], o_ref)
    assert_lse(lse[0, h][r_t], lse_ref)
    dk_ref = np.zeros((len(cols), 128))
    dv_ref = np.zeros((len(cols), 128))
    for hq in range(hk * 8, hk * 8 + 8):
        dq_r, dk_c, dv_c, _ = oracle.backward_head(pr, 0, hq, x["q"], x["k"], x["v"], x["do"],
                                                   rows=rows if hq == h else rows[:1],
                                                   cols=cols, row_chunk=4096)
        if hq == h:
            assert_close("dq rows", dq[0, h][r_t], dq_r)
        dk_ref += dk_c
        dv_ref += dv_c
    assert_close("dk cols (group sum)", dk[0, hk][c_t], dk_ref)
    assert_close("dv cols (group sum)", dv[0, hk][c_t], dv_ref)
    # key sums: dK's vanish; dV's equal the group's query-sum of dO
    dk64 = dk.double()
    rel = dk64.sum(dim=2).abs().max().item() / dk64.abs().sum(dim=2).max().item()
    assert rel < 2e-2, f"key-sum of dK is not ~0 (relative {rel:.3e})"
    do_sum = x["do"].double().sum(dim=2).reshape(1, 4, 8, 128).sum(dim=2).numpy()
    assert_close("sum_j dV", dv.double().sum(dim=2).cpu(), do_sum, rel=3e-2)


def test_dropout_element_index_past_2_pow_32():
    """b1 h8 s32768 d64 with dropout: the last head's linear element indices
    pass 2^32 (the Philox counter's high word is in use). Sampled query rows
    of that head (O, LSE, dQ over all keys) against the oracle, and the last
    keep-bit words the GPU draws against the oracle's Philox."""
    case = Case(1, 8, 32768, 32768, 64, 64, causal=True, p=0.1)
    x = make_inputs(case.shape, case.dtype)
    o, lse, dq, dk, dv, _ = run_gpu(case, x)
    pr = case.problem()
    h = 7
    rows = np.array([0, 1, 4097, 20000, 32766, 32767])
    assert (h * 32768 + int(rows[0])) * 32768 > (1 << 32)
    r_t = torch.as_tensor(rows, device=o.device)
    o_ref, lse_ref = oracle.forward_head(pr, 0, h, x["q"], x["k"], x["v"], rows=rows)
    assert_close("o rows", o[0, h][r_t], o_ref)
    assert_lse(lse[0, h][r_t], lse_ref)
    dq_r, _, _, _ = oracle.backward_head(pr, 0, h, x["q"], x["k"], x["v"], x["do"], rows=rows,
                                         cols=np.array([], dtype=np.int64))
    assert_close("dq rows", dq[0, h][r_t], dq_r)
    same_bits_with_keep_bits(case, x, (o, lse, dq, dk, dv))
    total = 8 * 32768 * 32768
    words = sdpa_dropout_mask(1, 8, 32768, 32768, case.p, case.seed, case.offset)
    last = words[-64:].cpu().numpy().view(np.uint32)
    lin = np.arange(total - 64 * 32, total, dtype=np.uint64)
    keep = philox.random_words(lin, case.seed, case.offset) >= np.uint32(philox.drop_threshold(case.p))
    ref = (keep.reshape(-1, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)).sum(axis=1)
    assert np.array_equal(last, ref.astype(np.uint32))
