"""GPU parity against the fp64 oracle on whole small problems (every element).

Sizes span several 128-row tiles and ragged tails; every feature alone and
combined; bf16 and fp16; every supported head-size pair.
"""
import numpy as np
import pytest
import torch

from oracle import philox
from parity_util import Case, check_full

pytestmark = pytest.mark.gpu

CASES = [
    # the small configuration: b1 h2 s128 d64, scale 1/8, no mask / bias / dropout
    Case(1, 2, 128, 128, 64, 64, scale=0.125),
    Case(2, 2, 256, 384, 64, 64),
    Case(1, 2, 256, 256, 128, 128, causal=True),
    Case(2, 1, 384, 384, 128, 128, causal=True, dtype="fp16"),
    Case(1, 2, 256, 256, 192, 128, causal=True, bias=True),
    Case(2, 2, 128, 256, 64, 64, dtype="fp16", p=0.1),
    Case(2, 2, 256, 256, 128, 128, causal=True, bias=True, p=0.2),
    # ragged tails and s_q != s_kv
    Case(1, 1, 1, 1, 64, 64),
    Case(1, 1, 17, 17, 64, 64, causal=True),
    Case(1, 2, 100, 260, 128, 128, p=0.15),
    Case(1, 1, 129, 257, 128, 128, causal=True, bias=True),
    Case(2, 1, 257, 129, 192, 128, causal=True),
    Case(1, 2, 200, 72, 64, 64, causal=True, bias=True, dtype="fp16"),
    Case(1, 1, 300, 300, 192, 128, bias=True, p=0.3),
    # several query-tile pairs per head, the last pair without its second tile,
    # causal with more keys than queries
    Case(1, 2, 640, 1000, 128, 128, causal=True),
    # grouped K/V heads (GQA, MQA): dK / dV summed over each group of query heads
    Case(2, 4, 256, 256, 128, 128, causal=True, H_kv=2),
    Case(1, 6, 200, 332, 64, 64, bias=True, p=0.1, H_kv=3, dtype="fp16"),
    Case(1, 4, 384, 256, 128, 128, causal=True, H_kv=1),
    Case(2, 4, 192, 192, 192, 128, causal=True, bias=True, H_kv=2),
    # the sign of the scale: the plain kernels take the row max from the raw
    # scores (the smallest under a negative scale); a zero scale runs the
    # kernel that scales first (uniform weights over the visible keys)
    Case(1, 2, 300, 300, 128, 128, causal=True, scale=-0.09),
    Case(1, 1, 200, 260, 64, 64, scale=-0.125, dtype="fp16"),
    Case(1, 2, 256, 300, 128, 128, causal=True, scale=0.0),
    # one key tile that every query tile meets: the fused kernel writes dQ
    # directly (no accumulator, no convert pass)
    Case(2, 2, 300, 100, 128, 128),
    Case(1, 3, 200, 128, 64, 64, causal=True, p=0.1, dtype="fp16"),
    Case(2, 2, 256, 64, 128, 128, causal=True, bias=True),
    Case(1, 4, 130, 96, 128, 128, H_kv=2),
    # a bias whose rows are not a multiple of 16 bytes: the deterministic dQ
    # kernel reads it from global memory instead of by TMA
    Case(1, 2, 130, 130, 192, 128, causal=True, bias=True),
    Case(2, 1, 100, 70, 64, 64, bias=True, dtype="fp16"),
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: (
    f"b{c.B}h{c.H}q{c.S_q}k{c.S_kv}d{c.D_qk}-{c.D_v}-{c.dtype}"
    f"{'-causal' if c.causal else ''}{'-bias' if c.bias else ''}{f'-p{c.p}' if c.p else ''}"))
def test_fwd_bwd_match_oracle(case):
    check_full(case)


@pytest.mark.parametrize("shape,p,seed,offset", [
    ((1, 2, 16, 32), 0.1, 0x1234, 0),
    ((2, 3, 17, 20), 0.5, 7, 2**33 + 5),
    ((1, 1, 1, 36), 0.9, 2**63 + 11, 123),
])
def test_dropout_mask_bit_exact(shape, p, seed, offset):
    from scaled_dot_product_06_gb300 import sdpa_dropout_mask
    B, H, S_q, S_kv = shape
    got = sdpa_dropout_mask(B, H, S_q, S_kv, p, seed, offset).cpu().numpy().view(np.uint32)
    ref = philox.packed_mask_words(B, H, S_q, S_kv, p, seed, offset)
    np.testing.assert_array_equal(got, ref)


def test_zero_sized_problem_is_noop():
    from scaled_dot_product_06_gb300 import sdpa_fwd
    q = torch.zeros(1, 1, 0, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16, device="cuda")
    o, lse = sdpa_fwd(q, k, k)
    assert o.shape == (1, 1, 0, 64) and lse.shape == (1, 1, 0)


@pytest.mark.parametrize("deterministic", [True, False])
def test_backward_is_bitwise_reproducible(deterministic):
    """Deterministic backward: dQ, dK and dV are summed in a fixed order inside
    one CTA each, so two runs on the same inputs give identical bits (dBias is
    reproducible for b <= 2: two fp32 addends onto zero commute exactly). The
    default backward keeps dK and dV (and O, LSE, dBias at b <= 2) bitwise
    reproducible; its dQ sums fp32 reductions in arrival order, so two runs
    agree within the tolerance but not necessarily in the last bits."""
    from parity_util import assert_close, run_gpu
    from scaled_dot_product_06_gb300.inputs import make_inputs
    case = Case(2, 3, 384, 320, 128, 128, causal=True, bias=True, p=0.1)
    x = make_inputs(case.shape, case.dtype, with_bias=True)
    first = run_gpu(case, x, deterministic=deterministic)
    second = run_gpu(case, x, deterministic=deterministic)
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv", "dbias"), first, second):
        if name == "dq" and not deterministic:
            assert_close("dq run to run", a, b.double().cpu().numpy(), rel=1e-2)
        else:
            assert torch.equal(a, b), f"{name} differs between two runs"


@pytest.mark.parametrize("deterministic", [True, False])
def test_grouped_backward_is_bitwise_reproducible(deterministic):
    """With grouped K/V heads, dK and dV of a K/V head are summed over its
    query heads in a fixed order (inside one CTA, or over the CTAs of a split
    key tile in split order whichever finishes last): identical bits run to
    run, in both backward modes (dQ too in the deterministic one)."""
    from parity_util import run_gpu
    from scaled_dot_product_06_gb300.inputs import make_inputs
    case = Case(1, 8, 256, 256, 128, 128, causal=True, H_kv=2)
    x = make_inputs(case.shape, case.dtype)
    first = run_gpu(case, x, deterministic=deterministic)
    second = run_gpu(case, x, deterministic=deterministic)
    for a, b in zip(first[2 if deterministic else 3:5], second[2 if deterministic else 3:5]):
        assert torch.equal(a, b)


def test_default_and_deterministic_backward_agree():
    """The fused backward (dQ accumulated with fp32 reductions) and the
    deterministic split form the same products; their dK (whose K-steps the
    deterministic kernel adds in a different order), dV and dQ agree up to
    fp32 summation order."""
    from parity_util import assert_close, run_gpu
    from scaled_dot_product_06_gb300.inputs import make_inputs
    for case in (Case(2, 4, 640, 520, 128, 128, causal=True),
                 Case(1, 4, 300, 512, 64, 64, dtype="fp16", p=0.1, bias=True),
                 Case(1, 8, 384, 384, 128, 128, causal=True, H_kv=1)):
        x = make_inputs(case.shape, case.dtype, with_bias=case.bias)
        a = run_gpu(case, x)
        b = run_gpu(case, x, deterministic=True)
        for name, i in (("dq", 2), ("dk", 3), ("dv", 4)):
            assert_close(f"{name} fused vs deterministic", a[i], b[i].double().cpu().numpy(),
                         rel=1e-2)


def test_grouped_backward_without_split_room():
    """Given only the ungrouped workspace size, a grouped backward runs one CTA
    per key tile (no split) and still matches the oracle."""
    import oracle
    from parity_util import assert_close
    from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_bwd_workspace_size, sdpa_fwd
    from scaled_dot_product_06_gb300.inputs import make_inputs
    case = Case(1, 4, 384, 256, 128, 128, causal=True, H_kv=1)
    x = make_inputs(case.shape, case.dtype)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    small = sdpa_bwd_workspace_size(1, 4, 384, 256, 128, 128)
    assert small < sdpa_bwd_workspace_size(1, 4, 384, 256, 128, 128, h_kv=1)
    ws = torch.empty(small, dtype=torch.uint8, device="cuda")
    o, lse = sdpa_fwd(q, k, v, is_causal=True)
    dq, dk, dv, _ = sdpa_bwd(q, k, v, o, do, lse, is_causal=True, workspace=ws)
    torch.cuda.synchronize()
    _, dk_r, dv_r, _ = oracle.backward(case.problem(), x["q"], x["k"], x["v"], x["do"])
    assert_close("dk", dk, dk_r)
    assert_close("dv", dv, dv_r)


@pytest.mark.parametrize("h_kv", [8, 2])
def test_concurrent_backward_equals_phases_bitwise(h_kv):
    """The deterministic sdpa_bwd runs dK/dV on a side stream next to dQ; the
    same kernels run one after the other through sdpa_bwd_phases give the same
    bits."""
    from scaled_dot_product_06_gb300 import (SDPA_BWD_DKDV, SDPA_BWD_DQ, SDPA_BWD_PREPROCESS,
                                             sdpa_bwd, sdpa_bwd_phases, sdpa_bwd_workspace_size,
                                             sdpa_fwd)
    from scaled_dot_product_06_gb300.inputs import make_inputs
    case = Case(2, 8, 640, 640, 128, 128, causal=True, H_kv=h_kv)
    x = make_inputs(case.shape, case.dtype, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse = sdpa_fwd(q, k, v, is_causal=True)
    a = sdpa_bwd(q, k, v, o, do, lse, is_causal=True, deterministic=True)
    ws = torch.empty(sdpa_bwd_workspace_size(2, 8, 640, 640, 128, 128, h_kv=h_kv,
                                             deterministic=True),
                     dtype=torch.uint8, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for ph in (SDPA_BWD_PREPROCESS, SDPA_BWD_DKDV, SDPA_BWD_DQ):
        sdpa_bwd_phases(ph, q, k, v, o, do, lse, is_causal=True, dq=dq, dk=dk, dv=dv,
                        workspace=ws, deterministic=True)
    torch.cuda.synchronize()
    for x1, x2 in zip(a[:3], (dq, dk, dv)):
        assert torch.equal(x1, x2)


def test_fused_backward_phases_equal_the_whole_call():
    """The default backward's three phases (preprocess, fused key/value-stationary
    kernel, dQ convert) issued one by one give sdpa_bwd's dK and dV bits and
    its dQ up to the order of the fp32 reductions."""
    from parity_util import assert_close
    from scaled_dot_product_06_gb300 import (SDPA_BWD_DKDV, SDPA_BWD_DQ, SDPA_BWD_PREPROCESS,
                                             sdpa_bwd, sdpa_bwd_phases, sdpa_bwd_workspace_size,
                                             sdpa_fwd)
    from scaled_dot_product_06_gb300.inputs import make_inputs
    case = Case(2, 4, 640, 640, 128, 128, causal=True)
    x = make_inputs(case.shape, case.dtype, device="cuda")
    q, k, v, do = x["q"], x["k"], x["v"], x["do"]
    o, lse = sdpa_fwd(q, k, v, is_causal=True)
    a = sdpa_bwd(q, k, v, o, do, lse, is_causal=True)
    ws = torch.empty(sdpa_bwd_workspace_size(2, 4, 640, 640, 128, 128), dtype=torch.uint8,
                     device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    for ph in (SDPA_BWD_PREPROCESS, SDPA_BWD_DKDV, SDPA_BWD_DQ):
        sdpa_bwd_phases(ph, q, k, v, o, do, lse, is_causal=True, dq=dq, dk=dk, dv=dv,
                        workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(a[1], dk) and torch.equal(a[2], dv)
    assert_close("dq phases vs whole call", dq, a[0].double().cpu().numpy(), rel=1e-2)


@pytest.mark.parametrize("case", [
    Case(2, 4, 384, 512, 64, 64, dtype="fp16", p=0.1),
    Case(1, 4, 300, 332, 128, 128, causal=True, p=0.2, H_kv=2),
    Case(2, 2, 256, 256, 192, 128, causal=True, bias=True, p=0.15),
], ids=["d64-fp16", "d128-causal-gqa-ragged", "d192-bias"])
def test_dropout_bits_drawn_beforehand_give_the_same_bits(case):
    """With the keep bits of sdpa_dropout_mask passed in, every kernel reads them
    instead of drawing Philox numbers: O, LSE, dQ, dK, dV, dBias identical
    (deterministic backward, whose every output is reproducible bit for bit)."""
    from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_dropout_mask, sdpa_fwd
    from scaled_dot_product_06_gb300.inputs import make_inputs
    x = make_inputs(case.shape, case.dtype, with_bias=case.bias, device="cuda")
    q, k, v, do, bias = x["q"], x["k"], x["v"], x["do"], x["bias"]
    kw = dict(scale=case.sc, is_causal=case.causal, dropout_p=case.p, seed=case.seed,
              offset=case.offset, bias=bias, deterministic=True)
    fkw = {n: a for n, a in kw.items() if n != "deterministic"}
    o1, l1 = sdpa_fwd(q, k, v, **fkw)
    g1 = sdpa_bwd(q, k, v, o1, do, l1, **kw)
    mask = sdpa_dropout_mask(case.B, case.H, case.S_q, case.S_kv, case.p, case.seed, case.offset)
    o2, l2 = sdpa_fwd(q, k, v, dropout_mask=mask, **fkw)
    g2 = sdpa_bwd(q, k, v, o2, do, l2, dropout_mask=mask, **kw)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for a, b in zip(g1, g2):
        assert (a is None and b is None) or torch.equal(a, b)


@pytest.mark.parametrize("case", [
    Case(2, 2, 256, 384, 64, 64, dtype="fp16", p=0.1),
    Case(1, 4, 300, 320, 128, 128, causal=True, p=0.2, H_kv=2),
    Case(1, 2, 200, 256, 192, 128, causal=True, bias=True, p=0.15),
], ids=["d64-fp16", "d128-causal-gqa-ragged", "d192-bias"])
def test_forward_keep_bit_record(case):
    """A forward asked to record its dropout keep bits writes exactly
    sdpa_dropout_mask's words (every query row sees every key tile here, or
    the causal diagonal and below, which the comparison covers), its O and LSE
    are those of the forward without a record, and a backward given the
    record reproduces the backward that draws its own bits: every gradient of
    the deterministic backward bit for bit, dK and dV of the default one bit
    for bit and its dQ up to the order of its fp32 reductions."""
    from parity_util import assert_close
    from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_dropout_mask, sdpa_fwd
    from scaled_dot_product_06_gb300.inputs import make_inputs
    x = make_inputs(case.shape, case.dtype, with_bias=case.bias, device="cuda")
    q, k, v, do, bias = x["q"], x["k"], x["v"], x["do"], x["bias"]
    kw = dict(scale=case.sc, is_causal=case.causal, dropout_p=case.p, seed=case.seed,
              offset=case.offset, bias=bias)
    words = (case.B * case.H * case.S_q * case.S_kv + 31) // 32
    rec = torch.zeros(words, dtype=torch.int32, device="cuda")
    o1, l1 = sdpa_fwd(q, k, v, **kw)
    o2, l2 = sdpa_fwd(q, k, v, dropout_mask_out=rec, **kw)
    ref = sdpa_dropout_mask(case.B, case.H, case.S_q, case.S_kv, case.p, case.seed, case.offset)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    got_w = rec.cpu().numpy().view(np.uint32).reshape(case.B * case.H, case.S_q, case.S_kv // 32)
    ref_w = ref.cpu().numpy().view(np.uint32).reshape(case.B * case.H, case.S_q, case.S_kv // 32)
    if case.causal:  # words holding a key at or below the diagonal: the forward visits their tile
        rows = np.arange(case.S_q)[:, None]
        first_key = 32 * np.arange(case.S_kv // 32)[None, :]
        keep = np.broadcast_to((first_key // 128) * 128 <= rows, got_w.shape)
        np.testing.assert_array_equal(got_w[keep], ref_w[keep])
    else:
        np.testing.assert_array_equal(got_w, ref_w)
    for det in (True, False):
        g1 = sdpa_bwd(q, k, v, o1, do, l1, deterministic=det, **kw)
        g2 = sdpa_bwd(q, k, v, o1, do, l1, dropout_mask=rec, deterministic=det, **kw)
        torch.cuda.synchronize()
        for name, a, b in zip(("dq", "dk", "dv", "dbias"), g1, g2):
            if a is None:
                continue
            if name == "dq" and not det and case.D_qk <= 128:
                assert_close("dq with the record", b, a.double().cpu().numpy(), rel=1e-2)
            else:
                assert torch.equal(a, b), (name, det)
