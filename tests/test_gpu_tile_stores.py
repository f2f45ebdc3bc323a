"""Every output element is written, whichever way a tile leaves its kernel.

dK / dV (both backwards) and the deterministic dQ go out as whole tiles by
tensor-map stores from shared memory, except a packed sequence's ragged tile,
which is written row by row. The outputs here start as NaN, so an element no
store reaches shows up. The cases hold key tiles that no query sees (top-left
causal with s_kv > s_q: their dK and dV are exactly zero), ragged last tiles
of unpacked tensors (the store must drop the rows past the end, which belong
to the next head) and every head size, against the oracle."""
import pytest
import torch

import oracle
from parity_util import Case, assert_close
from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_device_error, sdpa_fwd
from scaled_dot_product_06_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu

CASES = [
    Case(1, 2, 129, 385, 64, 64, causal=True),
    Case(2, 1, 129, 300, 128, 128, causal=True),
    Case(1, 2, 129, 260, 192, 128, causal=True),
    Case(2, 2, 200, 333, 64, 64, dtype="fp16"),
]


@pytest.mark.parametrize("deterministic", [False, True])
@pytest.mark.parametrize("case", CASES, ids=lambda c: f"b{c.B}h{c.H}-{c.S_q}x{c.S_kv}-d{c.D_qk}")
def test_every_output_element_is_stored(case, deterministic):
    x = make_inputs(case.shape, case.dtype)
    pr = case.problem()
    dq_ref, dk_ref, dv_ref, _ = oracle.backward(pr, x["q"], x["k"], x["v"], x["do"], None)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o, lse = sdpa_fwd(q, k, v, scale=case.sc, is_causal=case.causal)
    # each gradient is a view at the start of a NaN buffer with 4096 elements
    # to spare: the stores must stop at the tensor's end, leaving that tail NaN
    bufs = {n: torch.full((t.numel() + 4096,), float("nan"), dtype=t.dtype, device="cuda")
            for n, t in (("dq", q), ("dk", k), ("dv", v))}
    dq = bufs["dq"][: q.numel()].view(q.shape)
    dk = bufs["dk"][: k.numel()].view(k.shape)
    dv = bufs["dv"][: v.numel()].view(v.shape)
    sdpa_bwd(q, k, v, o, do, lse, scale=case.sc, is_causal=case.causal, dq=dq, dk=dk, dv=dv,
             deterministic=deterministic)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert not torch.isnan(t).any(), f"{name}: elements left unwritten"
    for name, t in (("dq", q), ("dk", k), ("dv", v)):
        assert torch.isnan(bufs[name][t.numel():]).all(), f"{name}: a store ran past the tensor's end"
    if case.causal and case.S_kv > case.S_q:  # keys past the last query row: no query sees them
        assert torch.count_nonzero(dk[:, :, case.S_q:]) == 0
        assert torch.count_nonzero(dv[:, :, case.S_q:]) == 0
    assert_close("dq", dq, dq_ref)
    assert_close("dk", dk, dk_ref)
    assert_close("dv", dv, dv_ref)
