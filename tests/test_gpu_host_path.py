"""The host side of the calls on the GPU: a step captured in a CUDA graph and
replayed gives the eager step's results, and the encoded tensor maps the
library keeps per host thread follow each call's pointers and shapes (two
problems over one storage, alternating, each against its own oracle)."""
import pytest
import torch

import oracle
from parity_util import Case, assert_close, assert_lse
from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_bwd_workspace_size, sdpa_device_error, sdpa_fwd
from scaled_dot_product_06_gb300.inputs import make_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("deterministic", [True, False])
def test_graph_replay_equals_eager(deterministic):
    """sdpa_fwd + sdpa_bwd captured once in a CUDA graph: a replay gives the
    eager call's bits (dQ of the default backward within fp32 summation
    order: its reductions add in arrival order)."""
    case = Case(2, 2, 384, 384, 128, 128, causal=True)
    x = make_inputs(case.shape, case.dtype)
    q, k, v, do = (x[n].cuda() for n in ("q", "k", "v", "do"))
    o = torch.empty_like(q)
    lse = torch.empty(case.B, case.H, case.S_q, dtype=torch.float32, device="cuda")
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(sdpa_bwd_workspace_size(case.B, case.H, case.S_q, case.S_kv, case.D_qk, case.D_v,
                                             deterministic=deterministic),
                     dtype=torch.uint8, device="cuda")

    def step():
        sdpa_fwd(q, k, v, out=o, lse=lse, is_causal=True)
        sdpa_bwd(q, k, v, o, do, lse, is_causal=True, workspace=ws, dq=dq, dk=dk, dv=dv,
                 deterministic=deterministic)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # eager, on the stream the capture will use
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    eager = [t.clone() for t in (o, lse, dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=side):
        step()
    for t in (o, lse, dq, dk, dv):
        t.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    for name, a, b in zip(("o", "lse", "dq", "dk", "dv"), (o, lse, dq, dk, dv), eager):
        if name == "dq" and not deterministic:
            assert_close("dq replay vs eager", a, b.double().cpu().numpy(), rel=1e-2)
        else:
            assert torch.equal(a, b), f"{name}: replay differs from the eager call"


def test_tensor_maps_follow_pointers_and_shapes():
    """Two problems whose tensors start at the same addresses (views of one
    storage) but differ in shape, called alternately three times each: every
    call matches its own oracle, so no call reuses a map encoded for the
    other shape."""
    a = Case(1, 2, 256, 256, 64, 64, causal=True)
    b = Case(2, 1, 128, 384, 64, 64)
    xa = make_inputs(a.shape, a.dtype)
    xb = make_inputs(b.shape, b.dtype)
    refs = {}
    for c, xc in ((a, xa), (b, xb)):
        pr = c.problem()
        refs[c] = (*oracle.forward(pr, xc["q"], xc["k"], xc["v"], None),
                   *oracle.backward(pr, xc["q"], xc["k"], xc["v"], xc["do"], None)[:3])
    n = max(a.B * a.H * max(a.S_q, a.S_kv), b.B * b.H * max(b.S_q, b.S_kv)) * 64
    store = {name: torch.empty(n, dtype=torch.bfloat16, device="cuda")
             for name in ("q", "k", "v", "do", "o", "dq", "dk", "dv")}
    lse_store = torch.empty(n // 64, dtype=torch.float32, device="cuda")

    def view(name, shape):
        return store[name][: torch.Size(shape).numel()].view(shape)

    for _ in range(3):
        for c, xc in ((a, xa), (b, xb)):
            sh = c.shape
            q, k, v, do = (view(nm, xc[nm].shape) for nm in ("q", "k", "v", "do"))
            for nm, t in (("q", q), ("k", k), ("v", v), ("do", do)):
                t.copy_(xc[nm])
            o = view("o", (sh.B, sh.H, sh.S_q, sh.D_v))
            lse = lse_store[: sh.B * sh.H * sh.S_q].view(sh.B, sh.H, sh.S_q)
            dq, dk, dv = view("dq", q.shape), view("dk", k.shape), view("dv", v.shape)
            sdpa_fwd(q, k, v, out=o, lse=lse, is_causal=c.causal)
            sdpa_bwd(q, k, v, o, do, lse, is_causal=c.causal, dq=dq, dk=dk, dv=dv)
            torch.cuda.synchronize()
            assert sdpa_device_error() == 0
            o_ref, lse_ref, dq_ref, dk_ref, dv_ref = refs[c]
            assert_close("o", o, o_ref)
            assert_lse(lse, lse_ref)
            assert_close("dq", dq, dq_ref)
            assert_close("dk", dk, dk_ref)
            assert_close("dv", dv, dv_ref)
