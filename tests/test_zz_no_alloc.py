"""sdpa_bwd_noalloc: the backward pass for callers that cannot allocate.

Some callers cannot allocate device memory when they run the backward pass
(a framework that owns all GPU memory through its own pool, or a
latency-critical loop that cannot pay for cudaMalloc's implicit
synchronisation). sdpa_bwd_noalloc serves them with a fixed 16 MiB scratch
array inside the library instead of a caller workspace, running the
deterministic backward. These tests call it through the C ABI and compare it
with the deterministic sdpa_bwd on the same inputs, bit for bit, twice in a
row (the second call reuses the scratch the first one left behind, so stale
contents that changed even the last bit would show). The size limit is
checked on the host and tested in test_abi.py.

The file is named so that pytest collects it last.
"""
import ctypes

import pytest
import torch

from scaled_dot_product_06_gb300 import _native, sdpa_bwd, sdpa_device_error, sdpa_fwd
from scaled_dot_product_06_gb300.inputs import Shape, make_inputs

pytestmark = pytest.mark.gpu

_DT = {"bf16": _native.SDPA_BF16, "fp16": _native.SDPA_FP16}


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_noalloc(shape, dtype, scale, causal, p, seed, offset, x, o, lse, outs):
    dq, dk, dv, dbias = outs
    return _native.lib().sdpa_bwd_noalloc(
        shape.B, shape.H, shape.S_q, shape.S_kv, shape.D_qk, shape.D_v, scale, int(causal), p,
        seed, offset, _DT[dtype], _p(x["q"]), _p(x["k"]), _p(x["v"]), _p(x["bias"]), _p(o),
        _p(x["do"]), _p(lse), _p(dq), _p(dk), _p(dv), _p(dbias),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("shape,dtype,causal,with_bias,p", [
    (Shape(1, 2, 256, 256, 128, 128), "bf16", True, False, 0.0),
    (Shape(2, 2, 200, 136, 64, 64), "fp16", False, True, 0.1),
    (Shape(1, 1, 129, 257, 192, 128), "bf16", True, True, 0.0),
])
def test_noalloc_matches_workspace_backward_twice(shape, dtype, causal, with_bias, p):
    x = {n: (t.cuda() if t is not None else None)
         for n, t in make_inputs(shape, dtype, with_bias=with_bias).items()}
    scale, seed, offset = 1.0 / shape.D_qk ** 0.5, 0x1234, 7
    kw = dict(scale=scale, is_causal=causal, dropout_p=p, seed=seed, offset=offset,
              bias=x["bias"])
    o, lse = sdpa_fwd(x["q"], x["k"], x["v"], **kw)
    ref = sdpa_bwd(x["q"], x["k"], x["v"], o, x["do"], lse, deterministic=True, **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0
    for _ in range(2):
        outs = (torch.empty_like(x["q"]), torch.empty_like(x["k"]), torch.empty_like(x["v"]),
                torch.empty_like(x["bias"]) if with_bias else None)
        st = call_noalloc(shape, dtype, scale, causal, p, seed, offset, x, o, lse, outs)
        assert st == _native.SDPA_OK, _native.lib().sdpa_last_error().decode()
        torch.cuda.synchronize()
        assert sdpa_device_error() == 0
        for name, got, want in zip(("dq", "dk", "dv", "dbias"), outs, ref):
            if want is not None:
                assert torch.equal(got, want), f"{name} differs from the deterministic sdpa_bwd"

