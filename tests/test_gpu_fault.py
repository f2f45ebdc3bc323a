"""Hang safety on the GPU without a fault: a bounded wait that runs out.

With the test hook of the C ABI set, the forward kernel's producer warp
issues no K/V loads, so the MMA issuer's wait can never complete. The wait is
bounded by wall-clock time (50 ms here): when it runs out the kernel records
its site in the device error word, every role leaves its loop, drains what
is in flight, frees tensor memory and returns. The host then reads
SDPA_ERR_DEVICE_TIMEOUT, and the next normal call on the same context
matches the oracle. Nothing traps or faults.
"""
import ctypes

import pytest
import torch

from scaled_dot_product_06_gb300 import _native, sdpa_debug_fault, sdpa_device_error, sdpa_fwd
from scaled_dot_product_06_gb300.inputs import Shape, make_inputs
from parity_util import Case, check_full

# site bits of the forward's MMA issuer and softmax warps in the error word:
# whichever of their waits runs out first records its site, the other role
# then sees the CTA's abort flag and leaves without recording one
K_SITES_FWD = (1 << 1) | (1 << 2)


@pytest.mark.gpu
def test_forward_wait_runs_out_and_context_stays_usable():
    x = make_inputs(Shape(1, 2, 256, 256, 64, 64), "bf16", device="cuda")
    assert sdpa_device_error() == 0
    sdpa_debug_fault(1, 50_000_000)
    try:
        sdpa_fwd(x["q"], x["k"], x["v"], is_causal=True)
        torch.cuda.synchronize()
        w = ctypes.c_uint32(0)
        st = _native.lib().sdpa_device_error(ctypes.byref(w), 1)
        assert st == _native.SDPA_ERR_DEVICE_TIMEOUT
        assert w.value != 0 and (w.value & ~K_SITES_FWD) == 0
    finally:
        sdpa_debug_fault(0, 0)
    assert sdpa_device_error() == 0
    # the context is healthy: a normal forward + backward still matches the oracle
    check_full(Case(1, 2, 256, 256, 64, 64, causal=True))
    assert sdpa_device_error() == 0
