"""Helpers for the GPU-vs-oracle parity tests.

Tolerances (from the method's precision contract): O, dQ, dK, dV and dBias
within max|err| <= 2e-2 * max|ref| of the fp64 oracle; LSE within 1e-3
absolute; dropout keep bits bit-exact.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np
import torch

import oracle
from scaled_dot_product_06_gb300 import sdpa_bwd, sdpa_device_error, sdpa_fwd
from scaled_dot_product_06_gb300.inputs import Shape, make_inputs

REL_TOL = 2e-2
LSE_TOL = 1e-3


@dataclass(frozen=True)
class Case:
    B: int
    H: int
    S_q: int
    S_kv: int
    D_qk: int
    D_v: int
    dtype: str = "bf16"
    causal: bool = False
    bias: bool = False
    p: float = 0.0
    scale: float | None = None
    seed: int = 0x1234
    offset: int = 0
    H_kv: int = 0  # K/V heads (grouped-query attention); 0 means H

    @property
    def shape(self):
        return Shape(self.B, self.H, self.S_q, self.S_kv, self.D_qk, self.D_v, self.H_kv)

    @property
    def sc(self):
        return self.scale if self.scale is not None else 1.0 / np.sqrt(self.D_qk)

    def problem(self):
        return oracle.Problem(self.B, self.H, self.S_q, self.S_kv, self.D_qk, self.D_v, self.sc,
                              self.causal, self.p, self.seed, self.offset, self.H_kv)


def assert_close(name, got, ref, rel=REL_TOL):
    got = got.double().cpu().numpy() if isinstance(got, torch.Tensor) else np.asarray(got)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{name}: non-finite values"
    err = np.abs(got - ref).max() if ref.size else 0.0
    scale = np.abs(ref).max() if ref.size else 0.0
    assert err <= rel * scale + 1e-6, f"{name}: max|err| {err:.4e} > {rel} * max|ref| {scale:.4e}"
    return err, scale


def assert_lse(got, ref):
    got = got.double().cpu().numpy()
    ninf = np.isneginf(ref)
    assert np.array_equal(np.isneginf(got), ninf), "lse: -inf rows differ"
    err = np.abs(got[~ninf] - ref[~ninf]).max() if (~ninf).any() else 0.0
    assert err <= LSE_TOL, f"lse: max|err| {err:.3e} > {LSE_TOL}"


def fused_applies(case: Case) -> bool:
    """The default backward accumulates dQ in the key/value-stationary kernel
    at d_qk <= 128; at d_qk = 192 it is the deterministic backward."""
    return case.D_qk <= 128


def run_gpu(case: Case, x: dict, dev="cuda", deterministic=False):
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    bias = None if x["bias"] is None else x["bias"].to(dev)
    kw = dict(scale=case.sc, is_causal=case.causal, dropout_p=case.p, seed=case.seed,
              offset=case.offset, bias=bias)
    o, lse = sdpa_fwd(q, k, v, **kw)
    dq, dk, dv, dbias = sdpa_bwd(q, k, v, o, do, lse, deterministic=deterministic, **kw)
    torch.cuda.synchronize()
    assert sdpa_device_error() == 0, "a kernel wait ran out"
    return o, lse, dq, dk, dv, dbias


def check_full(case: Case):
    """Element-by-element comparison of every output on the whole problem, for
    the default backward and (where it differs) the deterministic one."""
    x = make_inputs(case.shape, case.dtype, with_bias=case.bias)
    pr = case.problem()
    o_ref, lse_ref = oracle.forward(pr, x["q"], x["k"], x["v"], x["bias"])
    dq_ref, dk_ref, dv_ref, db_ref = oracle.backward(pr, x["q"], x["k"], x["v"], x["do"],
                                                     x["bias"])
    for deterministic in ((False, True) if fused_applies(case) else (False,)):
        o, lse, dq, dk, dv, dbias = run_gpu(case, x, deterministic=deterministic)
        tag = " (deterministic)" if deterministic else ""
        assert_close("o", o, o_ref)
        assert_lse(lse, lse_ref)
        assert_close("dq" + tag, dq, dq_ref)
        assert_close("dk" + tag, dk, dk_ref)
        assert_close("dv" + tag, dv, dv_ref)
        if case.bias:
            assert_close("dbias" + tag, dbias, db_ref)
