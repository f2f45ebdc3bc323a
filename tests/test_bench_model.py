"""bench.py's counting model, on the CPU: the visible (query, key) pairs a mask
leaves, the forward FLOPs by the convention, the algorithmic bytes each kernel
moves and the roofline each workload is held to. The pair counts are checked
against brute force over small masks; the bytes against the tensors the
kernels read and write, summed one by one."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def brute_pairs(s_q, s_kv, window, bottom_right):
    """Visible pairs by enumeration: key j is visible to row i when
    i + off - left <= j <= i + off + right (a negative side is unbounded)."""
    left, right = window
    off = s_kv - s_q if bottom_right else 0
    n = 0
    for i in range(s_q):
        for j in range(s_kv):
            if (left < 0 or j >= i + off - left) and (right < 0 or j <= i + off + right):
                n += 1
    return n


@pytest.mark.parametrize("s_q,s_kv,window,br", [
    (17, 17, (4, 0), False), (20, 33, (5, 2), True), (33, 20, (-1, 0), False),
    (9, 40, (3, -1), True), (12, 12, (0, 0), False), (30, 7, (2, 3), True)])
def test_visible_pairs_match_enumeration(s_q, s_kv, window, br):
    assert bench.visible_pairs(s_q, s_kv, window, br) == brute_pairs(s_q, s_kv, window, br)


def test_causal_pairs_are_the_lower_triangle():
    for s in (1, 5, 128, 300):
        w = dict(S_q=s, S_kv=s, causal=True)
        assert bench.visible_pairs_per_head(w) == s * (s + 1) // 2
    # fewer keys than rows: the rows past the last key see every key
    w = dict(S_q=10, S_kv=4, causal=True)
    assert bench.visible_pairs_per_head(w) == brute_pairs(10, 4, (-1, 0), False)


def test_forward_flops_convention():
    w = bench.resolve(bench.WORKLOADS["b1h32-s16384-d128-causal"])
    # 4 b h s_q s_kv (d_qk + d_v) / 2 per forward, halved for causal
    assert bench.fwd_flops(w) == 4.0 * 32 * 16384 * 16384 * 256 / 2 / 2
    # a causal window of the whole sequence counts the causal pairs, 2 (d_qk + d_v) FLOPs each
    ww = dict(w, window=(16384, 0), bottom_right=False)
    assert bench.fwd_flops(ww) == 2.0 * 32 * (16384 * 16385 // 2) * 256


def test_headline_kernel_bytes_are_the_tensors():
    w = bench.resolve(bench.WORKLOADS["b1h32-s16384-d128-causal"])
    rows = 32 * 16384
    q = k = v = o = do = dq = dk = dv = rows * 128 * 2   # bf16
    lse, stats = rows * 4, rows * 8
    acc = rows * 128 * 4                                  # the fp32 dQ accumulator
    kb = bench.kernel_bytes(w, fused=True)
    assert kb["fwd"] == q + k + v + o + lse
    assert kb["bwd_pre"] == o + do + lse + stats
    assert kb["bwd_fused"] == q + do + k + v + stats + dk + dv
    assert kb["dq_convert"] == acc + dq
    kd = bench.kernel_bytes(w, fused=False)
    assert kd["bwd_dkdv"] == kb["bwd_fused"]
    assert kd["bwd_dq"] == q + do + k + v + stats + dq


def test_bias_bytes_read_over_visible_pairs_and_written_in_full():
    w = bench.resolve(bench.WORKLOADS["b2h16-s4096-d192x128-causal-bias"])
    kb = bench.kernel_bytes(w, fused=False)
    plain = bench.kernel_bytes(dict(w, bias=False), fused=False)
    pairs = 4096 * 4097 // 2
    # the bias is one [h, s_q, s_kv] fp32 tensor shared by the batch
    assert kb["fwd"] - plain["fwd"] == 16 * pairs * 4
    assert kb["bwd_dkdv"] - plain["bwd_dkdv"] == 16 * pairs * 4 + 16 * 4096 * 4096 * 4
    assert kb["bwd_dq"] - plain["bwd_dq"] == 16 * pairs * 4


def test_packed_workload_counts_each_sequence():
    w = bench.resolve(bench.WORKLOADS["varlen16-h32-d128-causal"])
    lens = w["lens"]
    assert len(lens) == 16 and sum(lens) == 74372
    assert bench.visible_pairs_per_head(w) == sum(n * (n + 1) // 2 for n in lens)
    assert bench.fwd_flops(w) == pytest.approx(sum(4.0 * 32 * n * n * 256 / 2 / 2 for n in lens))


@pytest.mark.parametrize("name,draws,bound", [
    ("b1h32-s16384-d128-causal", False, "tensor"),
    ("b2h16-s4096-d192x128-causal-bias", False, "hbm"),
    ("b8h16-s1024x2048-d64-fp16-dropout0.1", True, "alu"),
    ("b8h16-s1024x2048-d64-fp16-dropout0.1", False, "tensor"),
    ("b1h2-s128-d64", False, "hbm")])
def test_workload_bound(name, draws, bound):
    w = bench.resolve(bench.WORKLOADS[name])
    assert bench.workload_bound(w, bench.fwd_flops(w) / 1e9, draws) == bound


def test_visible_pairs_of_the_window_workload():
    w = bench.resolve(bench.WORKLOADS["b1h32-s16384-d128-window4096"])
    # row i sees keys max(0, i - 4096) .. i
    i = np.arange(16384)
    assert bench.visible_pairs_per_head(w) == int((i - np.maximum(i - 4096, 0) + 1).sum())
