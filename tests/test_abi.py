"""The C ABI loads, exports every function include/sdpa.h declares, and
rejects bad arguments with the documented status before touching CUDA (so
these run without a GPU: validation happens before any CUDA call)."""
import ctypes
import os
import re

import pytest

from scaled_dot_product_06_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sdpa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_native.LIB_PATH):
        from scaled_dot_product_06_gb300 import build
        build.build()
    return _native.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sdpa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("sdpa_fwd", "sdpa_bwd", "sdpa_bwd_workspace_size", "sdpa_dropout_mask",
                 "sdpa_device_error", "sdpa_status_string"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    assert set(declared_functions()) == set(_native.SIGNATURES), \
        "binding signatures and header disagree"


def test_status_strings(lib):
    for code in range(7):
        assert _native.status_string(code).startswith("SDPA_")
    assert lib.sdpa_version() >= 10000


NULL = None
P = ctypes.c_void_p(1 << 20)        # a 16-byte aligned non-null value (never dereferenced)
MIS = ctypes.c_void_p((1 << 20) + 8)


def fwd(lib, b=1, h=1, sq=128, skv=128, dqk=64, dv=64, p=0.0, dtype=0, q=P, k=P, v=P, bias=NULL,
        o=P, lse=P, scale=0.125):
    return lib.sdpa_fwd(b, h, sq, skv, dqk, dv, scale, 0, p, 0, 0, dtype, q, k, v, bias, o, lse,
                        None)


def test_fwd_argument_errors(lib):
    assert fwd(lib, b=-1) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, dqk=96, dv=96) == _native.SDPA_ERR_UNSUPPORTED
    assert fwd(lib, dqk=128, dv=64) == _native.SDPA_ERR_UNSUPPORTED
    assert fwd(lib, dtype=7) == _native.SDPA_ERR_UNSUPPORTED
    assert fwd(lib, p=1.0) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, p=-0.1) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, p=float("nan")) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, p=0.1, skv=130) == _native.SDPA_ERR_UNSUPPORTED
    for bad in (float("nan"), float("inf"), -float("inf"), 3.0e38):  # scale * log2(e) not finite
        assert fwd(lib, scale=bad) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, q=NULL) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, lse=NULL) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(lib, k=MIS) == _native.SDPA_ERR_MISALIGNED
    assert fwd(lib, bias=MIS) == _native.SDPA_ERR_MISALIGNED
    # zero-sized problems are a no-op even with null pointers
    assert fwd(lib, sq=0, q=NULL, o=NULL, lse=NULL) == _native.SDPA_OK
    assert fwd(lib, b=0, q=NULL) == _native.SDPA_OK


def bwd(lib, b=1, h=1, sq=128, skv=128, dqk=64, dv=64, p=0.0, bias=NULL, dbias=NULL, ws=P,
        ws_bytes=None, dout=P, q=P, scale=0.125):
    if ws_bytes is None:
        ws_bytes = lib.sdpa_bwd_workspace_size(b, h, sq, skv, dqk, dv)
    return lib.sdpa_bwd(b, h, sq, skv, dqk, dv, scale, 1, p, 0, 0, 0, q, P, P, bias, P, dout, P,
                        P, P, P, dbias, ws, ws_bytes, None)


def test_workspace_size(lib):
    b, h, sq = 2, 3, 100
    s_pad = (sq + 127) // 128 * 128  # query rows padded to whole 128-row tiles
    stats = ((b * h * s_pad * 2 * 4 + 255) // 256) * 256  # -LSE*log2e and D, fp32 per row
    for dqk, dv in ((64, 64), (128, 128)):
        dq_acc = b * h * s_pad * dqk * 4  # the default backward's fp32 dQ accumulator
        assert lib.sdpa_bwd_workspace_size(b, h, sq, 50, dqk, dv) == stats + dq_acc
        assert lib.sdpa_bwd_workspace_size_ex(b, h, h, sq, 50, dqk, dv, 0) == stats + dq_acc
        assert lib.sdpa_bwd_workspace_size_ex(b, h, h, sq, 50, dqk, dv, 1) == stats
    # d_qk = 192 always runs the deterministic backward: statistics only
    assert lib.sdpa_bwd_workspace_size(b, h, sq, 50, 192, 128) == stats
    assert lib.sdpa_bwd_workspace_size_ex(b, h, h, sq, 50, 192, 128, 0) == stats
    assert lib.sdpa_bwd_workspace_size(1, 1, 8, 8, 80, 80) == 0
    assert lib.sdpa_bwd_workspace_size_ex(1, 4, 3, 8, 8, 64, 64, 0) == 0  # 3 does not divide 4
    # b and h are bounded one by one before their product is formed
    assert lib.sdpa_bwd_workspace_size(1 << 40, 1 << 40, 8, 8, 64, 64) == 0


def test_backward_phase_flags_validated(lib):
    for phases in (0, 8, 16, 7 | 16):  # no phase, the flag alone, unknown bits
        st = lib.sdpa_bwd_phases(phases, 1, 1, 128, 128, 64, 64, 0.125, 1, 0.0, 0, 0, 0, P, P, P,
                                 None, P, P, P, P, P, P, None, P, 1 << 20, None)
        assert st == _native.SDPA_ERR_INVALID_ARG


def test_deterministic_backward_needs_only_the_statistics(lib):
    # the default backward wants the dQ accumulator too; the deterministic
    # one is satisfied by the statistics alone (both rejected before any launch)
    stats = lib.sdpa_bwd_workspace_size_ex(1, 1, 1, 128, 128, 64, 64, 1)
    assert bwd(lib, ws_bytes=stats) == _native.SDPA_ERR_WORKSPACE
    st = lib.sdpa_bwd_phases(7 | 8, 1, 1, 128, 128, 64, 64, 0.125, 1, 0.0, 0, 0, 0, P, P, P, None,
                             P, P, P, P, P, P, None, P, stats - 256, None)
    assert st == _native.SDPA_ERR_WORKSPACE


def test_noalloc_rejects_problems_larger_than_its_scratch(lib):
    # Host-only: the size check runs before any CUDA call, so the pointers are
    # never dereferenced. 64 * 64 * 2048 query rows need 64 * 64 * 2048 * 8
    # bytes (~67 MB) of statistics, more than the 16 MiB static scratch.
    B, H, S, D = 64, 64, 2048, 128
    st = lib.sdpa_bwd_noalloc(B, H, S, S, D, D, 0.1, 1, 0.0, 0, 0, _native.SDPA_BF16, P, P, P, None,
                              P, P, P, P, P, P, None, None)
    assert st == _native.SDPA_ERR_WORKSPACE
    assert "16 MiB" in lib.sdpa_last_error().decode()


def test_bwd_argument_errors(lib):
    assert bwd(lib, dout=NULL) == _native.SDPA_ERR_INVALID_ARG
    assert bwd(lib, bias=P, dbias=NULL) == _native.SDPA_ERR_INVALID_ARG
    assert bwd(lib, bias=NULL, dbias=P) == _native.SDPA_ERR_INVALID_ARG
    assert bwd(lib, ws=NULL) == _native.SDPA_ERR_WORKSPACE
    assert bwd(lib, ws_bytes=16) == _native.SDPA_ERR_WORKSPACE
    assert bwd(lib, ws=ctypes.c_void_p((1 << 20) + 16)) == _native.SDPA_ERR_MISALIGNED
    assert bwd(lib, q=MIS) == _native.SDPA_ERR_MISALIGNED
    assert bwd(lib, dqk=192, dv=192) == _native.SDPA_ERR_UNSUPPORTED
    assert bwd(lib, scale=float("nan")) == _native.SDPA_ERR_INVALID_ARG
    assert bwd(lib, scale=-float("inf")) == _native.SDPA_ERR_INVALID_ARG
    assert bwd(lib, skv=0, q=NULL) == _native.SDPA_OK


def test_dropout_mask_argument_errors(lib):
    f = lib.sdpa_dropout_mask
    assert f(1, 1, 4, 4, 1.5, 0, 0, P, None) == _native.SDPA_ERR_INVALID_ARG
    assert f(1, 1, 4, 4, 0.5, 0, 0, NULL, None) == _native.SDPA_ERR_INVALID_ARG
    assert f(0, 1, 4, 4, 0.5, 0, 0, NULL, None) == _native.SDPA_OK


def test_debug_fault_hook_arguments(lib):
    # host-only: setting and clearing the test hook touches no device
    assert lib.sdpa_debug_fault(2, 0) == 1          # SDPA_ERR_INVALID_ARG
    assert lib.sdpa_debug_fault(-1, 0) == 1
    assert lib.sdpa_debug_fault(0, 0) == 0


def test_grouped_kv_heads_validated_before_any_device_work(lib):
    P = ctypes.c_void_p(16)  # never dereferenced: the calls fail validation first
    def fwd_gqa(h, h_kv):
        return lib.sdpa_fwd_gqa(1, h, h_kv, 64, 64, 64, 64, 0.125, 0, 0.0, 0, 0, 0, P, P, P, None,
                                P, P, None)
    assert fwd_gqa(4, 3) == _native.SDPA_ERR_INVALID_ARG   # 3 does not divide 4
    assert fwd_gqa(4, 0) == _native.SDPA_ERR_INVALID_ARG
    assert fwd_gqa(4, 8) == _native.SDPA_ERR_INVALID_ARG   # more K/V heads than query heads
    assert fwd_gqa(4, -2) == _native.SDPA_ERR_INVALID_ARG
    ws = ctypes.c_void_p(256)
    st = lib.sdpa_bwd_phases_gqa(7, 1, 6, 4, 64, 64, 64, 64, 0.125, 0, 0.0, 0, 0, 0, P, P, P, None,
                                 P, P, P, P, P, P, None, ws, 1 << 20, None)
    assert st == _native.SDPA_ERR_INVALID_ARG


def test_varlen_workspace_size(lib):
    # per head: total_q rounded up to 64, 192 rows per sequence and 128 rows of
    # slack, two floats each, the whole rounded up to 256 bytes
    def expect(b, h, total_q):
        rows = ((total_q + 63) // 64) * 64 + 192 * b + 128
        return (h * rows * 8 + 255) // 256 * 256
    for b, h, tq in ((1, 1, 1), (3, 4, 1000), (16, 32, 65536), (0, 2, 0)):
        assert lib.sdpa_bwd_varlen_workspace_size(b, h, tq) == expect(b, h, tq)
    assert lib.sdpa_bwd_varlen_workspace_size(-1, 2, 10) == 0
    assert lib.sdpa_bwd_varlen_workspace_size(2, 2, -10) == 0
    # the default backward at d_qk <= 128 adds its fp32 dQ accumulator over
    # the packed rows (per head, rows padded to 128); deterministic and d_qk =
    # 192 need the statistics alone
    for b, h, tq in ((1, 1, 1), (3, 4, 1000), (16, 32, 65536)):
        for d in (64, 128):
            acc = h * ((tq + 127) // 128) * 128 * d * 4
            assert lib.sdpa_bwd_varlen_workspace_size_ex(b, h, tq, d, 0) == expect(b, h, tq) + acc
            assert lib.sdpa_bwd_varlen_workspace_size_ex(b, h, tq, d, 1) == expect(b, h, tq)
        assert lib.sdpa_bwd_varlen_workspace_size_ex(b, h, tq, 192, 0) == expect(b, h, tq)
    assert lib.sdpa_bwd_varlen_workspace_size_ex(2, 2, 10, 96, 0) == 0
    assert lib.sdpa_bwd_varlen_workspace_size_ex(-1, 2, 10, 64, 0) == 0
    assert lib.sdpa_bwd_varlen_workspace_size_ex(2, 1 << 25, 10, 64, 0) == 0


def test_varlen_arguments_validated_before_any_device_work(lib):
    P = ctypes.c_void_p(16)  # never dereferenced: the calls fail validation first
    S = ctypes.c_void_p(64)  # a 4-byte-aligned "seqstart"

    def fwd(b=2, h=4, h_kv=4, tq=100, tk=100, mq=64, mk=64, d=64, p=0.0, sq=S, sk=S):
        return lib.sdpa_fwd_varlen(b, h, h_kv, tq, tk, mq, mk, d, d, 0.125, 1, p, 0, 0, 0, sq, sk,
                                   P, P, P, P, P, None)
    assert fwd(sq=None) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(sk=None) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(sq=None, sk=None, tq=0) == _native.SDPA_OK          # empty: a no-op
    assert fwd(tk=0) == _native.SDPA_OK
    assert fwd(mq=0) == _native.SDPA_OK
    assert fwd(sq=ctypes.c_void_p(66)) == _native.SDPA_ERR_MISALIGNED
    assert fwd(h_kv=3) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(d=96) == _native.SDPA_ERR_UNSUPPORTED
    assert fwd(p=0.1, mk=66) == _native.SDPA_ERR_UNSUPPORTED        # max_seqlen_k % 4 with dropout
    assert fwd(tq=-1) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(tq=1 << 40) == _native.SDPA_ERR_UNSUPPORTED

    def bwd(ws_bytes, b=2, h=4, tq=100):
        return lib.sdpa_bwd_phases_varlen(7, b, h, h, tq, 100, 64, 64, 64, 64, 0.125, 1, 0.0, 0, 0,
                                          0, S, S, P, P, P, P, P, P, P, P, P, ctypes.c_void_p(256),
                                          ws_bytes, None)
    need = lib.sdpa_bwd_varlen_workspace_size(2, 4, 100)
    assert bwd(need - 1) == _native.SDPA_ERR_WORKSPACE
    assert lib.sdpa_bwd_phases_varlen(8, 2, 4, 4, 100, 100, 64, 64, 64, 64, 0.125, 1, 0.0, 0, 0, 0,
                                      S, S, P, P, P, P, P, P, P, P, P, ctypes.c_void_p(256), need,
                                      None) == _native.SDPA_ERR_INVALID_ARG   # unknown phase bit


def test_alibi_arguments_validated_before_any_device_work(lib):
    P = ctypes.c_void_p(16)

    def fwd(slopes, stride, b=2, h=4):
        return lib.sdpa_fwd_ex(b, h, h, 64, 64, 64, 64, 0.125, -1, 0, 0, slopes, stride, None, None,
                               0.0, 0, 0, 0, P, P, P, None, P, P, None)
    assert fwd(ctypes.c_void_p(18), 0) == _native.SDPA_ERR_MISALIGNED
    assert fwd(ctypes.c_void_p(64), -1) == _native.SDPA_ERR_INVALID_ARG
    assert fwd(ctypes.c_void_p(64), 3) == _native.SDPA_ERR_INVALID_ARG   # 0 < stride < h
    assert fwd(ctypes.c_void_p(64), 1 << 40) == _native.SDPA_ERR_INVALID_ARG
    # dropout keep bits drawn beforehand, and a forward's record of them, must
    # be 4-byte aligned
    st = lib.sdpa_fwd_ex(2, 4, 4, 64, 64, 64, 64, 0.125, -1, 0, 0, None, 0, ctypes.c_void_p(66), None,
                         0.1, 0, 0, 0, P, P, P, None, P, P, None)
    assert st == _native.SDPA_ERR_MISALIGNED
    st = lib.sdpa_fwd_ex(2, 4, 4, 64, 64, 64, 64, 0.125, -1, 0, 0, None, 0, None, ctypes.c_void_p(66),
                         0.1, 0, 0, 0, P, P, P, None, P, P, None)
    assert st == _native.SDPA_ERR_MISALIGNED


def test_keep_bit_record_arguments_validated_before_any_device_work(lib):
    P = ctypes.c_void_p(1 << 20)

    def fwd(keep_in, keep_out, skv=64, p=0.1):
        return lib.sdpa_fwd_ex(1, 2, 2, 64, skv, 64, 64, 0.125, -1, 0, 0, None, 0, keep_in, keep_out,
                               p, 0, 0, 0, P, P, P, None, P, P, None)
    # a record needs whole 32-key words per row, and cannot come with input bits
    assert fwd(None, P, skv=68) == _native.SDPA_ERR_UNSUPPORTED
    assert fwd(P, P) == _native.SDPA_ERR_INVALID_ARG


def test_grouped_workspace_size(lib):
    """sdpa_bwd_workspace_size_gqa: the ungrouped bytes, plus for a large group
    on few key tiles one counter per tile (rounded to 256 bytes) and fp32
    partial rows for each split (the largest divisor of the group not above
    ceil(8 * 152 / tiles))."""
    base = lib.sdpa_bwd_workspace_size(1, 32, 16384, 16384, 128, 128)
    assert lib.sdpa_bwd_workspace_size_gqa(1, 32, 32, 16384, 16384, 128, 128) == base
    # MQA: 128 key tiles -> want ceil(1216 / 128) = 10 -> split 8
    tiles, split = 128, 8
    extra = 512 + tiles * split * 128 * 256 * 4
    assert lib.sdpa_bwd_workspace_size_gqa(1, 32, 1, 16384, 16384, 128, 128) == base + extra
    # GQA 8 groups of 4 K/V heads: 512 tiles -> want 3 -> split 2
    tiles, split = 512, 2
    extra = 2048 + tiles * split * 128 * 256 * 4
    assert lib.sdpa_bwd_workspace_size_gqa(1, 32, 4, 16384, 16384, 128, 128) == base + extra
    # many tiles: no split
    assert lib.sdpa_bwd_workspace_size_gqa(8, 32, 8, 8192, 8192, 128, 128) == \
        lib.sdpa_bwd_workspace_size(8, 32, 8192, 8192, 128, 128)
    assert lib.sdpa_bwd_workspace_size_gqa(1, 32, 3, 128, 128, 128, 128) == 0  # 3 does not divide 32
