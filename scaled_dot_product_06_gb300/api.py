"""PyTorch-facing binding of the C ABI (same names as include/sdpa.h).

PyTorch provides device memory and the stream; every step of the attention
computation runs in libsdpa.so's kernels. The functions here only check
tensor properties, allocate outputs with torch and pass raw pointers.
"""
from __future__ import annotations

import ctypes
import functools
import math

import torch

from . import _native

_DTYPE_CODE = {torch.bfloat16: _native.SDPA_BF16, torch.float16: _native.SDPA_FP16}


# The current stream's handle without building a torch.cuda.Stream object
# (which costs a few microseconds a call); the public route where the private
# accessor is missing.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream_ptr(stream, t: torch.Tensor) -> int:
    if stream is not None:
        return int(stream.cuda_stream)
    if _raw_stream is not None:
        return int(_raw_stream(t.get_device()))
    return int(torch.cuda.current_stream(t.device).cuda_stream)


def _check_io(name: str, t: torch.Tensor, shape, dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype:
        raise ValueError(f"{name} has dtype {t.dtype}, expected {dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous (BHSD)")


def _ptr(t):
    # an int converts to void* through the functions' argtypes
    return None if t is None else t.data_ptr()


def _window(is_causal, window, bottom_right, alibi_slopes, n_batch, h, dropout_mask=None,
            force=False):
    """(left, right, bottom_right, slopes pointer, slope stride, keep-bits
    pointer) for the *_ex entry points, or None for the plain causal / unmasked
    calls (unless force). alibi_slopes: fp32 CUDA [h] (every batch entry) or
    [n_batch, h]; dropout_mask: the int32 words of sdpa_dropout_mask (or of a
    forward's dropout_mask_out) for the same problem."""
    if (window is None and not bottom_right and alibi_slopes is None and dropout_mask is None
            and not force):
        return None
    if dropout_mask is not None and (not dropout_mask.is_cuda or dropout_mask.dtype != torch.int32
                                     or not dropout_mask.is_contiguous()):
        raise ValueError("dropout_mask must be the contiguous int32 CUDA words of sdpa_dropout_mask")
    left, right = window if window is not None else (-1, 0 if is_causal else -1)
    stride = 0
    if alibi_slopes is not None:
        a = alibi_slopes
        if not a.is_cuda or a.dtype != torch.float32 or not a.is_contiguous():
            raise ValueError("alibi_slopes must be a contiguous fp32 CUDA tensor")
        if tuple(a.shape) == (h,):
            stride = 0
        elif tuple(a.shape) == (n_batch, h):
            stride = h
        else:
            raise ValueError(f"alibi_slopes has shape {tuple(a.shape)}, expected ({h},) or "
                             f"({n_batch}, {h})")
    return int(left), int(right), int(bool(bottom_right)), _ptr(alibi_slopes), stride, _ptr(dropout_mask)


def _mask_out(t, words):
    """A forward's keep-bit record buffer: contiguous int32 CUDA words."""
    if t is None:
        return None
    if not t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous() or t.numel() < words:
        raise ValueError(f"dropout_mask_out must be a contiguous int32 CUDA tensor of at least "
                         f"{words} words")
    return _ptr(t)


def sdpa_fwd(q, k, v, *, scale=None, is_causal=False, dropout_p=0.0, seed=0, offset=0,
             bias=None, out=None, lse=None, stream=None, window=None, bottom_right=False,
             alibi_slopes=None, dropout_mask=None, dropout_mask_out=None):
    """Forward pass. Returns (o [b,h,s_q,d_v], lse fp32 [b,h,s_q]).

    k and v may have fewer heads than q (grouped-query attention): h_kv =
    k.shape[1] must divide h, and query head i reads K/V head i // (h // h_kv).
    window=(left, right) keeps key j visible to query i iff
    i + off - left <= j <= i + off + right (a negative size unbounded), with
    off = s_kv - s_q when bottom_right, else 0; is_causal is window (-1, 0).
    alibi_slopes (fp32 CUDA [h] or [b, h]) adds -slope * |j - i - off_a| to the
    scaled scores, off_a = 0 under a top-left window, else s_kv - s_q.
    dropout_mask_out (int32 CUDA, ceil(b*h*s_q*s_kv/32) words): the forward
    records the dropout keep bits it draws there, for sdpa_bwd's
    dropout_mask (needs s_kv % 32 == 0)."""
    b, h, s_q, d_qk = q.shape
    h_kv, s_kv, d_v = k.shape[1], k.shape[2], v.shape[3]
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("q, k, v must be bf16 or fp16")
    _check_io("q", q, (b, h, s_q, d_qk), dt)
    _check_io("k", k, (b, h_kv, s_kv, d_qk), dt)
    _check_io("v", v, (b, h_kv, s_kv, d_v), dt)
    if bias is not None:
        _check_io("bias", bias, (1, h, s_q, s_kv), torch.float32)
    scale = 1.0 / math.sqrt(d_qk) if scale is None else float(scale)
    if out is None:
        out = torch.empty((b, h, s_q, d_v), dtype=dt, device=q.device)
    if lse is None:
        lse = torch.empty((b, h, s_q), dtype=torch.float32, device=q.device)
    _check_io("out", out, (b, h, s_q, d_v), dt)
    _check_io("lse", lse, (b, h, s_q), torch.float32)
    w = _window(is_causal, window, bottom_right, alibi_slopes, b, h, dropout_mask,
                force=dropout_mask_out is not None)
    if w is None:
        st = _native.lib().sdpa_fwd_gqa(b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, int(bool(is_causal)),
                                        float(dropout_p), int(seed), int(offset), _DTYPE_CODE[dt],
                                        _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(out), _ptr(lse),
                                        _stream_ptr(stream, q))
        _native.check(st, "sdpa_fwd_gqa")
    else:
        rec = _mask_out(dropout_mask_out, (b * h * s_q * s_kv + 31) // 32)
        st = _native.lib().sdpa_fwd_ex(b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, *w, rec,
                                           float(dropout_p), int(seed), int(offset), _DTYPE_CODE[dt],
                                           _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(out),
                                           _ptr(lse), _stream_ptr(stream, q))
        _native.check(st, "sdpa_fwd_ex")
    return out, lse


def sdpa_bwd_workspace_size(b, h, s_q, s_kv, d_qk, d_v, h_kv=None, deterministic=False) -> int:
    """Backward workspace bytes: the row statistics, plus the fp32 dQ
    accumulator of the default backward at d_qk <= 128 (not with
    deterministic=True); with h_kv (grouped K/V heads) the room for splitting
    large groups over several CTAs per key tile is included."""
    return _workspace_size(int(b), int(h), int(h if h_kv is None else h_kv), int(s_q), int(s_kv),
                           int(d_qk), int(d_v), int(bool(deterministic)))


@functools.lru_cache(maxsize=256)
def _workspace_size(b, h, h_kv, s_q, s_kv, d_qk, d_v, deterministic) -> int:
    return int(_native.lib().sdpa_bwd_workspace_size_ex(b, h, h_kv, s_q, s_kv, d_qk, d_v, deterministic))


def sdpa_bwd(q, k, v, o, dout, lse, *, scale=None, is_causal=False, dropout_p=0.0, seed=0,
             offset=0, bias=None, workspace=None, dq=None, dk=None, dv=None, dbias=None,
             stream=None, window=None, bottom_right=False, alibi_slopes=None,
             dropout_mask=None, deterministic=False):
    """Backward pass. Returns (dq, dk, dv, dbias or None); dk and dv have k's
    and v's shapes (with grouped K/V heads, sums over each group).
    deterministic=True runs the deterministic backward (dQ from the
    query-stationary kernel, bitwise reproducible) instead of accumulating dQ
    with fp32 reductions."""
    return sdpa_bwd_phases(_native.SDPA_BWD_ALL, q, k, v, o, dout, lse, scale=scale,
                           is_causal=is_causal, dropout_p=dropout_p, seed=seed, offset=offset,
                           bias=bias, workspace=workspace, dq=dq, dk=dk, dv=dv, dbias=dbias,
                           stream=stream, window=window, bottom_right=bottom_right,
                           alibi_slopes=alibi_slopes, dropout_mask=dropout_mask,
                           deterministic=deterministic)


def sdpa_bwd_phases(phases, q, k, v, o, dout, lse, *, scale=None, is_causal=False, dropout_p=0.0,
                    seed=0, offset=0, bias=None, workspace=None, dq=None, dk=None, dv=None,
                    dbias=None, stream=None, window=None, bottom_right=False, alibi_slopes=None,
                    dropout_mask=None, deterministic=False):
    """The backward phases selected by ``phases`` (SDPA_BWD_* bit mask; the
    SDPA_BWD_DETERMINISTIC bit, or deterministic=True, selects the
    deterministic backward)."""
    deterministic = bool(deterministic) or bool(int(phases) & _native.SDPA_BWD_DETERMINISTIC)
    phases = int(phases) | (_native.SDPA_BWD_DETERMINISTIC if deterministic else 0)
    b, h, s_q, d_qk = q.shape
    h_kv, s_kv, d_v = k.shape[1], k.shape[2], v.shape[3]
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("q, k, v must be bf16 or fp16")
    for name, t, shp in (("q", q, (b, h, s_q, d_qk)), ("k", k, (b, h_kv, s_kv, d_qk)),
                         ("v", v, (b, h_kv, s_kv, d_v)), ("o", o, (b, h, s_q, d_v)),
                         ("dout", dout, (b, h, s_q, d_v))):
        _check_io(name, t, shp, dt)
    _check_io("lse", lse, (b, h, s_q), torch.float32)
    if bias is not None:
        _check_io("bias", bias, (1, h, s_q, s_kv), torch.float32)
    scale = 1.0 / math.sqrt(d_qk) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if bias is not None and dbias is None:
        dbias = torch.empty_like(bias)
    need = sdpa_bwd_workspace_size(b, h, s_q, s_kv, d_qk, d_v, h_kv, deterministic)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    w = _window(is_causal, window, bottom_right, alibi_slopes, b, h, dropout_mask)
    if w is None:
        st = _native.lib().sdpa_bwd_phases_gqa(
            int(phases), b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, int(bool(is_causal)),
            float(dropout_p), int(seed), int(offset), _DTYPE_CODE[dt], _ptr(q), _ptr(k), _ptr(v),
            _ptr(bias), _ptr(o), _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias),
            _ptr(workspace), workspace.numel(), _stream_ptr(stream, q))
        _native.check(st, "sdpa_bwd_phases_gqa")
    else:
        st = _native.lib().sdpa_bwd_phases_ex(
            int(phases), b, h, h_kv, s_q, s_kv, d_qk, d_v, scale, *w, float(dropout_p), int(seed),
            int(offset), _DTYPE_CODE[dt], _ptr(q), _ptr(k), _ptr(v), _ptr(bias), _ptr(o),
            _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(dbias), _ptr(workspace),
            workspace.numel(), _stream_ptr(stream, q))
        _native.check(st, "sdpa_bwd_phases_ex")
    return dq, dk, dv, dbias


def _check_seqstart(name: str, t: torch.Tensor) -> int:
    if not t.is_cuda or t.dtype != torch.int32 or t.dim() != 1 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous 1-D int32 CUDA tensor")
    if t.numel() < 1:
        raise ValueError(f"{name} needs b + 1 entries")
    return t.numel() - 1


def sdpa_fwd_varlen(q, k, v, seqstart_q, seqstart_k, max_seqlen_q, max_seqlen_k, *, scale=None,
                    is_causal=False, dropout_p=0.0, seed=0, offset=0, out=None, lse=None,
                    stream=None, window=None, bottom_right=False, alibi_slopes=None,
                    dropout_mask=None, dropout_mask_out=None):
    """Forward pass over packed variable-length sequences. q [h, total_q, d_qk],
    k [h_kv, total_k, d_qk], v [h_kv, total_k, d_v]; seqstart_q / seqstart_k
    int32 CUDA tensors of b + 1 row offsets (sequence i owns query rows
    seqstart_q[i] .. seqstart_q[i+1] - 1 and the matching key rows).
    Returns (o [h, total_q, d_v], lse fp32 [h, total_q])."""
    h, total_q, d_qk = q.shape
    h_kv, total_k, d_v = k.shape[0], k.shape[1], v.shape[2]
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("q, k, v must be bf16 or fp16")
    b = _check_seqstart("seqstart_q", seqstart_q)
    if _check_seqstart("seqstart_k", seqstart_k) != b:
        raise ValueError("seqstart_q and seqstart_k must have the same length")
    _check_io("q", q, (h, total_q, d_qk), dt)
    _check_io("k", k, (h_kv, total_k, d_qk), dt)
    _check_io("v", v, (h_kv, total_k, d_v), dt)
    scale = 1.0 / math.sqrt(d_qk) if scale is None else float(scale)
    if out is None:
        out = torch.empty((h, total_q, d_v), dtype=dt, device=q.device)
    if lse is None:
        lse = torch.empty((h, total_q), dtype=torch.float32, device=q.device)
    _check_io("out", out, (h, total_q, d_v), dt)
    _check_io("lse", lse, (h, total_q), torch.float32)
    w = _window(is_causal, window, bottom_right, alibi_slopes, b, h, dropout_mask,
                force=dropout_mask_out is not None)
    if w is None:
        st = _native.lib().sdpa_fwd_varlen(
            b, h, h_kv, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), d_qk, d_v, scale,
            int(bool(is_causal)), float(dropout_p), int(seed), int(offset), _DTYPE_CODE[dt],
            _ptr(seqstart_q), _ptr(seqstart_k), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
            _stream_ptr(stream, q))
        _native.check(st, "sdpa_fwd_varlen")
    else:
        rec = _mask_out(dropout_mask_out, (b * h * int(max_seqlen_q) * int(max_seqlen_k) + 31) // 32)
        st = _native.lib().sdpa_fwd_varlen_ex(
            b, h, h_kv, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), d_qk, d_v, scale, *w,
            rec, float(dropout_p), int(seed), int(offset), _DTYPE_CODE[dt], _ptr(seqstart_q),
            _ptr(seqstart_k), _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
            _stream_ptr(stream, q))
        _native.check(st, "sdpa_fwd_varlen_ex")
    return out, lse


def sdpa_bwd_varlen_workspace_size(b, h, total_q, d_qk=None, deterministic=False) -> int:
    """Workspace bytes of the packed backward. Without d_qk: the row
    statistics alone, which run the deterministic backward; with d_qk: the
    bytes of the backward ``deterministic`` selects (the default one at
    d_qk <= 128 adds its fp32 dQ accumulator)."""
    if d_qk is None:
        return int(_native.lib().sdpa_bwd_varlen_workspace_size(b, h, total_q))
    return int(_native.lib().sdpa_bwd_varlen_workspace_size_ex(b, h, total_q, int(d_qk),
                                                               int(bool(deterministic))))


def sdpa_bwd_varlen(q, k, v, o, dout, lse, seqstart_q, seqstart_k, max_seqlen_q, max_seqlen_k, *,
                    scale=None, is_causal=False, dropout_p=0.0, seed=0, offset=0, workspace=None,
                    dq=None, dk=None, dv=None, stream=None, window=None, bottom_right=False,
                    alibi_slopes=None, dropout_mask=None, deterministic=False):
    """Backward pass over packed sequences (layouts as sdpa_fwd_varlen).
    Returns (dq, dk, dv) shaped like q, k, v. deterministic=True runs the
    deterministic backward, as sdpa_bwd."""
    return sdpa_bwd_phases_varlen(_native.SDPA_BWD_ALL, q, k, v, o, dout, lse, seqstart_q,
                                  seqstart_k, max_seqlen_q, max_seqlen_k, scale=scale,
                                  is_causal=is_causal, dropout_p=dropout_p, seed=seed,
                                  offset=offset, workspace=workspace, dq=dq, dk=dk, dv=dv,
                                  stream=stream, window=window, bottom_right=bottom_right,
                                  alibi_slopes=alibi_slopes, dropout_mask=dropout_mask,
                                  deterministic=deterministic)


def sdpa_bwd_phases_varlen(phases, q, k, v, o, dout, lse, seqstart_q, seqstart_k, max_seqlen_q,
                           max_seqlen_k, *, scale=None, is_causal=False, dropout_p=0.0, seed=0,
                           offset=0, workspace=None, dq=None, dk=None, dv=None, stream=None,
                           window=None, bottom_right=False, alibi_slopes=None,
                           dropout_mask=None, deterministic=False):
    """The packed-sequence backward phases selected by ``phases`` (the
    SDPA_BWD_DETERMINISTIC bit, or deterministic=True, selects the
    deterministic backward). A caller-given workspace smaller than the
    default backward's size runs the deterministic one."""
    deterministic = bool(deterministic) or bool(int(phases) & _native.SDPA_BWD_DETERMINISTIC)
    phases = int(phases) | (_native.SDPA_BWD_DETERMINISTIC if deterministic else 0)
    h, total_q, d_qk = q.shape
    h_kv, total_k, d_v = k.shape[0], k.shape[1], v.shape[2]
    dt = q.dtype
    if dt not in _DTYPE_CODE:
        raise ValueError("q, k, v must be bf16 or fp16")
    b = _check_seqstart("seqstart_q", seqstart_q)
    if _check_seqstart("seqstart_k", seqstart_k) != b:
        raise ValueError("seqstart_q and seqstart_k must have the same length")
    for name, t, shp in (("q", q, (h, total_q, d_qk)), ("k", k, (h_kv, total_k, d_qk)),
                         ("v", v, (h_kv, total_k, d_v)), ("o", o, (h, total_q, d_v)),
                         ("dout", dout, (h, total_q, d_v))):
        _check_io(name, t, shp, dt)
    _check_io("lse", lse, (h, total_q), torch.float32)
    scale = 1.0 / math.sqrt(d_qk) if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = sdpa_bwd_varlen_workspace_size(b, h, total_q, d_qk, deterministic)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    w = _window(is_causal, window, bottom_right, alibi_slopes, b, h, dropout_mask)
    if w is None:
        st = _native.lib().sdpa_bwd_phases_varlen(
            int(phases), b, h, h_kv, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), d_qk,
            d_v, scale, int(bool(is_causal)), float(dropout_p), int(seed), int(offset),
            _DTYPE_CODE[dt], _ptr(seqstart_q), _ptr(seqstart_k), _ptr(q), _ptr(k), _ptr(v), _ptr(o),
            _ptr(dout), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
            _stream_ptr(stream, q))
        _native.check(st, "sdpa_bwd_phases_varlen")
    else:
        st = _native.lib().sdpa_bwd_phases_varlen_ex(
            int(phases), b, h, h_kv, total_q, total_k, int(max_seqlen_q), int(max_seqlen_k), d_qk,
            d_v, scale, *w, float(dropout_p), int(seed), int(offset), _DTYPE_CODE[dt],
            _ptr(seqstart_q), _ptr(seqstart_k), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout),
            _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), workspace.numel(),
            _stream_ptr(stream, q))
        _native.check(st, "sdpa_bwd_phases_varlen_ex")
    return dq, dk, dv


def sdpa_dropout_mask(b, h, s_q, s_kv, dropout_p, seed, offset, device="cuda", stream=None,
                      out=None):
    """Packed keep bits as an int32 tensor of ceil(b*h*s_q*s_kv/32) words (into
    ``out`` when given). Passed back as ``dropout_mask``, the attention calls
    read these bits instead of drawing them."""
    words = (b * h * s_q * s_kv + 31) // 32
    bits = torch.empty(max(words, 1), dtype=torch.int32, device=device) if out is None else out
    if out is not None and (out.dtype != torch.int32 or out.numel() < words or not out.is_cuda):
        raise ValueError(f"out must be an int32 CUDA tensor of at least {words} words")
    st = _native.lib().sdpa_dropout_mask(b, h, s_q, s_kv, float(dropout_p), int(seed), int(offset),
                                         _ptr(bits), _stream_ptr(stream, bits))
    _native.check(st, "sdpa_dropout_mask")
    return bits[:words]


def sdpa_device_error(clear: bool = True) -> int:
    """The device error word (synchronises); 0 when every kernel completed."""
    w = ctypes.c_uint32(0)
    st = _native.lib().sdpa_device_error(ctypes.byref(w), int(bool(clear)))
    if st not in (_native.SDPA_OK, _native.SDPA_ERR_DEVICE_TIMEOUT):
        _native.check(st, "sdpa_device_error")
    return int(w.value)


def sdpa_debug_fault(fault: int = 0, wait_limit_ns: int = 0) -> None:
    """Test hook of the C ABI (see include/sdpa.h): fault 1 makes later forward
    launches time out in a bounded wait; sdpa_debug_fault() restores normal operation."""
    _native.check(_native.lib().sdpa_debug_fault(int(fault), int(wait_limit_ns)), "sdpa_debug_fault")


def sdpa_status_string(status: int) -> str:
    return _native.status_string(status)
