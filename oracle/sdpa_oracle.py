"""fp64 CPU oracle of fused scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module; the
product path never does, and this module imports nothing from the product.

What it computes is the equation block at the head of CK tile's
``fmha_bwd_kernel.hpp`` (the comment that opens the file, S = Q K^T through
dQ = dS K * scale), with the parameter set of PyTorch cudnn ``MHA.cpp``
``run_cudnn_SDP_fprop`` / ``run_cudnn_SDP_bprop`` (fp32 softmax statistics of
shape [b, h, s_q], BHSD tensors, optional bias, dropout by seed and offset).
Every matrix is materialised; there is no tiling and no online softmax. Matrix
products are numpy ``@`` in float64.

Readings taken where the pages are silent:

* The saved statistic is the natural-log logsumexp of the scaled, biased,
  masked scores, taken before dropout: LSE_i = m_i + ln(sum_j exp(s_ij - m_i)).
* Causal masking is top-left aligned: key j is visible to query i iff j <= i.
* Local windows and the bottom-right alignment follow the parameters of CK
  tile fmha_bwd_kernel.hpp's mask arguments (window_size_left,
  window_size_right, mask_type top-left or bottom-right): with
  off = S_kv - S_q for bottom-right and 0 for top-left, key j is visible to
  query i iff i + off - left <= j <= i + off + right, a negative size leaving
  that side unbounded. Causal is the window (-1, 0); no mask is (-1, -1).
* ALiBi: CK tile fmha_bwd_kernel.hpp reads one slope per (batch, head)
  (alibi_slope_ptr at i_batch * alibi_slope_stride + i_nhead), takes it into
  the log2 domain beside the scale, and aligns the position encoding
  bottom-right when there is no mask, else as the mask is aligned; the form
  of the encoding is not on the page. Reading: the linear distance penalty of
  ALiBi, -slope * |j - i - off| added to the scaled score (not multiplied by
  the scale), off = 0 under a top-left mask and S_kv - S_q otherwise; the
  slopes are constants (no gradient).
* A row with no visible key (possible only through a -inf bias) has P = 0,
  O = 0, LSE = -inf and contributes nothing to any gradient.
* Dropout multiplies P by Z = keep / (1 - p) before the product with V; the
  row sum and LSE are those of P before dropout. The keep bits come from
  ``oracle.philox``.
* D_i = sum_d dO_id * O_id uses the dropout-applied output O, which equals
  sum_j P_ij Z_ij dP_ij; dS = P * (dP * Z - D) with dP = dO V^T.
* dBias has shape [1, H, S_q, S_kv] and is the sum over the batch of dS.
* Grouped K/V heads (GQA / MQA, H_kv < H): query head h reads K/V head
  h // (H / H_kv), so consecutive query heads share one K/V head, as in CK
  tile fmha_bwd_kernel.hpp (the kernel arguments' nhead_ratio_qk, the K and V
  pointers taken at i_nhead / nhead_ratio_qk) and oneDNN sdpa micro.cpp
  (kv_group_size = query heads / KV heads; the query heads of a group add into
  the shared dK / dV). dK and dV of a K/V head are the sums over its group.
  The dropout bits and the bias are indexed by the query head.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from . import philox


@dataclass(frozen=True)
class Problem:
    """Sizes and scalar parameters of one attention call (BHSD layout)."""

    B: int
    H: int
    S_q: int
    S_kv: int
    D_qk: int
    D_v: int
    scale: float
    is_causal: bool = False
    dropout_p: float = 0.0
    seed: int = 0
    offset: int = 0
    H_kv: int = 0  # K/V heads; 0 means H (no grouping)
    # Local window (left, right) around the aligned diagonal, a negative size
    # unbounded; None means (-1, 0) when is_causal, else (-1, -1).
    window: tuple | None = None
    bottom_right: bool = False  # diagonal through (S_q - 1, S_kv - 1), not (0, 0)
    # Index space of the dropout bits: (B', S_q', S_kv', b0) makes element
    # (b, h, i, j) draw the bit of element (b0 + b, h, i, j) of a
    # [B', H, S_q', S_kv'] problem (a packed sequence draws from the padded
    # batch); None means this problem's own shape.
    drop_frame: tuple | None = None
    # ALiBi slopes, [B][H] (nested sequences) or None
    alibi_slopes: tuple | None = None

    def alibi_offset(self) -> int:
        """Diagonal of the ALiBi distance: top-left under a top-left mask."""
        left, right = self.window if self.window is not None else (-1, 0 if self.is_causal else -1)
        masked = left >= 0 or right >= 0
        return 0 if (masked and not self.bottom_right) else self.S_kv - self.S_q

    @property
    def kv_heads(self) -> int:
        return self.H_kv if self.H_kv else self.H

    def kv_head(self, h: int) -> int:
        """K/V head read by query head h."""
        return h // (self.H // self.kv_heads)


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # torch tensor on the CPU
        x = x.detach().to(dtype=__import__("torch").float64).numpy()
    return np.asarray(x, dtype=np.float64)


def visible(prob: Problem, rows: np.ndarray, cols: np.ndarray) -> np.ndarray:
    """Boolean [len(rows), len(cols)]: key j visible to query i (module text)."""
    left, right = prob.window if prob.window is not None else (-1, 0 if prob.is_causal else -1)
    off = prob.S_kv - prob.S_q if prob.bottom_right else 0
    d = np.asarray(cols)[None, :] - np.asarray(rows)[:, None] - off  # offset from the diagonal
    vis = np.ones(d.shape, dtype=bool)
    if left >= 0:
        vis &= d >= -left
    if right >= 0:
        vis &= d <= right
    return vis


def scores(prob: Problem, q_h: np.ndarray, k_h: np.ndarray, bias_h, rows: np.ndarray,
           cols: np.ndarray, slope: float = 0.0) -> np.ndarray:
    """S'' = (Q K^T) * scale + Bias on the (rows, cols) block, -inf where masked.

    CK tile fmha_bwd_kernel.hpp header: S = Q K^T, S' = S * Scale, S'' = S' + Bias.
    """
    s = prob.scale * (q_h[rows] @ k_h[cols].T)
    if bias_h is not None:
        s = s + bias_h[np.ix_(rows, cols)]
    if slope != 0.0:  # ALiBi (module text)
        dist = np.asarray(cols)[None, :] - np.asarray(rows)[:, None] - prob.alibi_offset()
        s = s - slope * np.abs(dist)
    s = np.where(visible(prob, rows, cols), s, -np.inf)
    return s


def softmax_rows(s: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """P = softmax over each row of s, and LSE = ln(sum exp(s)) per row.

    CK tile fmha_bwd_kernel.hpp header: P = Softmax(S''). Rows whose entries are
    all -inf give P = 0 and LSE = -inf.
    """
    m = s.max(axis=1)
    m0 = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m0[:, None])
    l = e.sum(axis=1)
    alive = l > 0
    p = np.where(alive[:, None], e / np.where(alive, l, 1.0)[:, None], 0.0)
    lse = np.where(alive, m0 + np.log(np.where(alive, l, 1.0)), -np.inf)
    return p, lse


def alibi_slope(prob: Problem, b: int, h: int) -> float:
    return 0.0 if prob.alibi_slopes is None else float(prob.alibi_slopes[b][h])


def dropout_scale(prob: Problem, b: int, h: int, rows: np.ndarray, cols: np.ndarray):
    """Z = keep / (1 - p) on the (rows, cols) block, or 1.0 without dropout."""
    if prob.dropout_p == 0.0:
        return 1.0
    fb, fq, fk, b0 = prob.drop_frame or (prob.B, prob.S_q, prob.S_kv, 0)
    keep = philox.keep_mask(fb, prob.H, fq, fk, prob.dropout_p, prob.seed, prob.offset, b0 + b, h,
                            rows)[:, cols]
    return keep.astype(np.float64) / (1.0 - prob.dropout_p)


def forward_head(prob: Problem, b: int, h: int, q, k, v, bias=None, rows=None):
    """O and LSE of the (b, h) slice for the query rows ``rows`` (default: all).

    q, k, v: [B, H, S, D] arrays; bias: [1, H, S_q, S_kv] or None.
    Returns O [len(rows), D_v] and LSE [len(rows)].
    """
    rows = np.arange(prob.S_q) if rows is None else np.asarray(rows)
    cols = np.arange(prob.S_kv)
    hk = prob.kv_head(h)
    q_h, k_h, v_h = _f64(q[b, h]), _f64(k[b, hk]), _f64(v[b, hk])
    bias_h = None if bias is None else _f64(bias[0, h])
    p, lse = softmax_rows(scores(prob, q_h, k_h, bias_h, rows, cols, alibi_slope(prob, b, h)))
    z = dropout_scale(prob, b, h, rows, cols)
    return (p * z) @ v_h, lse


def forward(prob: Problem, q, k, v, bias=None):
    """O [B, H, S_q, D_v] and LSE [B, H, S_q] of the whole problem."""
    o = np.zeros((prob.B, prob.H, prob.S_q, prob.D_v))
    lse = np.zeros((prob.B, prob.H, prob.S_q))
    for b in range(prob.B):
        for h in range(prob.H):
            o[b, h], lse[b, h] = forward_head(prob, b, h, q, k, v, bias)
    return o, lse


def backward_head(prob: Problem, b: int, h: int, q, k, v, do, bias=None, rows=None,
                  cols=None, row_chunk=None):
    """Gradients of the (b, h) slice (h a query head).

    Returns (dQ[rows], dK[cols], dV[cols], dS[rows][:, cols]) with rows / cols
    defaulting to all queries / keys. dQ and dS on a query row need only that
    row; dK and dV of a key sum over every query row, which is taken
    ``row_chunk`` rows at a time when given (to bound memory at long sequence
    lengths) and all at once otherwise.

    CK tile fmha_bwd_kernel.hpp header: dV = P^T dO, dP = dO V^T,
    D = rowsum(dO * O), dS = P * (dP - D), dK = dS^T Q * Scale,
    dQ = dS K * Scale; dropout enters through Z as described in the module text.
    """
    all_rows = np.arange(prob.S_q)
    all_cols = np.arange(prob.S_kv)
    rows = all_rows if rows is None else np.asarray(rows)
    cols = all_cols if cols is None else np.asarray(cols)
    hk = prob.kv_head(h)
    q_h, k_h, v_h, do_h = _f64(q[b, h]), _f64(k[b, hk]), _f64(v[b, hk]), _f64(do[b, h])
    bias_h = None if bias is None else _f64(bias[0, h])

    def grads_of_rows(rr, want_dq):
        p, _ = softmax_rows(scores(prob, q_h, k_h, bias_h, rr, all_cols, alibi_slope(prob, b, h)))
        z = dropout_scale(prob, b, h, rr, all_cols)
        pz = p * z
        o = pz @ v_h
        d = (do_h[rr] * o).sum(axis=1)
        dp = do_h[rr] @ v_h.T
        ds = p * (dp * z - d[:, None])
        dq = prob.scale * (ds @ k_h) if want_dq else None
        return pz, ds, dq

    _, ds_rows, dq = grads_of_rows(rows, True)
    ds_block = ds_rows[:, cols]

    dk = np.zeros((len(cols), prob.D_qk))
    dv = np.zeros((len(cols), prob.D_v))
    if len(cols) == 0:  # no key column asked for: the sums over every row are empty
        return dq, dk, dv, ds_block
    step = prob.S_q if row_chunk is None else int(row_chunk)
    for r0 in range(0, prob.S_q, step):
        rr = all_rows[r0:r0 + step]
        pz, ds, _ = grads_of_rows(rr, False)
        dv += pz[:, cols].T @ do_h[rr]
        dk += prob.scale * (ds[:, cols].T @ q_h[rr])
    return dq, dk, dv, ds_block


def backward(prob: Problem, q, k, v, do, bias=None):
    """dQ [B, H, S_q, D_qk], dK / dV [B, H_kv, S_kv, D] (summed over each K/V
    head's group of query heads) and dBias [1, H, S_q, S_kv] (None without bias)."""
    dq = np.zeros((prob.B, prob.H, prob.S_q, prob.D_qk))
    dk = np.zeros((prob.B, prob.kv_heads, prob.S_kv, prob.D_qk))
    dv = np.zeros((prob.B, prob.kv_heads, prob.S_kv, prob.D_v))
    dbias = None if bias is None else np.zeros((1, prob.H, prob.S_q, prob.S_kv))
    for b in range(prob.B):
        for h in range(prob.H):
            dq[b, h], dk_h, dv_h, ds = backward_head(prob, b, h, q, k, v, do, bias)
            dk[b, prob.kv_head(h)] += dk_h
            dv[b, prob.kv_head(h)] += dv_h
            if dbias is not None:
                dbias[0, h] += ds
    return dq, dk, dv, dbias
