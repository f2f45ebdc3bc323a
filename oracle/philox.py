"""Philox4x32-10 and the dropout keep rule, written out plainly in numpy.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module. The
product path never does.

Philox4x32-10 follows the published algorithm (Salmon, Moraes, Dror, Shaw,
"Parallel random numbers: as easy as 1, 2, 3", SC'11): a 128-bit counter
(four 32-bit words) and a 64-bit key (two words) go through ten rounds; each
round multiplies counter words 0 and 2 by the two round multipliers, keeps the
high and low halves of the 64-bit products, and mixes them with the other
two counter words and the key; between rounds the key is bumped by the two
Weyl constants.

Which element draws which number (the pages name no generator; see the
CK tile fmha_bwd_kernel.hpp dropout arguments ``drop_seed`` / ``drop_offset``
and PyTorch cudnn MHA.cpp's seed/offset tensors for the parameters that exist):

* key = (low 32 bits of seed, high 32 bits of seed)
* linear element index L = ((b * H + h) * S_q + i) * S_kv + j
* group g = L // 4, word w = L % 4
* counter = (low32(offset), high32(offset), low32(g), high32(g))
* r = output word w of Philox4x32-10(counter, key)
* element kept iff r >= T, with T = floor(p * 2**32) computed in double.

One 128-bit Philox output therefore feeds four consecutive elements.
"""
from __future__ import annotations

import math

import numpy as np

# Round multipliers and Weyl key increments of Philox4x32 (Salmon et al., SC'11).
PHILOX_M0 = 0xD2511F53
PHILOX_M1 = 0xCD9E8D57
PHILOX_W0 = 0x9E3779B9
PHILOX_W1 = 0xBB67AE85
PHILOX_ROUNDS = 10
ELEMS_PER_CALL = 4

_MASK32 = np.uint64(0xFFFFFFFF)


def _mulhilo(a: int, b: np.ndarray) -> tuple[np.ndarray, np.ndarray]:
    """High and low 32-bit halves of the 64-bit product a*b (b uint64 holding u32)."""
    prod = np.uint64(a) * b
    return prod >> np.uint64(32), prod & _MASK32


def philox4x32_10(counter: np.ndarray, key: tuple[int, int]) -> np.ndarray:
    """Philox4x32-10 on an array of counters.

    counter: integer array [..., 4] of 32-bit words (c0, c1, c2, c3).
    key: (k0, k1) 32-bit words.
    Returns uint32 array [..., 4] with the four output words.
    """
    c = np.asarray(counter, dtype=np.uint64) & _MASK32
    c0, c1, c2, c3 = c[..., 0], c[..., 1], c[..., 2], c[..., 3]
    k0, k1 = int(key[0]) & 0xFFFFFFFF, int(key[1]) & 0xFFFFFFFF
    for rnd in range(PHILOX_ROUNDS):
        if rnd > 0:
            k0 = (k0 + PHILOX_W0) & 0xFFFFFFFF
            k1 = (k1 + PHILOX_W1) & 0xFFFFFFFF
        hi0, lo0 = _mulhilo(PHILOX_M0, c0)
        hi1, lo1 = _mulhilo(PHILOX_M1, c2)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint64(k0), lo1, hi0 ^ c3 ^ np.uint64(k1), lo0)
    return np.stack([c0, c1, c2, c3], axis=-1).astype(np.uint32)


def drop_threshold(p: float) -> int:
    """T = floor(p * 2**32): an element is dropped iff its 32-bit draw is < T."""
    if not (0.0 <= p < 1.0):
        raise ValueError("dropout probability must lie in [0, 1)")
    return int(math.floor(float(p) * 4294967296.0))


def random_words(lin: np.ndarray, seed: int, offset: int) -> np.ndarray:
    """The 32-bit draw of each linear element index in ``lin`` (uint64 array)."""
    lin = np.asarray(lin, dtype=np.uint64)
    g = lin >> np.uint64(2)
    w = (lin & np.uint64(3)).astype(np.int64)
    ctr = np.stack(
        [
            np.full_like(g, offset & 0xFFFFFFFF),
            np.full_like(g, (offset >> 32) & 0xFFFFFFFF),
            g & _MASK32,
            g >> np.uint64(32),
        ],
        axis=-1,
    )
    out = philox4x32_10(ctr, (seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF))
    return np.take_along_axis(out, w[..., None], axis=-1)[..., 0]


def keep_mask(B: int, H: int, S_q: int, S_kv: int, p: float, seed: int, offset: int,
              b: int, h: int, rows: np.ndarray | None = None) -> np.ndarray:
    """Boolean keep mask [len(rows), S_kv] of the (b, h) slice (rows default: all)."""
    if rows is None:
        rows = np.arange(S_q)
    rows = np.asarray(rows, dtype=np.uint64)
    j = np.arange(S_kv, dtype=np.uint64)
    lin = ((np.uint64(b) * np.uint64(H) + np.uint64(h)) * np.uint64(S_q) + rows[:, None]) \
        * np.uint64(S_kv) + j[None, :]
    if p == 0.0:
        return np.ones(lin.shape, dtype=bool)
    return random_words(lin, seed, offset) >= np.uint32(drop_threshold(p))


def packed_mask_words(B: int, H: int, S_q: int, S_kv: int, p: float, seed: int,
                      offset: int) -> np.ndarray:
    """Keep bits of the whole problem packed little-endian into uint32 words:
    bit (L % 32) of word L // 32 is element L's keep flag (L as above)."""
    total = B * H * S_q * S_kv
    lin = np.arange(total, dtype=np.uint64)
    keep = random_words(lin, seed, offset) >= np.uint32(drop_threshold(p))
    pad = (-total) % 32
    keep = np.concatenate([keep, np.zeros(pad, dtype=bool)]).reshape(-1, 32)
    weights = (np.uint64(1) << np.arange(32, dtype=np.uint64))
    return (keep.astype(np.uint64) * weights).sum(axis=1).astype(np.uint32)
