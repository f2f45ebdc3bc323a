"""The tile ranges the kernels walk, taken from the library itself and
checked against the oracle's visibility rule: every visible (query, key) pair
lies in a tile the kernel processes, every tile coordinate lies inside the
problem, and the plain causal ranges skip the tiles wholly above the
diagonal.

sdpa_tile_ranges (a host-only test hook of the C ABI) enumerates the
(query tile, key tile) pairs of each kernel with the functions of
common.cuh that the backward kernels call (key_tiles_of_rows,
key_tiles_plain, query_tiles_of_keys) and whose arithmetic the forward
writes out (query_pair, key_tiles_of_rows, fwd_iters / fwd_tile_iters; the
calls themselves changed its compiled code):

* the forward: a CTA owns a pair of 128-row query tiles (with an odd number
  of tiles, tile 0 alone and pairs (1, 2), (3, 4), ...) and walks the key
  tiles from the highest one either query tile sees down; query tile t joins
  the iterations of its own key range;
* the key/value-stationary backward (dK/dV, fused): a CTA owns a 128-key
  tile and walks the query tiles (128 rows, 64 at d_qk = 192) holding a row
  that sees one of its keys;
* the dQ kernel: a CTA owns a 128-row query tile and walks the key tiles
  holding a key one of its rows sees.

Windows take the band [i + lo, i + hi] of visible keys of row i; the plain
masks (top-left causal or none) closed forms, or the band as well when
`windowed` is set (the kernels' ALiBi instances).
"""
import ctypes

import numpy as np
import pytest

import oracle
from scaled_dot_product_06_gb300 import _native

BM = BN = 128


def tiles(kernel, S_q, S_kv, wl, wr, br, windowed=False, rows=128):
    """(first query row, query rows, key tile) triples from the library."""
    lib = _native.lib()
    n = lib.sdpa_tile_ranges(kernel, S_q, S_kv, wl, wr, int(br), int(windowed), rows, None, 0)
    assert n >= 0
    buf = (ctypes.c_int32 * max(3 * n, 1))()
    assert lib.sdpa_tile_ranges(kernel, S_q, S_kv, wl, wr, int(br), int(windowed), rows,
                                ctypes.addressof(buf), n) == n
    return np.frombuffer(buf, dtype=np.int32, count=3 * n).reshape(n, 3)


def visible(S_q, S_kv, wl, wr, br):
    pr = oracle.Problem(1, 1, S_q, S_kv, 4, 4, 1.0, False, window=(wl, wr), bottom_right=br)
    return oracle.sdpa_oracle.visible(pr, np.arange(S_q), np.arange(S_kv))


def check(S_q, S_kv, wl, wr, br, windowed=False):
    vis = visible(S_q, S_kv, wl, wr, br)
    for kernel, rows in ((0, 128), (1, 128), (1, 64), (2, 128)):
        cov = np.zeros_like(vis)
        t = tiles(kernel, S_q, S_kv, wl, wr, br, windowed, rows)
        for q0, nr, kt in t:
            assert nr == rows and 0 <= q0 < S_q and q0 % rows == 0, (kernel, q0, nr)
            assert 0 <= kt * BN < S_kv, (kernel, kt)
            cov[q0:q0 + nr, kt * BN:kt * BN + BN] = True
        assert len({tuple(x) for x in t}) == len(t), f"kernel {kernel}: a tile pair visited twice"
        assert not (vis & ~cov).any(), f"kernel {kernel} ({rows}-row query tiles) misses a visible pair"


@pytest.mark.parametrize("S_q,S_kv,wl,wr,br", [
    (640, 640, 100, 0, False), (300, 700, -1, 0, True), (700, 300, -1, 0, True),
    (400, 520, 64, 200, False), (384, 384, 0, 0, False), (512, 512, 256, 32, False),
    (333, 1000, 130, 130, True), (700, 700, -1, 0, False), (700, 700, 5000, 5000, False),
    (100, 200, 50, 10, True), (300, 150, 50, 10, True), (7, 64, 50, 10, True),
    (256, 256, 50, 10, True), (1, 1, 0, 0, False), (129, 257, -1, -1, False),
])
def test_windowed_ranges_cover_every_visible_pair(S_q, S_kv, wl, wr, br):
    check(S_q, S_kv, wl, wr, br)


def test_windowed_ranges_on_random_shapes():
    rng = np.random.default_rng(0)
    for _ in range(150):
        S_q, S_kv = (int(v) for v in rng.integers(1, 700, 2))
        wl, wr = (int(v) for v in rng.integers(-1, 300, 2))
        check(S_q, S_kv, wl, wr, bool(rng.integers(0, 2)))


@pytest.mark.parametrize("S_q,S_kv", [(1, 1), (128, 128), (129, 257), (700, 300), (640, 1000),
                                      (383, 383)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("windowed", [False, True])
def test_plain_ranges_cover_every_visible_pair(S_q, S_kv, causal, windowed):
    """The plain masks (top-left causal or none), by the closed forms of the
    plain instances and by the band arithmetic of the ALiBi instances."""
    check(S_q, S_kv, -1, 0 if causal else -1, False, windowed)


@pytest.mark.parametrize("windowed", [False, True])
def test_causal_ranges_skip_tiles_above_the_diagonal(windowed):
    """The plain causal ranges are tight: no processed tile lies wholly above
    the diagonal (where no key is visible)."""
    S = 1000
    vis = visible(S, S, -1, 0, False)
    for kernel, rows in ((0, 128), (1, 128), (1, 64), (2, 128)):
        for q0, nr, kt in tiles(kernel, S, S, -1, 0, False, windowed, rows):
            assert vis[q0:q0 + nr, kt * BN:kt * BN + BN].any(), (kernel, q0, kt)


def test_tile_ranges_hook_rejects_bad_arguments():
    lib = _native.lib()
    assert lib.sdpa_tile_ranges(3, 128, 128, -1, 0, 0, 0, 128, None, 0) == -1
    assert lib.sdpa_tile_ranges(0, 128, 128, -1, 0, 0, 0, 96, None, 0) == -1
    assert lib.sdpa_tile_ranges(0, -1, 128, -1, 0, 0, 0, 128, None, 0) == -1
    assert lib.sdpa_tile_ranges(0, 128, 128, -1, 0, 0, 0, 128, None, 4) == -1
    assert lib.sdpa_tile_ranges(2, 0, 128, -1, 0, 0, 0, 128, None, 0) == 0


def test_packed_statistics_blocks_are_disjoint_and_inside_the_pad():
    """Packed sequences keep their softmax statistics (and D) in one block per
    sequence: sequence b's block starts at round_up(start_b, 64) + 192 b
    (common.cuh packed_stat_row) and spans its query rows rounded up to whole
    128-row tiles. The blocks must not overlap and must fit in
    packed_stat_pad(rows, n) = round_up(rows, 64) + 192 n + 128 rows, the size
    the backward workspace query reserves per head, for any lengths."""
    def stat_row(start, b):
        return (start + 63) // 64 * 64 + 192 * b

    def pad(rows, n):
        return (rows + 63) // 64 * 64 + 192 * n + 128

    rng = np.random.default_rng(5)
    cases = [[1], [128], [129, 1, 0, 255], [0, 0, 0], [64] * 9, [63, 65, 127, 129]]
    cases += [list(rng.integers(0, 700, int(rng.integers(1, 40)))) for _ in range(300)]
    for lens in cases:
        starts = np.concatenate([[0], np.cumsum(lens)])
        rows = int(starts[-1])
        end_prev = 0
        for b, n in enumerate(lens):
            first = stat_row(int(starts[b]), b)
            size = (int(n) + BM - 1) // BM * BM
            assert first >= end_prev, (lens, b)
            end_prev = first + size
            assert end_prev <= pad(rows, len(lens)), (lens, b)
