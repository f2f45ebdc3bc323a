"""The tile ranges the three kernels walk, restated here from the kernels and
checked against the oracle's visibility rule: every visible (query, key) pair
lies in a tile the kernel processes, and every tile coordinate it loads lies
inside the problem.

* Forward (fwd_kernel.cuh): a CTA owns a pair of 128-row query tiles (with an
  odd number of tiles, tile 0 alone and pairs (1, 2), (3, 4), ...) and walks
  the 128-key tiles from the highest one either query tile sees down to the
  lowest one of tile 0 (of tile 1 when tile 0 sees none); query tile t joins
  the iterations of its own key range.
* dK / dV (bwd_dkdv_kernel.cuh): a CTA owns a 128-key tile and walks the
  query tiles (128 rows, 64 at d_qk = 192) holding a row that sees one of its
  keys.
* dQ (bwd_dq_kernel.cuh): a CTA owns a 128-row query tile and walks the key
  tiles holding a key that one of its rows sees.

The windowed kernels take these ranges from the band [i + lo, i + hi] of
visible keys of row i; the plain kernels (top-left causal or unmasked) from
the closed forms below. These are CPU restatements of the kernels' integer
arithmetic: a change to a kernel's ranges has to be made here too.
"""
import numpy as np
import pytest

import oracle

U = 1 << 30  # an unbounded side of the band
BM = BN = 128


def band(wl, wr, br, S_q, S_kv):
    off = S_kv - S_q if br else 0
    return (-U if wl < 0 else off - wl, U if wr < 0 else off + wr)


def visible(S_q, S_kv, wl, wr, br):
    pr = oracle.Problem(1, 1, S_q, S_kv, 4, 4, 1.0, False, window=(wl, wr), bottom_right=br)
    return oracle.sdpa_oracle.visible(pr, np.arange(S_q), np.arange(S_kv))


def fwd_tiles(S_q, S_kv, lo, hi):
    """(query tile start, key tile) pairs the forward processes."""
    out = []
    n_qt = (S_q + BM - 1) // BM
    odd = n_qt & 1
    for qt in range((n_qt + 1) // 2):
        lone = odd and qt == 0
        q0 = (max(2 * qt - 1, 0) if odd else 2 * qt) * BM
        rng = []
        for t in (0, 1):
            qs = q0 + t * BM
            if (t == 1 and lone) or qs >= S_q:
                rng.append(None)
                continue
            l, h = max(qs + lo, 0), min(min(qs + BM, S_q) - 1 + hi, S_kv - 1)
            rng.append((l // BN, h // BN) if l <= h else None)
        if rng[0] is None and rng[1] is None:
            continue
        khi = max(r[1] for r in rng if r)
        klo = rng[0][0] if rng[0] else rng[1][0]
        for j in range(khi - klo + 1):
            kt = khi - j
            assert 0 <= kt * BN < S_kv
            users = [t for t in (0, 1) if rng[t] and rng[t][0] <= kt <= rng[t][1]]
            assert users, "an iteration without a query tile"
            out += [(q0 + t * BM, kt) for t in users]
    return out


def dkdv_tiles(S_q, S_kv, lo, hi, bm, plain_causal=None):
    out = []
    n_qt = (S_q + bm - 1) // bm
    for kt in range((S_kv + BN - 1) // BN):
        k0 = kt * BN
        if plain_causal is None:
            qlo, qhi = max(k0 - hi, 0), min(min(k0 + BN, S_kv) - 1 - lo, S_q - 1)
            it0 = qlo // bm
            n_per = qhi // bm - it0 + 1 if qlo <= qhi else 0
        else:
            it0 = min(n_qt, k0 // bm) if plain_causal else 0
            n_per = n_qt - it0
        for i in range(n_per):
            q0 = (it0 + i) * bm
            assert 0 <= q0 < S_q
            out.append((q0, bm, kt))
    return out


def dq_tiles(S_q, S_kv, lo, hi, plain_causal=None):
    out = []
    n_kv_all = (S_kv + BN - 1) // BN
    for qt in range((S_q + BM - 1) // BM):
        q0 = qt * BM
        if plain_causal is None:
            l, h = max(q0 + lo, 0), min(min(q0 + BM, S_q) - 1 + hi, S_kv - 1)
            khi = h // BN
            n_kv = khi - l // BN + 1 if l <= h else 0
        else:
            n_kv = min(n_kv_all, (q0 + BM - 1) // BN + 1) if plain_causal else n_kv_all
            khi = n_kv - 1
        for j in range(n_kv):
            kt = khi - j
            assert 0 <= kt * BN < S_kv
            out.append((q0, kt))
    return out


def cover(shape, tiles_q_k, bm=BM):
    cov = np.zeros(shape, dtype=bool)
    for q0, kt in tiles_q_k:
        cov[q0:q0 + bm, kt * BN:kt * BN + BN] = True
    return cov


def check(S_q, S_kv, wl, wr, br):
    vis = visible(S_q, S_kv, wl, wr, br)
    lo, hi = band(wl, wr, br, S_q, S_kv)
    assert not (vis & ~cover(vis.shape, fwd_tiles(S_q, S_kv, lo, hi))).any(), "forward"
    for bm in (128, 64):
        cov = np.zeros_like(vis)
        for q0, b, kt in dkdv_tiles(S_q, S_kv, lo, hi, bm):
            cov[q0:q0 + b, kt * BN:kt * BN + BN] = True
        assert not (vis & ~cov).any(), f"dK/dV, {bm}-row query tiles"
    assert not (vis & ~cover(vis.shape, dq_tiles(S_q, S_kv, lo, hi))).any(), "dQ"


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
def test_plain_ranges_cover_every_visible_pair(S_q, S_kv, causal):
    """The plain kernels: top-left causal (window (-1, 0)) or unmasked."""
    vis = visible(S_q, S_kv, -1, 0 if causal else -1, False)
    lo, hi = -U, (0 if causal else U)  # the forward's plain band
    assert not (vis & ~cover(vis.shape, fwd_tiles(S_q, S_kv, lo, hi))).any()
    for bm in (128, 64):
        cov = np.zeros_like(vis)
        for q0, b, kt in dkdv_tiles(S_q, S_kv, lo, hi, bm, plain_causal=causal):
            cov[q0:q0 + b, kt * BN:kt * BN + BN] = True
        assert not (vis & ~cov).any()
    assert not (vis & ~cover(vis.shape, dq_tiles(S_q, S_kv, lo, hi, plain_causal=causal))).any()


def test_causal_ranges_skip_tiles_above_the_diagonal():
    """The plain causal ranges are tight: no processed tile lies wholly above
    the diagonal (where no key is visible)."""
    S = 1000
    vis = visible(S, S, -1, 0, False)
    for q0, kt in fwd_tiles(S, S, -U, 0) + dq_tiles(S, S, -U, 0, plain_causal=True):
        assert vis[q0:q0 + BM, kt * BN:kt * BN + BN].any()
    for q0, b, kt in dkdv_tiles(S, S, -U, 0, 128, plain_causal=True):
        assert vis[q0:q0 + b, kt * BN:kt * BN + BN].any()


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
