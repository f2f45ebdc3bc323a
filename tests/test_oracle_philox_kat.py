"""The oracle's Philox4x32-10 against the generator's published known-answer
vectors (tests/golden/philox4x32_10_kat.txt: Salmon et al., SC'11, the
vectors distributed with the authors' Random123 library). A wrong round
constant, key schedule, word order or multiplier fails them."""
import os

import numpy as np

from oracle import philox

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.txt")


def kat_rows():
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield [int(w, 16) for w in line.split()]


def test_philox4x32_10_known_answers():
    rows = list(kat_rows())
    assert len(rows) == 3
    for r in rows:
        ctr, key, want = r[0:4], r[4:6], r[6:10]
        got = philox.philox4x32_10(np.array([ctr], dtype=np.uint32), (key[0], key[1]))
        assert [int(x) for x in got.reshape(-1)] == want, (ctr, key)


def test_zero_seed_offset_block_zero_is_the_first_vector():
    """Element L = 0..3 of a problem with seed 0 and offset 0 draws counter
    (0, 0, 0, 0) under key (0, 0): the first known-answer vector, word L."""
    first = next(kat_rows())
    words = philox.random_words(np.arange(4, dtype=np.uint64), 0, 0)
    assert [int(w) for w in words] == first[6:10]
