"""Pin the oracle's Philox4x32-10 to an independent implementation.

PyTorch ships its Philox engine as a C++ source header
(ATen/core/PhiloxRNGEngine.h). ``at::philox_engine(seed, subsequence, offset)``
puts the key at (low, high) of seed, counter words 0-1 at offset and words 2-3
at subsequence; its first four draws are the four output words of one
Philox4x32-10 block. This test compiles that header on the host and compares.
"""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

from oracle import philox

HEADER_DIR = os.path.join(os.path.dirname(torch.__file__), "include")

PROGRAM = r"""
#include <ATen/core/PhiloxRNGEngine.h>
#include <cstdio>
#include <cstdint>
int main() {
  unsigned long long seed, sub, off;
  while (std::scanf("%llu %llu %llu", &seed, &sub, &off) == 3) {
    at::philox_engine e(seed, sub, off);
    uint32_t a = e(), b = e(), c = e(), d = e();
    std::printf("%u %u %u %u\n", a, b, c, d);
  }
  return 0;
}
"""


@pytest.fixture(scope="module")
def torch_philox(tmp_path_factory):
    if shutil.which("g++") is None or not os.path.exists(
            os.path.join(HEADER_DIR, "ATen", "core", "PhiloxRNGEngine.h")):
        pytest.skip("g++ or the PyTorch Philox header is not available")
    d = tmp_path_factory.mktemp("philox")
    src = d / "p.cpp"
    src.write_text(PROGRAM)
    exe = d / "p"
    subprocess.run(["g++", "-std=c++17", "-O1", "-I", HEADER_DIR, str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    return exe


def test_oracle_philox_matches_torch_header(torch_philox):
    rng = np.random.default_rng(5)
    triples = [(0, 0, 0), (1, 0, 0), (0x1234, 7, 0), (2**64 - 1, 2**64 - 1, 2**64 - 1),
               (0xDEADBEEFCAFEF00D, 2**32 + 5, 2**33 + 1)]
    triples += [tuple(int(x) for x in rng.integers(0, 2**63, size=3)) for _ in range(300)]
    text = "".join(f"{s} {g} {o}\n" for s, g, o in triples)
    out = subprocess.run([str(torch_philox)], input=text, capture_output=True, text=True,
                         check=True).stdout.split("\n")
    for (seed, sub, off), line in zip(triples, out):
        want = [int(x) for x in line.split()]
        ctr = np.array([off & 0xFFFFFFFF, off >> 32, sub & 0xFFFFFFFF, sub >> 32], dtype=np.uint64)
        got = philox.philox4x32_10(ctr, (seed & 0xFFFFFFFF, seed >> 32))
        assert [int(x) for x in got] == want, (seed, sub, off)


def test_random_words_use_group_of_four(torch_philox):
    """Element L draws word L % 4 of the block whose subsequence is L // 4."""
    seed, offset = 0x1234, 3
    lin = np.array([0, 1, 2, 3, 4, 5, 1023, 2**40 + 6], dtype=np.uint64)
    words = philox.random_words(lin, seed, offset)
    text = "".join(f"{seed} {int(L) // 4} {offset}\n" for L in lin)
    out = subprocess.run([str(torch_philox)], input=text, capture_output=True, text=True,
                         check=True).stdout.split("\n")
    for L, w, line in zip(lin, words, out):
        assert int(w) == int(line.split()[int(L) % 4])
