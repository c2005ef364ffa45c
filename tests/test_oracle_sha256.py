"""Pins of the oracle's SHA-256 against the FIPS 180-4 example digests and hashlib."""

import hashlib
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def test_fips180_examples():
    n = 0
    with open(os.path.join(GOLDEN, "sha256_fips180.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip("\n"):
                continue
            msg, digest = line.rstrip("\n").split("\t")
            assert oracle.sha256(msg.encode()).hex() == digest, msg
            n += 1
    assert n == 3


def test_matches_hashlib_across_padding_boundaries():
    rng = np.random.default_rng(3)
    for n in list(range(0, 200)) + [1000, 4096, 65537]:
        data = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert oracle.sha256(data) == hashlib.sha256(data).digest(), n
