"""Pins for the oracle's Philox4x32-10 and noise-token map."""
import os

import numpy as np
import pytest
from scipy import stats

from oracle import philox4x32_10, noise_tokens, seed_key

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "philox_kat.txt")


def _kat():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            v = [int(x, 16) for x in line.split()]
            rows.append((v[0:4], v[4:6], v[6:10]))
    return rows


@pytest.mark.parametrize("ctr,key,want", _kat())
def test_known_answer_vectors(ctr, key, want):
    got = philox4x32_10(np.array(ctr, np.uint32), np.array(key, np.uint32))
    assert [int(x) for x in got] == want


def test_vectorised_matches_scalar():
    rng = np.random.default_rng(5)
    ctr = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64).astype(np.uint32)
    key = rng.integers(0, 2**32, size=(64, 2), dtype=np.uint64).astype(np.uint32)
    batch = philox4x32_10(ctr, key)
    for i in range(64):
        assert np.array_equal(batch[i], philox4x32_10(ctr[i], key[i]))


def test_seed_key_split():
    k = seed_key(0x0123456789ABCDEF)
    assert int(k[0]) == 0x89ABCDEF and int(k[1]) == 0x01234567


def test_noise_tokens_range_and_uniformity():
    V = 1024
    toks = np.concatenate([noise_tokens(7, req, step, 64, 16, V).ravel()
                           for req in range(8) for step in range(8)])
    assert toks.min() >= 0 and toks.max() < V
    counts = np.bincount(toks // 64, minlength=16)
    p = stats.chisquare(counts).pvalue
    assert p > 1e-4


def test_noise_token_is_top_bits_of_word0():
    seed, req, step, V = 123456789012345, 3, 5, 262144
    toks = noise_tokens(seed, req, step, 4, 3, V)
    for r in range(4):
        for s in range(3):
            w0 = philox4x32_10(np.array([req, step, r, s], np.uint32), seed_key(seed))[0]
            assert toks[r, s] == int(w0) >> (32 - 18)


def test_noise_tokens_reject_non_power_of_two():
    with pytest.raises(ValueError):
        noise_tokens(0, 0, 0, 1, 1, 1000)


def test_distinct_counters_distinct_draws():
    toks = noise_tokens(0, 0, 0, 4, 26, 2**32 // 2)
    assert len(np.unique(toks)) == toks.size
