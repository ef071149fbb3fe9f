"""Pins for the oracle's entropy-ordered commit."""
import itertools

import numpy as np
import pytest

from oracle import commit


def _brute(ent, cand, gamma):
    """Largest candidate subset that is closed under 'more confident' (entropy, then
    position) and either has one element or total entropy <= gamma."""
    idx = [i for i in range(len(ent)) if cand[i]]
    rank = {i: (ent[i], i) for i in idx}
    best = set()
    for k in range(len(idx) + 1):
        for sub in itertools.combinations(idx, k):
            s = set(sub)
            closed = all(rank[j] >= rank[i] or j in s for i in s for j in idx)
            if not closed:
                continue
            if len(s) > 1 and sum(ent[i] for i in s) > gamma:
                continue
            if len(s) > len(best):
                best = s
    return best


@pytest.mark.parametrize("seed", range(40))
def test_matches_brute_force(seed):
    rng = np.random.default_rng(seed)
    C = 9
    ent = np.round(rng.uniform(0, 3, C), 1)   # rounding creates ties
    cand = rng.random(C) < 0.7
    gamma = float(rng.uniform(0, 8))
    arg = rng.integers(0, 1000, C)
    cm, tk, n = commit(ent[None], arg[None], cand[None].astype(np.uint8), np.array([gamma]))
    want = _brute(ent, cand, gamma)
    assert set(np.nonzero(cm[0])[0]) == want
    assert n[0] == len(want)
    for i in range(C):
        assert tk[0, i] == (arg[i] if i in want else -1)


def test_invariants_and_monotone_in_gamma():
    rng = np.random.default_rng(100)
    ent = rng.uniform(0, 12, (1, 256))
    cand = np.ones((1, 256), np.uint8)
    arg = rng.integers(0, 262144, (1, 256))
    prev = 0
    for gamma in np.linspace(0, 200, 41):
        cm, _, n = commit(ent, arg, cand, np.array([gamma]))
        order = np.lexsort((np.arange(256), ent[0]))
        k = int(n[0])
        assert k >= 1 and k >= prev
        assert set(np.nonzero(cm[0])[0]) == set(order[:k])
        if k > 1:
            assert ent[0, order[:k]].sum() <= gamma
        if k < 256:
            assert ent[0, order[:k + 1]].sum() > gamma
        prev = k


def test_threshold_is_inclusive_and_first_always_accepted():
    ent = np.array([[1.0, 2.0, 3.0]])
    arg = np.array([[5, 6, 7]])
    cand = np.ones((1, 3), np.uint8)
    _, _, n = commit(ent, arg, cand, np.array([3.0]))
    assert n[0] == 2
    _, _, n = commit(ent, arg, cand, np.array([0.5]))
    assert n[0] == 1


def test_no_candidates_commits_nothing():
    cm, tk, n = commit(np.ones((2, 4)), np.zeros((2, 4), int), np.zeros((2, 4), np.uint8),
                       np.array([9.0, 9.0]))
    assert n.tolist() == [0, 0] and cm.sum() == 0 and np.all(tk == -1)
