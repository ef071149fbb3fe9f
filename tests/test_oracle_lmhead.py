"""Pins for the oracle's lm-head -> log-softmax -> entropy statistics."""
import numpy as np
from scipy import special, stats

from oracle import lmhead_stats, label_logits


def _case(M=7, V=300, D=40, seed=0):
    rng = np.random.default_rng(seed)
    h = rng.standard_normal((M, D))
    w = rng.standard_normal((V, D)) / np.sqrt(D)
    inv_t = 1.0 / rng.uniform(0.5, 2.0, M)
    return h, w, inv_t


def test_lse_matches_scipy_logsumexp():
    h, w, inv_t = _case()
    lse, _, _, _ = lmhead_stats(h, w, inv_t)
    z = (h @ w.T) * inv_t[:, None]
    np.testing.assert_allclose(lse, special.logsumexp(z, axis=1), rtol=0, atol=1e-12)


def test_entropy_matches_scipy_entropy():
    h, w, inv_t = _case(seed=1)
    _, ent, _, _ = lmhead_stats(h, w, inv_t)
    z = (h @ w.T) * inv_t[:, None]
    p = special.softmax(z, axis=1)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-12)
    np.testing.assert_allclose(ent, stats.entropy(p, axis=1), rtol=0, atol=1e-10)


def test_uniform_logits_give_ln_v():
    for V in (1024, 262144 // 64):
        h = np.zeros((3, 16))
        w = np.random.default_rng(2).standard_normal((V, 16))
        lse, ent, maxz, arg = lmhead_stats(h, w, np.ones(3))
        np.testing.assert_allclose(ent, np.log(V), atol=1e-12)
        np.testing.assert_allclose(lse, np.log(V), atol=1e-12)
        assert np.all(maxz == 0) and np.all(arg == 0)


def test_argmax_ties_go_to_lowest_id_and_ignore_temperature():
    rng = np.random.default_rng(3)
    w = rng.standard_normal((50, 8))
    h = rng.standard_normal((4, 8))
    best = np.argmax(h @ w.T, axis=1)
    w2 = np.concatenate([w, w[best]], axis=0)       # duplicates at higher ids
    w2 = np.concatenate([w2[50:], w2[:50]], axis=0)  # ... now at lower ids
    _, _, _, arg = lmhead_stats(h, w2, np.ones(4))
    want = [int(np.nonzero(best == best[i])[0][0]) for i in range(4)]
    np.testing.assert_array_equal(arg, want)
    _, _, _, arg_t = lmhead_stats(h, w2, np.full(4, 3.7))
    np.testing.assert_array_equal(arg_t, arg)


def test_dominant_logit_gives_near_zero_entropy():
    h = np.zeros((1, 4))
    h[0, 0] = 1.0
    w = np.zeros((100, 4))
    w[37, 0] = 1.0
    lse, ent, maxz, arg = lmhead_stats(h, w, np.array([200.0]))
    assert arg[0] == 37 and maxz[0] == 200.0
    assert ent[0] < 1e-70


def test_label_logits_are_gathered_full_logits():
    h, w, inv_t = _case(M=3, V=200, seed=4)
    ids = np.array([[5, 7, 199, -1], [0, 1, -1, -1], [10, 20, 30, 40]])
    n = np.array([3, 2, 4])
    zl = label_logits(h, w, inv_t, ids, n)
    z = (h @ w.T) * inv_t[:, None]
    lse, _, _, _ = lmhead_stats(h, w, inv_t)
    logp = special.log_softmax(z, axis=1)
    for s in range(3):
        np.testing.assert_allclose(zl[s, :n[s]] - lse[s], logp[s, ids[s, :n[s]]], atol=1e-12)
        assert np.all(np.isnan(zl[s, n[s]:]))
