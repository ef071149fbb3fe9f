"""Pins for the oracle's self-conditioning expected embedding and the step loop."""
import numpy as np
from scipy import special

from oracle import selfcond_embed, canvas_update, denoise_loop, bf16_round, lmhead_stats


def _case(M=5, V=120, D=12, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((M, D)), rng.standard_normal((V, D)) / np.sqrt(D),
            rng.standard_normal((V, D)), 1.0 / rng.uniform(0.5, 2, M))


def test_matches_library_softmax_times_table():
    h, w, e, inv_t = _case()
    ref = special.softmax((h @ w.T) * inv_t[:, None], axis=1) @ e
    np.testing.assert_allclose(selfcond_embed(h, w, e, inv_t), ref, atol=1e-12)


def test_equal_logits_give_column_mean():
    h, w, e, _ = _case(seed=1)
    out = selfcond_embed(np.zeros_like(h), w, e, np.ones(h.shape[0]))
    np.testing.assert_allclose(out, np.broadcast_to(e.mean(axis=0), out.shape), atol=1e-12)


def test_dominant_row_gives_its_embedding():
    D, V = 6, 40
    w = np.zeros((V, D))
    w[13, 0] = 1.0
    h = np.zeros((1, D))
    h[0, 0] = 1.0
    e = np.random.default_rng(2).standard_normal((V, D))
    out = selfcond_embed(h, w, e, np.array([500.0]))
    np.testing.assert_allclose(out[0], e[13], atol=1e-12)


def test_linear_in_table():
    h, w, e1, inv_t = _case(seed=3)
    e2 = np.random.default_rng(4).standard_normal(e1.shape)
    a = selfcond_embed(h, w, e1 + 2.5 * e2, inv_t)
    b = selfcond_embed(h, w, e1, inv_t) + 2.5 * selfcond_embed(h, w, e2, inv_t)
    np.testing.assert_allclose(a, b, atol=1e-11)


def test_canvas_update_rows():
    rng = np.random.default_rng(5)
    h0 = bf16_round(rng.standard_normal((4, 8)).astype(np.float32))
    esc = rng.standard_normal((4, 8)) * 0.3
    emb = bf16_round(rng.standard_normal((10, 8)).astype(np.float32))
    out = canvas_update(h0, esc, emb, np.array([0, 7, 0, 2]), np.array([0, 1, 0, 1]))
    np.testing.assert_array_equal(out[1], bf16_round(h0[1] + emb[7]))
    np.testing.assert_array_equal(out[3], bf16_round(h0[3] + emb[2]))
    np.testing.assert_array_equal(out[0], bf16_round(h0[0] + esc[0].astype(np.float32)))


def test_loop_commits_progress_and_leave_candidates():
    rng = np.random.default_rng(6)
    C, V, D = 16, 64, 8
    h0 = bf16_round(rng.standard_normal((C, D)).astype(np.float32))
    w = bf16_round((rng.standard_normal((V, D)) / np.sqrt(D)).astype(np.float32))
    e = bf16_round((rng.standard_normal((V, D)) / np.sqrt(D)).astype(np.float32))
    inv_t = (1.0 / rng.uniform(0.5, 2, C)).astype(np.float32)
    steps, committed, tokens = denoise_loop(h0, w, e, inv_t, np.ones(C, bool), 0.5 * np.log(V) * 2.2, 5)
    seen = np.zeros(C, bool)
    for st in steps:
        new = st["commit"].astype(bool)
        assert st["n_commit"] >= 1
        assert not np.any(new & seen)        # committed rows never re-enter
        seen |= new
    assert np.array_equal(seen, committed)
    # the first step's statistics are those of the unconditioned canvas
    lse, ent, _, arg = lmhead_stats(h0, w, inv_t)
    np.testing.assert_allclose(steps[0]["entropy"], ent)
    for st in steps:
        new = st["commit"].astype(bool)
        np.testing.assert_array_equal(tokens[new], st["tokens"][new])
        np.testing.assert_array_equal(st["tokens"][new], st["argmax"][new])
