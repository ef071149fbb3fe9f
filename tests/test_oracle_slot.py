"""Pins for the oracle's noise rows, slot read, gated resample and ask_if gating."""
import numpy as np
import pytest
import torch

from oracle import slot_read, slot_noise_rows, noise_tokens, ask_if_fires, bf16_round


def _one(z_draws, n=None, samples=4, gate=0.1, lse=None):
    z = np.asarray(z_draws, dtype=np.float64)[None]          # [1, R, K]
    S, R, K = z.shape
    n = K if n is None else n
    lse = np.zeros((1, R)) if lse is None else np.asarray(lse, dtype=np.float64)[None]
    return slot_read(z, lse, np.array([n]), samples, gate)


@pytest.mark.parametrize("K", [2, 5, 26])
def test_equal_label_logits_give_ln_k(K):
    out = _one(np.full((4, K), 0.37))
    assert out["h_slot"][0] == pytest.approx(np.log(K), abs=1e-14)
    np.testing.assert_allclose(out["q_avg"][0, :K], 1.0 / K, atol=1e-15)


def test_distribution_is_proper_and_shift_invariant():
    rng = np.random.default_rng(0)
    z = rng.standard_normal((4, 26)) * 2
    a = _one(z, lse=rng.standard_normal(4))
    b = _one(z + 11.5, lse=rng.standard_normal(4) + 3)
    q = a["q_avg"][0]
    assert np.all(q >= 0) and q.sum() == pytest.approx(1.0, abs=1e-14)
    np.testing.assert_allclose(a["q_avg"], b["q_avg"], atol=1e-14)
    assert a["chosen"][0] == b["chosen"][0]


def test_samples_one_reads_once():
    z = np.random.default_rng(1).standard_normal((4, 26))
    out = _one(z, samples=1)
    assert out["n_reads"][0] == 1 and out["resampled"][0] == 0
    again = _one(z, samples=1)
    assert np.array_equal(out["q_avg"], again["q_avg"])


def test_gate_fires_strictly_above_threshold():
    # two labels, logit gap g: H(g) decreases in g; bisect for H == 0.1
    def h_of(g):
        p = 1 / (1 + np.exp(-g))
        return -(p * np.log(p) + (1 - p) * np.log(1 - p))
    lo, hi = 0.0, 20.0
    for _ in range(200):
        mid = 0.5 * (lo + hi)
        lo, hi = (mid, hi) if h_of(mid) > 0.1 else (lo, mid)
    above = _one(np.tile([lo - 1e-3, 0.0], (4, 1)))
    below = _one(np.tile([hi + 1e-3, 0.0], (4, 1)))
    assert above["h_draw"][0, 0] > 0.1 and above["resampled"][0] == 1 and above["n_reads"][0] == 4
    assert below["h_draw"][0, 0] < 0.1 and below["resampled"][0] == 0 and below["n_reads"][0] == 1


def test_average_uses_exactly_four_reads():
    # read 0 spreads its mass evenly over labels 0..3 (entropy ln 4 > 0.1, so the gate
    # fires); reads 1..3 put (almost) all mass on labels 4, 5, 4.  The mean of exactly
    # these four reads is (1/16 x4, 1/2, 1/4) with entropy 2 ln 2.
    z = np.full((4, 6), -60.0)
    z[0, :4] = 60.0
    z[1, 4] = z[2, 5] = z[3, 4] = 60.0
    out = _one(z)
    assert out["resampled"][0] == 1 and out["n_reads"][0] == 4
    np.testing.assert_allclose(out["q_avg"][0], [1 / 16] * 4 + [0.5, 0.25], atol=1e-12)
    assert out["h_slot"][0] == pytest.approx(2 * np.log(2), abs=1e-10)
    assert out["chosen"][0] == 4
    # a four-way tie in the average goes to the lowest label index
    z2 = np.full((4, 6), -60.0)
    z2[:, 1:5] = 60.0
    tie = _one(z2)
    assert tie["resampled"][0] == 1 and tie["chosen"][0] == 1


def test_logprobs_are_label_logit_minus_lse():
    z = np.random.default_rng(2).standard_normal((4, 5))
    lse = np.array([3.0, 4.0, 5.0, 6.0])
    out = _one(z, lse=lse)
    np.testing.assert_allclose(out["lp"][0], z - lse[:, None], atol=1e-15)


def test_padding_labels_are_ignored():
    z = np.random.default_rng(3).standard_normal((4, 26))
    a = _one(z, n=5)
    b = _one(z[:, :5], n=5)
    np.testing.assert_allclose(a["q_avg"][0, :5], b["q_avg"][0], atol=1e-15)
    assert a["chosen"][0] == b["chosen"][0]


def test_noise_rows_add_embedding_of_philox_token():
    rng = np.random.default_rng(4)
    V, D = 64, 16
    h = bf16_round(rng.standard_normal((10, D)).astype(np.float32))
    e = bf16_round((rng.standard_normal((V, D)) / 4).astype(np.float32))
    rows, toks = slot_noise_rows(h, e, np.array([2, 7]), np.array([0, 1]), 99, 3, 4, V)
    for s, (row, req) in enumerate([(2, 0), (7, 1)]):
        want_toks = noise_tokens(99, req, 3, 4, 2, V)[:, s]
        np.testing.assert_array_equal(toks[s], want_toks)
        for r in range(4):
            ref = torch.tensor(h[row] + e[want_toks[r]], dtype=torch.float32).to(torch.bfloat16)
            np.testing.assert_array_equal(rows[s * 4 + r], ref.float().numpy())


def test_bf16_round_matches_torch():
    x = np.random.default_rng(5).standard_normal(100000).astype(np.float32) * 37
    x[:4] = [1.0 + 2**-8, 1.0 + 3 * 2**-8, -(1.0 + 2**-8), 0.0]   # exact ties
    ref = torch.tensor(x).to(torch.bfloat16).float().numpy()
    np.testing.assert_array_equal(bf16_round(x), ref)


def test_ask_if():
    assert ask_if_fires(3, 3) and not ask_if_fires(2, 3)


def test_ask_if_select_two_stage_grouping():
    from oracle import ask_if_select
    # 2 requests; stage-1 slots 0 (request 0 group) and 1 (request 1 group), 3 groups;
    # questions q = 3*b + g own stage-2 slot b and ask if group g was chosen
    chosen1 = np.array([2, 0])
    cond_slot = np.array([0, 0, 0, 1, 1, 1])
    cond_value = np.array([0, 1, 2, 0, 1, 2])
    q_owner = np.array([0, 0, 0, 1, 1, 1])
    q_n = np.array([9, 9, 5, 9, 9, 5])
    q_lab = np.full((6, 26), -1)
    for q in range(6):
        q_lab[q, :q_n[q]] = 100 * q + np.arange(q_n[q])
    lab2, n2, fired = ask_if_select(chosen1, cond_slot, cond_value, q_owner, q_lab, q_n, 3)
    assert fired.tolist() == [0, 0, 1, 1, 0, 0]        # exactly one per request
    assert n2.tolist() == [5, 9, 0]                    # slot 2 owned by nobody: not asked
    assert lab2[0, :5].tolist() == [200, 201, 202, 203, 204] and lab2[0, 5] == -1
    assert lab2[1, :9].tolist() == list(range(300, 309))
    assert np.all(lab2[2] == -1)
    # an out-of-range condition slot never fires
    _, _, f2 = ask_if_select(chosen1, np.array([5]), np.array([0]), np.array([0]), q_lab[:1],
                             q_n[:1], 1)
    assert f2.tolist() == [0]


def test_not_asked_slot_is_not_read():
    z = np.random.default_rng(9).standard_normal((1, 4, 26))
    out = slot_read(z, np.zeros((1, 4)), np.array([0]), 4, 0.1)
    assert out["chosen"][0] == -1 and out["n_reads"][0] == 0 and out["resampled"][0] == 0
    assert np.all(out["q_avg"][0] == 0) and out["h_slot"][0] == 0
