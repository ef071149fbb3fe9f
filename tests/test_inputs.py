"""The seeded input generator: reproducible, bf16-valued, shapes as the configs state."""
import numpy as np

from structured_slot_reads_gb300 import configs, inputs


def test_reproducible_and_bf16_valued():
    a = inputs.hidden(8, 64, seed=3)
    b = inputs.hidden(8, 64, seed=3)
    assert np.array_equal(a, b)
    assert np.array_equal(inputs.to_bf16(a), a)
    assert not np.array_equal(a, inputs.hidden(8, 64, seed=4))


def test_weights_scale_and_temperature_range():
    w, e = inputs.weights(4096, 256, seed=0)
    assert abs(w.std() - 1 / 16) < 2e-3 and abs(e.std() - 1 / 16) < 2e-3
    assert not np.array_equal(w, e)
    it = inputs.inv_temperature(10000, seed=1)
    assert it.dtype == np.float32 and it.min() >= 0.5 - 1e-6 and it.max() <= 2.0 + 1e-6


def test_redraw_changes_only_given_rows():
    h = inputs.hidden(6, 32, seed=0)
    h2 = inputs.redraw_rows(h, [1, 4], seed=0, attempt=1)
    assert np.array_equal(h[[0, 2, 3, 5]], h2[[0, 2, 3, 5]])
    assert not np.array_equal(h[1], h2[1]) and not np.array_equal(h[4], h2[4])


def test_slot_table_and_candidates():
    shp = configs.SINGLE_READ
    row, req, lab, n = inputs.slot_table(configs.scaled(shp, V=4096), seed=0)
    assert list(n) == [2, 26, 5] and list(row) == [61, 125, 189]
    for s in range(3):
        ids = lab[s, :n[s]]
        assert len(set(ids.tolist())) == n[s] and ids.min() >= 0 and ids.max() < 4096
        assert np.all(lab[s, n[s]:] == -1)
    cand = inputs.candidates(shp, row)
    assert cand.sum() == 3 and cand[0, 125] == 1
    assert inputs.candidates(configs.FULL_CANVAS).sum() == 256


def test_paged_layout_round_trip():
    shp = configs.scaled(configs.MIXED_BATCH, B=3, P=100, Hq=2, Hkv=1, d_head=8)
    att = inputs.attention_inputs(shp, seed=2)
    pk, pv, table = inputs.paged_layout(att["kenc"], att["venc"], att["prompt_len"], 16, seed=2)
    for b in range(3):
        for j in range(int(att["prompt_len"][b])):
            assert np.array_equal(pk[table[b, j // 16], j % 16], att["kenc"][b, j])
    used = table[table >= 0]
    assert len(set(used.tolist())) == used.size


def test_two_stage_tables():
    shp = configs.scaled(configs.MIXED_BATCH, V=4096)
    t = inputs.two_stage_tables(shp, seed=0)
    assert len(t) == 32
    for r in t:
        assert len(r["group_labels"]) == 9 and len(r["item_labels"]) == 9
        assert sum(len(x) for x in r["item_labels"]) == 77
        assert 0 <= len(r["others"]) <= 3
        assert all(2 <= len(l) <= 26 for _, l in r["others"])
