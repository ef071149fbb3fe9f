"""GPU parity of the wide-label read (dg_slot_read_wide) against the oracle.

One read over up to 256 labels per slot (the 77-intent single read) with label
tables of row stride L: reduced shapes for strides 40, 77 and 256 (the three
epilogue widths), the full 262144 x 2816 vocabulary with a 77-label slot, and
agreement with dg_slot_read when the labels fit the 26-wide table.
"""
import numpy as np
import pytest

from structured_slot_reads_gb300 import configs, dg, inputs
from tests import margins
from tests.gpu_util import assert_abs, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _table(S, L, ns, V, seed):
    lab = np.full((S, L), -1, np.int32)
    for s, n in enumerate(ns):
        lab[s, :n] = inputs.label_set(n, V, seed, 77, s)
    return lab, np.array(ns, np.int32)


def _run_wide(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, step, samples,
              gate):
    M, D = h.shape
    V = w.shape[0]
    S, L = label_ids.shape
    d = dg.make_dims(d_model=D, V=V)
    f32, i32 = torch.float32, torch.int32
    q_avg = torch.empty((S, L), dtype=f32, device="cuda")
    h_slot = torch.empty(S, dtype=f32, device="cuda")
    chosen = torch.empty(S, dtype=i32, device="cuda")
    lp = torch.empty((S, samples, L), dtype=f32, device="cuda")
    res = torch.empty(S, dtype=torch.uint8, device="cuda")
    nr = torch.empty(S, dtype=i32, device="cuda")
    tok = torch.empty((S, samples), dtype=i32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_SLOT_READ, S * samples),
                     dtype=torch.uint8, device="cuda")
    rc = dg.dg_slot_read_wide(d, dev_bf16(h), M, w if torch.is_tensor(w) else dev_bf16(w),
                              e if torch.is_tensor(e) else dev_bf16(e), dev(inv_t), dev(slot_row),
                              dev(slot_req), dev(label_ids), dev(n_labels), S, L, seed, step,
                              samples, gate, q_avg, h_slot, chosen, lp, res, nr, tok, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return dict(q_avg=host(q_avg), h_slot=host(h_slot), chosen=host(chosen), lp=host(lp),
                resampled=host(res), n_reads=host(nr), tokens=host(tok))


def _compare(got, want, n_labels):
    assert np.array_equal(got["tokens"], want["tokens"]), "noise tokens"
    assert np.array_equal(got["resampled"], want["resampled"]), "resample decision"
    assert np.array_equal(got["n_reads"], want["n_reads"]), "read count"
    assert np.array_equal(got["chosen"], want["chosen"]), "chosen label"
    for s, n in enumerate(n_labels):
        assert_abs(got["q_avg"][s, :n], want["q_avg"][s, :n], what="label distribution")
        assert np.all(got["q_avg"][s, n:] == 0)
        assert_abs(got["lp"][s, :, :n], want["lp"][s, :, :n], what="label logprobs")
    assert_abs(got["h_slot"], want["h_slot"], what="slot entropy")


@pytest.mark.parametrize("L,ns", [(40, [40, 3]), (77, [77, 50, 2]), (256, [256, 77, 130])])
@pytest.mark.parametrize("seed", [0, 1])
def test_wide_read_reduced(L, ns, seed):
    M, D, V = 64, 256, 4096
    h = inputs.hidden(M, D, seed)
    w, e = inputs.weights(V, D, 3000 + seed)
    inv_t = inputs.inv_temperature(M, seed)
    S = len(ns)
    slot_row = np.array([5 + 17 * s for s in range(S)], np.int32)
    slot_req = np.zeros(S, np.int32)
    label_ids, n_labels = _table(S, L, ns, V, seed)
    mode = "high" if seed % 2 == 0 else "low"
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, seed, 0, 4, 0.1, [mode] * S)
    got = _run_wide(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, 0, 4, 0.1)
    _compare(got, want, n_labels)
    assert np.all(got["resampled"] == (1 if mode == "high" else 0))


def test_wide_read_matches_standard_read_when_labels_fit():
    """Slots of 2..26 labels in a stride-32 table give exactly dg_slot_read's outputs."""
    M, D, V = 64, 256, 4096
    seed = 4
    h = inputs.hidden(M, D, seed)
    w, e = inputs.weights(V, D, seed)
    inv_t = inputs.inv_temperature(M, seed)
    ns = [2, 26, 5, 13]
    S = len(ns)
    slot_row = np.array([3, 20, 41, 60], np.int32)
    slot_req = np.zeros(S, np.int32)
    lab32, n_labels = _table(S, 32, ns, V, seed)
    got = _run_wide(h, w, e, inv_t, slot_row, slot_req, lab32, n_labels, seed, 2, 4, 0.1)
    d = dg.make_dims(d_model=D, V=V)
    f32, i32 = torch.float32, torch.int32
    q_avg = torch.empty((S, 26), dtype=f32, device="cuda")
    h_slot = torch.empty(S, dtype=f32, device="cuda")
    chosen = torch.empty(S, dtype=i32, device="cuda")
    lp = torch.empty((S, 4, 26), dtype=f32, device="cuda")
    res = torch.empty(S, dtype=torch.uint8, device="cuda")
    nr = torch.empty(S, dtype=i32, device="cuda")
    tok = torch.empty((S, 4), dtype=i32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_SLOT_READ, S * 4), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_slot_read(d, dev_bf16(h), M, dev_bf16(w), dev_bf16(e), dev(inv_t), dev(slot_row),
                         dev(slot_req), dev(np.ascontiguousarray(lab32[:, :26])), dev(n_labels),
                         S, seed, 2, 4, 0.1, q_avg, h_slot, chosen, lp, res, nr, tok, ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    assert np.array_equal(got["chosen"], host(chosen))
    assert np.array_equal(got["resampled"], host(res))
    assert np.array_equal(got["tokens"], host(tok))
    assert np.array_equal(got["q_avg"][:, :26], host(q_avg))
    assert np.array_equal(got["lp"][:, :, :26], host(lp))
    assert np.array_equal(got["h_slot"], host(h_slot))


@pytest.mark.parametrize("seed", [0, 1])
def test_wide_read_full_vocabulary_77_intents(seed):
    """Full 2816 x 262144 shapes: a 77-label slot and a 9-label slot in one stride-77 call."""
    shape = configs.SINGLE_READ
    w, e = inputs.weights(shape.V, shape.D, 2025)
    M = shape.B * shape.C
    h = inputs.hidden(M, shape.D, seed)
    inv_t = inputs.inv_temperature(M, seed)
    slot_row = np.array([61, 125], np.int32)
    slot_req = np.zeros(2, np.int32)
    label_ids, n_labels = _table(2, 77, [77, 9], shape.V, seed)
    mode = "high" if seed % 2 == 0 else "low"
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, seed, 0, 4, 0.1, [mode] * 2)
    got = _run_wide(h, dev_bf16(w), dev_bf16(e), inv_t, slot_row, slot_req, label_ids, n_labels,
                    seed, 0, 4, 0.1)
    _compare(got, want, n_labels)
