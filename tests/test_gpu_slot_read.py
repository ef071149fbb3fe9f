"""GPU parity of the structured read (dg_slot_read / dg_slot_finish) against the oracle.

Half of the seeds plant a high-entropy first read (the 0.1 gate fires and four
reads are averaged), half plant a dominant label (one read).  Decisions are
bit-exact, probabilities and logprobs within 2e-3.
"""
import numpy as np
import pytest

from structured_slot_reads_gb300 import configs, dg, inputs
from tests.gpu_util import assert_abs, dev, dev_bf16, host
from tests import margins

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _run_read(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, step, samples, gate):
    M, D = h.shape
    V = w.shape[0]
    S = len(slot_row)
    d = dg.make_dims(d_model=D, V=V)
    f32, i32 = torch.float32, torch.int32
    q_avg = torch.empty((S, 26), dtype=f32, device="cuda")
    h_slot = torch.empty(S, dtype=f32, device="cuda")
    chosen = torch.empty(S, dtype=i32, device="cuda")
    lp = torch.empty((S, samples, 26), dtype=f32, device="cuda")
    res = torch.empty(S, dtype=torch.uint8, device="cuda")
    nr = torch.empty(S, dtype=i32, device="cuda")
    tok = torch.empty((S, samples), dtype=i32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_SLOT_READ, S * samples),
                     dtype=torch.uint8, device="cuda")
    assert dg.dg_validate_slots(d, slot_row, label_ids, n_labels, S, M) == dg.DG_OK
    rc = dg.dg_slot_read(d, dev_bf16(h), M, w if torch.is_tensor(w) else dev_bf16(w),
                         e if torch.is_tensor(e) else dev_bf16(e), dev(inv_t), dev(slot_row),
                         dev(slot_req), dev(label_ids), dev(n_labels), S, seed, step, samples,
                         gate, q_avg, h_slot, chosen, lp, res, nr, tok, ws)
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


def _case(shape, seed, samples=4):
    M = shape.B * shape.C
    h = inputs.hidden(M, shape.D, seed)
    w, e = inputs.weights(shape.V, shape.D, 1000 + seed // 2)
    inv_t = inputs.inv_temperature(M, seed)
    slot_row, slot_req, label_ids, n_labels = inputs.slot_table(shape, seed)
    return h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
@pytest.mark.parametrize("samples", [4, 1])
def test_slot_read_reduced(seed, samples):
    shape = configs.scaled(configs.SINGLE_READ, C=64, D=256, V=4096,
                           slots=[(5, 2), (30, 26), (50, 5)])
    h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels = _case(shape, seed)
    mode = "high" if seed % 2 == 0 else "low"
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, seed, 0, samples, 0.1, [mode] * 3)
    got = _run_read(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, 0, samples, 0.1)
    _compare(got, want, n_labels)
    if samples == 4:
        assert np.all(got["resampled"] == (1 if mode == "high" else 0))
    else:
        assert np.all(got["n_reads"] == 1)


@pytest.mark.parametrize("seed", [0, 1])
def test_slot_read_more_than_16_draw_rows(seed):
    """Six slots x 4 reads = 24 draw rows: past the skinny form, the W pass is the
    GEMM form with the label gather in its epilogue (two requests' canvases)."""
    shape = configs.scaled(configs.SINGLE_READ, B=2, C=64, D=256, V=4096,
                           slots=[(5, 2), (30, 26), (50, 5), (7, 9), (40, 17), (63, 3)])
    h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels = _case(shape, seed)
    S = len(slot_row)
    assert S * 4 > 16
    mode = "high" if seed % 2 == 0 else "low"
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, seed, 0, 4, 0.1, [mode] * S)
    got = _run_read(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, seed, 0, 4, 0.1)
    _compare(got, want, n_labels)
    assert np.all(got["resampled"] == (1 if mode == "high" else 0))


def test_slot_read_tiny_config():
    shape = configs.TINY
    h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels = _case(shape, 0)
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, 0, 0, 4, 0.1, [None])
    got = _run_read(h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels, 0, 0, 4, 0.1)
    _compare(got, want, n_labels)


@pytest.fixture(scope="module")
def full_weights():
    shape = configs.SINGLE_READ
    w, e = inputs.weights(shape.V, shape.D, 2024)
    return w, e, dev_bf16(w), dev_bf16(e)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_slot_read_single_structured_read_full_size(seed, full_weights):
    """Full 2816 x 262144 shapes: three slots (2, 26, 5 labels), resample forced for even seeds."""
    shape = configs.SINGLE_READ
    w, e, wd, ed = full_weights
    M = shape.B * shape.C
    h = inputs.hidden(M, shape.D, seed)
    inv_t = inputs.inv_temperature(M, seed)
    slot_row, slot_req, label_ids, n_labels = inputs.slot_table(shape, seed)
    mode = "high" if seed % 2 == 0 else "low"
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, seed, 0, 4, 0.1, [mode] * 3)
    got = _run_read(h, wd, ed, inv_t, slot_row, slot_req, label_ids, n_labels, seed, 0, 4, 0.1)
    _compare(got, want, n_labels)
    assert np.all(got["resampled"] == (1 if mode == "high" else 0))


def test_device_label_count_beyond_26_is_not_read():
    """A slot whose label count reaches the device out of range (27, or negative: a
    table that skipped the host check) is not read: chosen -1, no reads, zero
    distribution, entropy and logprobs, and DG_DEV_BAD_LABEL is set; the other
    slots of the call are read as usual."""
    shape = configs.scaled(configs.SINGLE_READ, C=64, D=256, V=4096,
                           slots=[(5, 2), (30, 26), (50, 5)])
    h, w, e, inv_t, slot_row, slot_req, label_ids, n_labels = _case(shape, 4)
    h, want = margins.prepare_slot_inputs(h, w, e, inv_t, slot_row, slot_req, label_ids,
                                          n_labels, 4, 0, 4, 0.1, [None] * 3)
    bad_n = n_labels.copy()
    bad_n[1] = 27
    bad_n[2] = -1
    M, D = h.shape
    S = len(slot_row)
    d = dg.make_dims(d_model=D, V=shape.V)
    f32, i32 = torch.float32, torch.int32
    out = dict(q_avg=torch.full((S, 26), 7.0, dtype=f32, device="cuda"),
               h_slot=torch.full((S,), 7.0, dtype=f32, device="cuda"),
               chosen=torch.full((S,), 7, dtype=i32, device="cuda"),
               lp=torch.full((S, 4, 26), 7.0, dtype=f32, device="cuda"),
               res=torch.full((S,), 7, dtype=torch.uint8, device="cuda"),
               nr=torch.full((S,), 7, dtype=i32, device="cuda"),
               tok=torch.empty((S, 4), dtype=i32, device="cuda"))
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_SLOT_READ, S * 4), dtype=torch.uint8,
                     device="cuda")
    dg.dg_clear_status()
    rc = dg.dg_slot_read(d, dev_bf16(h), M, dev_bf16(w), dev_bf16(e), dev(inv_t), dev(slot_row),
                         dev(slot_req), dev(label_ids), dev(bad_n), S, 4, 0, 4, 0.1,
                         out["q_avg"], out["h_slot"], out["chosen"], out["lp"], out["res"],
                         out["nr"], out["tok"], ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    assert dg.dg_get_status() & dg.DG_DEV_BAD_LABEL
    dg.dg_clear_status()
    got = {k: host(v) for k, v in out.items()}
    for s in (1, 2):
        assert got["chosen"][s] == -1 and got["nr"][s] == 0 and got["res"][s] == 0
        assert np.all(got["q_avg"][s] == 0) and got["h_slot"][s] == 0
        assert np.all(got["lp"][s] == 0)
    assert got["chosen"][0] == want["chosen"][0] and got["nr"][0] == want["n_reads"][0]
    assert_abs(got["q_avg"][0, :2], want["q_avg"][0, :2], what="slot 0 distribution")
