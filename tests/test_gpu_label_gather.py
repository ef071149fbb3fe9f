"""GPU parity of the label gather fused into the lm-head passes (tau-home.com,
"Refusing JSON token generation": the read takes the logprobs of the allowed label
ids from the one denoise forward).

dg_lmhead_logsoftmax_entropy (and its e4m3 / NVFP4 forms) with slot tables writes
label_lp[s][k] = z[slot_row[s], label_k] - lse, taken from the accumulators in the
pass's epilogue; dg_denoise_heads writes the draw rows' label logits z/T the same
way.  Both are compared with the oracle's float64 label logits and statistics
(2e-3 absolute).  Label tables mix a contiguous run of ids (every label in one
32-column chunk of one CTA), the ragged end of the vocabulary, random ids,
duplicates, a single label and a slot with none.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import assert_abs, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L = 26
SENTINEL = 12345.0


def _tables(S, V, seed):
    """Label tables [S, 26] and counts exercising every shape of the gather."""
    rng = np.random.default_rng(seed)
    ids = np.zeros((S, L), np.int32)
    n = np.full(S, L, np.int32)
    for s in range(S):
        ids[s] = rng.choice(V, L, replace=False)
    ids[0] = np.arange(L)                      # a contiguous run at the start
    if S > 1:
        ids[1] = np.arange(V - L, V)           # the ragged end of the vocabulary
    if S > 2:
        n[2] = 0                               # a question not asked
    if S > 3:
        n[3] = 1
    if S > 4:
        ids[4, :5] = ids[4, 5]                 # duplicate ids
        n[4] = 9
    if S > 5:
        n[5] = 17
    return ids, n


def _want_lp(h_rows, w, inv_t_rows, ids, n):
    z = oracle.label_logits(h_rows, w, inv_t_rows, ids, n)
    lse, _, _, _ = oracle.lmhead_stats(h_rows, w, inv_t_rows)
    return z - lse[:, None]


def _check_lp(got, want, n, what):
    checked = 0
    for s in range(len(n)):
        if n[s]:
            assert_abs(got[s, :n[s]], want[s, :n[s]], what=f"{what} slot {s}")
        assert np.all(got[s, n[s]:] == SENTINEL), f"{what}: slot {s} written past n_labels"
        checked += int(n[s])
    assert checked > 0


def _lm_call(kind, d, M, args, inv_t, slot_row, ids, n, S):
    f32 = torch.float32
    lse, ent, mz = (torch.empty(M, dtype=f32, device="cuda") for _ in range(3))
    arg = torch.empty(M, dtype=torch.int32, device="cuda")
    lp = torch.full((max(S, 1), L), SENTINEL, dtype=f32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, M), dtype=torch.uint8,
                     device="cuda")
    slots = (dev(slot_row), dev(ids), dev(n), S, lse, ent, mz, arg, lp, ws)
    if kind == "bf16":
        rc = dg.dg_lmhead_logsoftmax_entropy(d, args[0], M, args[1], dev(inv_t), *slots)
    elif kind == "fp8":
        rc = dg.dg_lmhead_logsoftmax_entropy_fp8(d, args[0], args[1], M, args[2], args[3],
                                                 dev(inv_t), *slots)
    else:
        rc = dg.dg_lmhead_logsoftmax_entropy_nvfp4(d, args[0], M, args[1], args[2], args[3],
                                                   dev(inv_t), *slots)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return host(lp), host(lse)


@pytest.mark.parametrize("M,S,V,D", [(12, 6, 4096, 256), (300, 40, 3000, 192),
                                     (256, 12, 8192, 512), (1, 1, 1024, 64)])
def test_lmhead_label_gather(M, S, V, D):
    h = inputs.hidden(M, D, 5 + M)
    w, _ = inputs.weights(V, D, 6 + V)
    inv_t = inputs.inv_temperature(M, 7)
    slot_row = np.random.default_rng(M).choice(M, S, replace=False).astype(np.int32)
    ids, n = _tables(S, V, S)
    dg.dg_clear_status()
    lp, lse = _lm_call("bf16", dg.make_dims(d_model=D, V=V), M, (dev_bf16(h), dev_bf16(w)),
                       inv_t, slot_row, ids, n, S)
    assert dg.dg_get_status() == 0
    want = _want_lp(h[slot_row], w, inv_t[slot_row], ids, n)
    _check_lp(lp, want, n, "label lp")
    # the statistics are those of the pass without slots
    o_lse, _, _, _ = oracle.lmhead_stats(h, w, inv_t)
    assert_abs(lse, o_lse, what="lse")


def test_lmhead_label_gather_fp8():
    M, S, V, D = 64, 8, 4096, 256
    h = inputs.hidden(M, D, 21)
    w, _ = inputs.weights(V, D, 22)
    inv_t = inputs.inv_temperature(M, 23)
    qs = []
    for x in (h, w):
        q = torch.empty(x.shape, dtype=torch.uint8, device="cuda")
        sc = torch.empty(x.shape[0], dtype=torch.float32, device="cuda")
        assert dg.dg_quantize_rows_e4m3(dev_bf16(x), x.shape[0], x.shape[1], q, sc) == dg.DG_OK
        qs += [q, sc]
    torch.cuda.synchronize()
    slot_row = np.arange(3, 3 + 5 * S, 5, dtype=np.int32)
    ids, n = _tables(S, V, 24)
    lp, _ = _lm_call("fp8", dg.make_dims(d_model=D, V=V), M, qs, inv_t, slot_row, ids, n, S)
    hd = oracle.dequantize_rows(host(qs[0]), host(qs[1]))
    wd = oracle.dequantize_rows(host(qs[2]), host(qs[3]))
    _check_lp(lp, _want_lp(hd[slot_row], wd, inv_t[slot_row], ids, n), n, "fp8 label lp")


@pytest.mark.parametrize("M,S,V,D", [(40, 6, 3000, 192), (12, 5, 4096, 256)])
def test_lmhead_label_gather_nvfp4(M, S, V, D):
    h = inputs.hidden(M, D, 31)
    w, _ = inputs.weights(V, D, 32)
    inv_t = inputs.inv_temperature(M, 33)
    codes = torch.empty((D // 64, V, 32), dtype=torch.uint8, device="cuda")
    scales = torch.empty((D // 64, V, 4), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    assert dg.dg_quantize_nvfp4(dev_bf16(w), V, D, codes, scales, g) == dg.DG_OK
    torch.cuda.synchronize()
    slot_row = np.random.default_rng(M).choice(M, S, replace=False).astype(np.int32)
    ids, n = _tables(S, V, 34)
    lp, _ = _lm_call("nvfp4", dg.make_dims(d_model=D, V=V), M, (dev_bf16(h), codes, scales, g),
                     inv_t, slot_row, ids, n, S)
    oc, osc = oracle.from_kblock_layout(host(codes), host(scales))
    wq = oracle.dequantize_nvfp4(oc, osc, host(g)[0])
    _check_lp(lp, _want_lp(h[slot_row], wq, inv_t[slot_row], ids, n), n, "nvfp4 label lp")


def test_lmhead_label_gather_flags_bad_ids_and_rows():
    """A label id outside [0, V) sets DG_DEV_BAD_LABEL and reads -inf (the other
    labels of the slot are still right); two slots on one row set DG_DEV_BAD_INDEX."""
    M, S, V, D = 16, 3, 2048, 128
    h = inputs.hidden(M, D, 41)
    w, _ = inputs.weights(V, D, 42)
    inv_t = inputs.inv_temperature(M, 43)
    d = dg.make_dims(d_model=D, V=V)
    slot_row = np.array([2, 5, 11], np.int32)
    ids, n = _tables(S, V, 44)
    ids[0, 3] = V
    ids[1, 7] = -1
    dg.dg_clear_status()
    lp, _ = _lm_call("bf16", d, M, (dev_bf16(h), dev_bf16(w)), inv_t, slot_row, ids, n, S)
    assert dg.dg_get_status() & dg.DG_DEV_BAD_LABEL
    dg.dg_clear_status()
    assert lp[0, 3] == -np.inf and lp[1, 7] == -np.inf
    good = ids.copy()
    good[0, 3], good[1, 7] = 0, 0
    want = _want_lp(h[slot_row], w, inv_t[slot_row], good, n)
    for s, k in ((0, 3), (1, 7)):
        want[s, k] = lp[s, k]
    ok = np.isfinite(want)
    assert_abs(lp[ok], want[ok], what="label lp beside bad ids")
    # two slots on one row
    _lm_call("bf16", d, M, (dev_bf16(h), dev_bf16(w)), inv_t, np.array([2, 2, 11], np.int32),
             ids * 0 + np.arange(L, dtype=np.int32), n, S)
    assert dg.dg_get_status() & dg.DG_DEV_BAD_INDEX
    dg.dg_clear_status()


def test_lmhead_label_gather_refusals():
    d = dg.make_dims(d_model=64, V=1024)
    M = 4
    buf = torch.empty(4096, dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, M), dtype=torch.uint8,
                     device="cuda")
    h = torch.zeros((M, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((1024, 64), dtype=torch.bfloat16, device="cuda")
    i32 = torch.zeros(64, dtype=torch.int32, device="cuda")
    outs = (buf, buf, buf, i32)
    call = lambda sr, S: dg.dg_lmhead_logsoftmax_entropy(d, h, M, w, buf, sr, i32, i32, S,  # noqa
                                                         *outs, buf, ws)
    assert call(i32, 5) == dg.DG_ERR_SHAPE     # more slots than rows
    assert call(None, 2) == dg.DG_ERR_ARG      # a missing slot table
    assert call(i32, -1) == dg.DG_ERR_ARG


@pytest.mark.parametrize("M,R,S,V,D", [(256, 4, 3, 8192, 512), (100, 4, 4, 3000, 200),
                                       (64, 2, 8, 2504, 192), (1, 1, 16, 1024, 128)])
def test_denoise_heads_gathers_draw_labels(M, R, S, V, D):
    """The draw rows' label logits z/T from the fused heads pass (draw j is draw
    j % R of slot j / R), then dg_slot_finish from them alone (rows = NULL) against
    the same finish computing its own label logits."""
    nd = R * S
    h = inputs.hidden(M, D, 51 + M)
    w, _ = inputs.weights(V, D, 52)
    inv_t = inputs.inv_temperature(M, 53)
    draws = inputs.hidden(nd, D, 54)
    inv_d = inputs.inv_temperature(nd, 55)
    ids, n = _tables(S, V, 56 + S)
    d = dg.make_dims(d_model=D, V=V)
    f32 = torch.float32
    lse, ent, maxz = (torch.empty(M, dtype=f32, device="cuda") for _ in range(3))
    arg = torch.empty(M, dtype=torch.int32, device="cuda")
    lse_d = torch.empty(nd, dtype=f32, device="cuda")
    scale = torch.empty(M, dtype=f32, device="cuda")
    z = torch.full((nd, L), SENTINEL, dtype=f32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_HEADS, M), dtype=torch.uint8,
                     device="cuda")
    idd, nn = dev(ids), dev(n)
    dg.dg_clear_status()
    rc = dg.dg_denoise_heads(d, dev_bf16(h), M, dev_bf16(draws), nd, dev_bf16(w), dev(inv_t),
                             dev(inv_d), lse, ent, maxz, arg, lse_d, idd, nn, R, z, scale, None,
                             0, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    assert dg.dg_get_status() == 0
    got = host(z)
    want = oracle.label_logits(draws, w, inv_d, np.repeat(ids, R, axis=0), np.repeat(n, R))
    _check_lp(got, want, np.repeat(n, R), "draw label logits")
    # the finish from the gathered logits equals the finish that computes them
    outs = []
    for rows in (None, dev_bf16(draws)):
        o = dict(q=torch.empty((S, L), dtype=f32, device="cuda"),
                 hs=torch.empty(S, dtype=f32, device="cuda"),
                 ch=torch.empty(S, dtype=torch.int32, device="cuda"),
                 lp=z.clone() if rows is None else torch.empty((nd, L), dtype=f32, device="cuda"),
                 rs=torch.empty(S, dtype=torch.uint8, device="cuda"),
                 nr=torch.empty(S, dtype=torch.int32, device="cuda"))
        rc = dg.dg_slot_finish(d, rows, None if rows is None else dev(inv_d), lse_d,
                               None if rows is None else dev_bf16(w), idd, nn, S, R, R, 0.1,
                               o["q"], o["hs"], o["ch"], o["lp"], o["rs"], o["nr"])
        assert rc == dg.DG_OK, dg.strerror(rc)
        torch.cuda.synchronize()
        outs.append({k: host(v) for k, v in o.items()})
    a, b = outs
    for s in np.flatnonzero(n):
        assert_abs(a["lp"].reshape(S, R, L)[s, :, :n[s]], b["lp"].reshape(S, R, L)[s, :, :n[s]],
                   what="lp from gathered vs computed logits")
    assert_abs(a["hs"], b["hs"], what="slot entropy")
    assert np.array_equal(a["nr"], b["nr"])
    assert np.array_equal(a["ch"][n == 0], b["ch"][n == 0])
