"""GPU parity of the batched two-stage read (mixed batch, paged prompt KV, ask_if).

Reduced shapes (4 requests, vocabulary 4096, d_model 256, ragged prompts of
up to 200 tokens in 16-token pages, 512-wide heads) and the full mixed batch
(32 requests, prompts U[512, 8192], vocabulary 262144, d_model 2816) are
compared on every decision of both stages: the slot rows are re-drawn until
each stage-1 slot and each asked stage-2 slot has its margin.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from structured_slot_reads_gb300.read import TwoStageRead
from tests import margins
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _build(shape, seed):
    M = shape.B * shape.C
    w, e = inputs.weights(shape.V, shape.D, seed)
    h = inputs.hidden(M, shape.D, seed)
    inv_t = inputs.inv_temperature(M, seed)
    plen = inputs.prompt_lengths(shape, seed, lo=min(512, shape.P // 2))
    att = inputs.attention_inputs(shape, seed, prompt_len=plen)
    pk, pv, table = inputs.paged_layout(att["kenc"], att["venc"], plen, shape.page_size, seed)
    tables = inputs.two_stage_tables(shape, seed)
    return dict(w=w, e=e, h=h, inv_t=inv_t, att=att, pk=pk, pv=pv, table=table, tables=tables,
                plen=plen)


def _runner(shape, x, seed, w_or):
    """The two-stage runner with its slot rows re-drawn until every decision of both
    stages (each stage-1 slot, each asked stage-2 slot) has its margin; returns the
    runner and the oracle's result for the final inputs."""
    tr = TwoStageRead(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), x["tables"], x["plen"],
                      seed=seed)
    rows1, lab1, n1 = tr.host_slots1
    slots1 = (rows1, host(tr.slot_req1), lab1, n1)
    slots2 = (host(tr.slot_row2), np.arange(tr.S2))
    x["h"], want = margins.prepare_two_stage_inputs(x["h"], w_or, x["e"], x["inv_t"], slots1,
                                                    tr.host_questions, slots2, seed, shape.R,
                                                    shape.gate)
    tr.h.copy_(dev_bf16(x["h"]))
    tr.inv_t.copy_(dev(x["inv_t"]))
    tr.q.copy_(dev_bf16(x["att"]["q"]))
    tr.kc.copy_(dev_bf16(x["att"]["kc"]))
    tr.vc.copy_(dev_bf16(x["att"]["vc"]))
    tr.set_kv(dev_bf16(x["pk"]), dev_bf16(x["pv"]), dev(x["table"]))
    return tr, want


def _check_stage(out, want, n_labels):
    """Every slot of a stage: distributions within 2e-3, decisions bit for bit (the
    inputs carry margins), not-asked slots (no labels) unread.  Returns the number
    of decisions compared."""
    got = {k: host(v) for k, v in out.items()}
    compared = 0
    for s, n in enumerate(n_labels):
        assert_abs(got["q_avg"][s, :n], want["q_avg"][s, :n], what="label distribution")
        assert got["chosen"][s] == want["chosen"][s]
        assert got["resampled"][s] == want["resampled"][s]
        assert got["n_reads"][s] == want["n_reads"][s]
        compared += int(n > 0)
    assert np.array_equal(got["tokens"], want["tokens"])
    return compared


def test_two_stage_reduced():
    shape = configs.scaled(configs.MIXED_BATCH, B=4, C=64, P=200, D=256, V=4096)
    seed = 3
    x = _build(shape, seed)
    tr, (st1, (lab2, n2, fired), st2) = _runner(shape, x, seed, x["w"])
    dg.dg_clear_status()
    tr.run()
    torch.cuda.synchronize()
    tr.check()
    kenc, venc = oracle.paged_to_contiguous(x["pk"], x["pv"], x["table"], x["plen"],
                                            shape.page_size)
    ref, ref_lse = oracle.attn_decode(x["att"]["q"], x["att"]["kc"], x["att"]["vc"], kenc, venc,
                                      x["plen"], shape.W)
    assert_rel(host(tr.attn_out), ref, what="paged attention")
    assert_abs(host(tr.attn_lse), ref_lse, what="paged attention lse")
    n1 = tr.host_slots1[2]
    assert _check_stage(tr.out1, st1, n1) == tr.S1
    # the gate picks exactly the oracle's stage-2 questions
    assert np.array_equal(host(tr.fired), fired)
    assert np.array_equal(host(tr.n_labels2), n2)
    assert np.array_equal(host(tr.label_ids2), lab2)
    assert host(tr.fired).sum() == shape.B          # exactly one question fires per request
    assert _check_stage(tr.out2, st2, n2) == shape.B


@pytest.mark.parametrize("S1,S2,Q", [(10, 6, 40), (30, 40, 300), (5, 1, 3), (4, 3, 97)])
def test_ask_if_select_matches_oracle(S1, S2, Q):
    """Several fired questions per stage-2 slot (the lowest index wins), slots with
    none, more questions than a warp's lanes, and out-of-range conditions."""
    rng = np.random.default_rng(7 + Q)
    chosen1 = rng.integers(-1, 5, S1).astype(np.int32)
    cs = rng.integers(0, S1, Q).astype(np.int32)
    cs[[1, Q - 1]] = [S1, -1]                                # out of range: flagged, never fire
    cv = rng.integers(0, 5, Q).astype(np.int32)
    own = rng.integers(0, S2, Q).astype(np.int32)
    qn = rng.integers(1, 27, Q).astype(np.int32)
    qlab = np.full((Q, 26), -1, np.int32)
    for q in range(Q):
        qlab[q, :qn[q]] = rng.choice(1000, qn[q], replace=False)
    lab2 = torch.empty((S2, 26), dtype=torch.int32, device="cuda")
    n2 = torch.empty(S2, dtype=torch.int32, device="cuda")
    fired = torch.empty(Q, dtype=torch.uint8, device="cuda")
    dg.dg_clear_status()
    rc = dg.dg_ask_if_select(dev(chosen1), S1, dev(cs), dev(cv), dev(own), dev(qlab), dev(qn), Q,
                             S2, lab2, n2, fired)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    w_lab, w_n, w_fired = oracle.ask_if_select(chosen1, cs, cv, own, qlab, qn, S2)
    assert np.array_equal(host(fired), w_fired)
    assert np.array_equal(host(n2), w_n)
    assert np.array_equal(host(lab2), w_lab)
    assert dg.dg_get_status() & dg.DG_DEV_BAD_INDEX   # the out-of-range conditions were flagged
    dg.dg_clear_status()


def test_two_stage_mixed_batch_full_size():
    shape = configs.MIXED_BATCH
    seed = 1
    x = _build(shape, seed)
    w64 = x["w"].astype(np.float64)
    tr, (st1, (lab2, n2, fired), st2) = _runner(shape, x, seed, w64)
    tr.run()
    torch.cuda.synchronize()
    tr.check()
    n1 = tr.host_slots1[2]
    # every stage-1 and every asked stage-2 decision, bit for bit
    assert _check_stage(tr.out1, st1, n1) == tr.S1
    assert np.array_equal(host(tr.fired), fired)
    assert np.array_equal(host(tr.label_ids2), lab2)
    assert host(tr.fired).sum() == shape.B
    assert _check_stage(tr.out2, st2, n2) == shape.B
    # a request reads each stage at most four times
    assert np.all(host(tr.out1["n_reads"]) <= shape.R)
    assert np.all(host(tr.out2["n_reads"]) <= shape.R)
    # paged attention on sampled requests: the longest prompt and request 0
    got = host(tr.attn_out)
    for b in sorted({0, int(np.argmax(x["plen"]))}):
        sl = slice(b, b + 1)
        kenc, venc = oracle.paged_to_contiguous(x["pk"], x["pv"], x["table"][sl], x["plen"][sl],
                                                shape.page_size)
        ref, _ = oracle.attn_decode(x["att"]["q"][sl], x["att"]["kc"][sl], x["att"]["vc"][sl],
                                    kenc, venc, x["plen"][sl], shape.W)
        assert_rel(got[sl], ref, what=f"paged attention, request {b}")
