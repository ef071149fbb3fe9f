"""The read-only step (ReadStep: attention + one slot read) on the GPU.

A reduced single-structured-read shape (2 requests, canvas 128, prompt 600,
512-wide heads, vocabulary 4096, d_model 256, slots of 2 / 26 / 5 labels):
the attention and the slot read against the oracle, and the side-stream
schedule (attention beside the slot read's W pass) equal to the one-stream
schedule — the slot read bit for bit, the attention against the oracle in
both (on the side stream it plans for fewer SMs, so its key splits and
rounding differ).
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from structured_slot_reads_gb300.read import ReadStep
from tests import margins
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_read_step_schedules_match_oracle():
    shape = configs.scaled(configs.SINGLE_READ, B=2, C=128, P=600, D=256, V=4096,
                           slots=[(61, 2), (100, 26), (120, 5)])
    x = inputs.step_inputs(shape, seed=4)
    st = ReadStep(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=0, concurrent=False)
    row, req, lab, n = (host(t) for t in (st.slot_row, st.slot_req, st.label_ids, st.n_labels))
    # slot rows re-drawn until every decision (of both requests' slots) has its margin
    x["h"], want = margins.prepare_slot_inputs(x["h"], x["w"], x["e"], x["inv_t"], row, req, lab,
                                               n, 0, 2, shape.R, shape.gate, [None] * len(row))
    st.h.copy_(dev_bf16(x["h"]))
    st.inv_t.copy_(dev(x["inv_t"]))
    for k in ("q", "kc", "vc", "kenc", "venc"):
        getattr(st, k).copy_(dev_bf16(x[k]))
    st.prompt_len.copy_(dev(x["prompt_len"]))
    keys = ("q_avg", "h_slot", "chosen", "lp", "resampled", "n_reads", "tokens")

    ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                      x["prompt_len"], shape.W)
    dg.dg_clear_status()
    st.run(step_idx=2)
    torch.cuda.synchronize()
    serial = {k: host(st.out[k]).copy() for k in keys}
    assert_rel(host(st.attn_out), ref, what="attention, one stream")
    assert_abs(host(st.attn_lse), ref_lse, what="attention lse, one stream")
    st.concurrent = True
    for _ in range(2):                       # the second run reuses the side stream
        st.run(step_idx=2)
        torch.cuda.synchronize()
        for k in keys:
            assert np.array_equal(host(st.out[k]), serial[k]), k
        assert_rel(host(st.attn_out), ref, what="attention, side stream")
        assert_abs(host(st.attn_lse), ref_lse, what="attention lse, side stream")
    st.check()
    assert np.array_equal(serial["tokens"], want["tokens"])
    for s, k in enumerate(n):
        assert_abs(serial["q_avg"][s, :k], want["q_avg"][s, :k], what="slot distribution")
    assert np.array_equal(serial["chosen"], want["chosen"])
    assert np.array_equal(serial["resampled"], want["resampled"])
    assert np.array_equal(serial["n_reads"], want["n_reads"])
