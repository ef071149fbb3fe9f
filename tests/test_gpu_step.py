"""Whole denoise steps on the GPU (DenoiseStep, every library call) against the oracle.

* tiny read shape: four consecutive steps of the loop (attention, lm-head,
  slot read, commit with state carried forward, self-conditioning, canvas
  update) compared step by step;
* full-canvas shape at full size (prompt 4096, canvas 256, vocab 262144,
  d_model 2816, 8/2 heads of 512): one step, with attention compared in full
  and the lm-head and self-conditioning compared on sampled rows.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from structured_slot_reads_gb300.step import DenoiseStep
from tests import margins
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _load(st, x):
    st.h0.copy_(dev_bf16(x["h"]))
    st.inv_t.copy_(dev(x["inv_t"]))
    st.q.copy_(dev_bf16(x["q"]))
    st.kc.copy_(dev_bf16(x["kc"]))
    st.vc.copy_(dev_bf16(x["vc"]))
    st.kenc.copy_(dev_bf16(x["kenc"]))
    st.venc.copy_(dev_bf16(x["venc"]))
    st.cand.copy_(dev(x["cand"]))
    st.prompt_len.copy_(dev(x["prompt_len"]))
    if st.with_slots:
        st.set_slots(x["slot_row"], x["slot_req"], x["label_ids"], x["n_labels"])
    st.reset_state()


def _tiny_inputs(n_steps, seed=0):
    shape = configs.TINY
    x, steps, reads = margins.prepare_loop_inputs(shape, n_steps, seed)
    return shape, x, steps, reads


@pytest.mark.parametrize("fused", [True, False])
def test_tiny_loop_step_by_step(fused):
    n_steps = 4
    shape, x, steps, reads = _tiny_inputs(n_steps)
    st = DenoiseStep(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=0, fused=fused)
    assert st.fused == fused
    _load(st, x)
    ref_attn, ref_attn_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                                x["prompt_len"], shape.W)
    h = x["h"]
    for t in range(n_steps):
        st.run(step_idx=t)
        torch.cuda.synchronize()
        ref = steps[t]
        assert_rel(host(st.attn_out), ref_attn, what=f"step {t} attention")
        assert_abs(host(st.attn_lse), ref_attn_lse, what=f"step {t} attention lse")
        assert_abs(host(st.lse), ref["lse"], what=f"step {t} lse")
        assert_abs(host(st.ent), ref["entropy"], what=f"step {t} entropy")
        assert np.array_equal(host(st.commit)[0], ref["commit"]), f"step {t} commit set"
        assert np.array_equal(host(st.tokens)[0], ref["tokens"]), f"step {t} tokens"
        assert host(st.n_commit)[0] == ref["n_commit"]
        assert_rel(host(st.e_sc), ref["e"], what=f"step {t} expected embedding")
        # the slot read of this step, from this step's canvas input (the oracle
        # chain's; the inputs carry the margins, so the decisions are compared)
        want = reads[t]
        assert np.array_equal(host(st.chosen), want["chosen"])
        assert np.array_equal(host(st.resampled), want["resampled"])
        assert_abs(host(st.q_avg)[0, :4], want["q_avg"][0, :4], what="slot distribution")
        # next step's canvas input
        committed = host(st.committed)[0]
        tok_state = host(st.tok_state)[0]
        h = oracle.canvas_update(x["h"], host(st.e_sc), x["e"], tok_state, committed)
        assert np.array_equal(host(st.h), h), f"step {t} canvas update"
    st.check()


@pytest.fixture(scope="module")
def full_inputs():
    """Full-canvas inputs with the slot rows re-drawn until the three slot reads have
    their margins (so their decisions are always compared)."""
    shape = configs.FULL_CANVAS
    x = inputs.step_inputs(shape, seed=0)
    w64 = x["w"].astype(np.float64)
    x["h"], want = margins.prepare_slot_inputs(x["h"], w64, x["e"], x["inv_t"], x["slot_row"],
                                               x["slot_req"], x["label_ids"], x["n_labels"], 0, 0,
                                               shape.R, shape.gate, [None] * len(shape.slots))
    return x, w64, want


@pytest.fixture(scope="module", params=[True, False], ids=["fused", "unfused"])
def full_canvas(request, full_inputs):
    shape = configs.FULL_CANVAS
    x = full_inputs[0]
    w, e = x["w"], x["e"]
    wd, ed = dev_bf16(w), dev_bf16(e)
    st = DenoiseStep(shape, wd, ed, seed=0, fused=request.param)
    _load(st, x)
    st.run(step_idx=0)
    torch.cuda.synchronize()
    return shape, x, st


def test_full_canvas_attention(full_canvas):
    shape, x, st = full_canvas
    ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                      x["prompt_len"], shape.W)
    assert_rel(host(st.attn_out), ref, what="attention output")
    assert_abs(host(st.attn_lse), ref_lse, what="attention lse")


def test_full_canvas_lmhead_and_selfcond_sampled_rows(full_canvas, full_inputs):
    shape, x, st = full_canvas
    rows = np.array([0, 1, 61, 125, 128, 189, 200, 255])
    w64 = full_inputs[1]
    lse, ent, maxz, arg = oracle.lmhead_stats(x["h"][rows], w64, x["inv_t"][rows])
    assert_abs(host(st.lse)[rows], lse, what="lse")
    assert_abs(host(st.ent)[rows], ent, what="entropy")
    assert_abs(host(st.maxz)[rows], maxz, what="max logit")
    e_ref = oracle.selfcond_embed(x["h"][rows], w64, x["e"], x["inv_t"][rows])
    assert_rel(host(st.e_sc)[rows], e_ref, what="expected embedding")


def test_full_canvas_commit_and_slots(full_canvas, full_inputs):
    shape, x, st = full_canvas
    ent = host(st.ent).astype(np.float64)[None]
    arg = host(st.argmax)[None]
    # the oracle's commit on the GPU's own entropies: same order, float64 prefix sums
    cm, tk, n = oracle.commit(ent, arg, x["cand"], x["gamma"].astype(np.float64))
    assert np.array_equal(host(st.commit), cm)
    assert np.array_equal(host(st.tokens), tk)
    assert host(st.n_commit)[0] == n[0] >= 1
    # slot reads of the same step: decisions (the inputs carry their margins) and
    # distributions
    want = full_inputs[2]
    for s, k in enumerate(x["n_labels"]):
        assert_abs(host(st.q_avg)[s, :k], want["q_avg"][s, :k], what="slot distribution")
    assert np.array_equal(host(st.chosen), want["chosen"])
    assert np.array_equal(host(st.resampled), want["resampled"])
    assert np.array_equal(host(st.noise_tok), want["tokens"])


def test_batched_step_with_slot_read_pass():
    """Eight requests of the tiny shape: 32 draw rows exceed the 16 that ride in the
    fused pass, so the step reads its slots through dg_slot_read.  Every row's
    statistics, every request's commit (where its margins hold), the expected
    embeddings and the slot decisions are compared with the oracle."""
    shape = configs.scaled(configs.TINY, B=8)
    x = inputs.step_inputs(shape, seed=5)
    x["h"], want = margins.prepare_slot_inputs(x["h"], x["w"], x["e"], x["inv_t"], x["slot_row"],
                                               x["slot_req"], x["label_ids"], x["n_labels"], 0, 0,
                                               shape.R, shape.gate, [None] * 8)
    st = DenoiseStep(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=0, fused=True)
    assert st.n_draw == 0 and st.S == 8
    _load(st, x)
    launched = st.run(step_idx=0)
    torch.cuda.synchronize()
    st.check()
    assert launched == st.kernels_per_step()
    lse, ent, maxz, arg = oracle.lmhead_stats(x["h"], x["w"], x["inv_t"])
    assert_abs(host(st.lse), lse, what="lse")
    assert_abs(host(st.ent), ent, what="entropy")
    assert_rel(host(st.e_sc), oracle.selfcond_embed(x["h"], x["w"], x["e"], x["inv_t"]),
               what="expected embedding")
    ref_attn, _ = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                     x["prompt_len"], shape.W)
    assert_rel(host(st.attn_out), ref_attn, what="attention")
    ent_b = ent.reshape(shape.B, shape.C)
    com, toks, n = oracle.commit(ent_b, arg.reshape(shape.B, shape.C), x["cand"], x["gamma"])
    z = (x["h"].astype(np.float64) @ x["w"].astype(np.float64).T) * x["inv_t"][:, None]
    gap = top2_gap(z).reshape(shape.B, shape.C)
    checked = 0
    for b in range(shape.B):
        if not (margins.commit_margins_ok(ent_b[b], x["cand"][b], shape.gamma)
                and np.all(gap[b][com[b] == 1] > margins.ARGMAX_MARGIN)):
            continue
        checked += 1
        assert np.array_equal(host(st.commit)[b], com[b]), f"request {b} commit set"
        assert np.array_equal(host(st.tokens)[b], toks[b]), f"request {b} tokens"
        assert host(st.n_commit)[b] == n[b]
    assert checked >= 4
    assert np.array_equal(host(st.noise_tok), want["tokens"])
    for s in range(st.S):
        assert_abs(host(st.q_avg)[s, :4], want["q_avg"][s, :4], what="slot distribution")
    assert np.array_equal(host(st.chosen), want["chosen"])
    assert np.array_equal(host(st.resampled), want["resampled"])


def test_graph_replay_equals_eager_step():
    """A captured step replays the same kernels: after one eager step from the same
    state, the replayed step's outputs equal the eager ones bit for bit."""
    shape, x, _, _ = _tiny_inputs(2)
    st = DenoiseStep(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=0)
    _load(st, x)
    st.run(step_idx=0)                      # one eager step: one-time set-up done
    torch.cuda.synchronize()
    _load(st, x)
    st.run(step_idx=1)
    torch.cuda.synchronize()
    eager = {k: host(getattr(st, k)).copy() for k in ("lse", "ent", "commit", "tokens", "e_sc", "h",
                                                        "chosen", "q_avg", "attn_out")}
    _load(st, x)
    st.capture(1)
    _load(st, x)                            # capture does not execute: state is reloaded
    st.replay(1)
    torch.cuda.synchronize()
    for k, v in eager.items():
        assert np.array_equal(host(getattr(st, k)), v), k


@pytest.mark.parametrize("size", ["tiny", "full_canvas"])
def test_concurrent_schedule_equals_serial(size):
    """The side-stream schedule (slot finish, commit and attention beside the
    self-conditioning GEMM) computes the same step: three consecutive steps,
    eager and replayed as graphs, equal the one-stream schedule bit for bit,
    carried state included.  The attention alone may differ in rounding: on
    the side stream it plans for fewer SMs (fewer key splits, another
    summation order), so each schedule's attention is compared with the
    oracle instead."""
    if size == "tiny":
        shape, x, _, _ = _tiny_inputs(3)
    else:
        shape = configs.FULL_CANVAS
        x = inputs.step_inputs(shape, seed=0)
    wd, ed = dev_bf16(x["w"]), dev_bf16(x["e"])
    keys = ("lse", "ent", "argmax", "commit", "tokens", "n_commit", "e_sc", "h", "committed",
            "tok_state", "chosen", "q_avg", "resampled", "attn_out", "attn_lse")

    def steps(concurrent, graphs):
        st = DenoiseStep(shape, wd, ed, seed=0, concurrent=concurrent)
        assert st.concurrent == concurrent
        _load(st, x)
        st.run(step_idx=0)                  # one eager step: one-time set-up done
        torch.cuda.synchronize()
        _load(st, x)
        out = []
        for t in range(3):
            if graphs:
                st.replay(t)
            else:
                st.run(step_idx=t)
            torch.cuda.synchronize()
            out.append({k: host(getattr(st, k)).copy() for k in keys})
        assert dg.dg_get_status() == 0
        return out

    serial = steps(False, False)
    ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                      x["prompt_len"], shape.W)
    for graphs in (False, True):
        got = steps(True, graphs)
        for t in range(3):
            for k in keys:
                if k in ("attn_out", "attn_lse"):
                    continue
                assert np.array_equal(got[t][k], serial[t][k]), (graphs, t, k)
            assert_rel(got[t]["attn_out"], ref, what="side-stream attention")
            assert_abs(got[t]["attn_lse"], ref_lse, what="side-stream attention lse")
