"""Eight consecutive denoise steps of the full-canvas workload on the GPU against the
oracle's loop (24-ai.news, "Token commit mechanism": committed tokens stay fixed
and leave the candidate set, the expected embedding feeds the next step;
"How does diffusion text generation differ?": the 256-token canvas is refined
over several steps).

The full-canvas workload's canvas (256 positions, all open), commit threshold
0.1 x 256, three answer slots (2 / 26 / 5 labels, four reads), 8 / 2 heads of
512 with W = 128, and eight steps; the vocabulary and d_model are reduced
(4096 x 256) and the prompt to 256 tokens so that the float64 loop runs in
seconds.  The hidden rows are re-drawn until every decision of all eight steps
has its margin, so every step's commit set, committed tokens and slot
decisions are compared bit for bit; row statistics within 2e-3, expected
embeddings within 1e-2 relative, the next step's canvas input bit for bit
(recomputed from the GPU's own expected embedding).  The same eight steps
replayed as CUDA graphs, as the benchmark launches them, give the same
results bit for bit.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs
from structured_slot_reads_gb300.step import DenoiseStep
from tests import margins
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

N_STEPS = 8
SHAPE = configs.scaled(configs.FULL_CANVAS, name="full_canvas_loop_reduced", P=256, D=256,
                       V=4096)
KEYS = ("lse", "ent", "argmax", "commit", "tokens", "n_commit", "committed", "tok_state", "e_sc",
        "h", "chosen", "q_avg", "resampled", "n_reads", "noise_tok")


def _load(st, x):
    st.h0.copy_(dev_bf16(x["h"]))
    st.inv_t.copy_(dev(x["inv_t"]))
    for k in ("q", "kc", "vc", "kenc", "venc"):
        getattr(st, k).copy_(dev_bf16(x[k]))
    st.cand.copy_(dev(x["cand"]))
    st.prompt_len.copy_(dev(x["prompt_len"]))
    st.set_slots(x["slot_row"], x["slot_req"], x["label_ids"], x["n_labels"])
    st.reset_state()


def test_eight_step_loop_against_oracle():
    assert SHAPE.steps == N_STEPS and SHAPE.C == 256 and SHAPE.all_open
    x, steps, reads = margins.prepare_loop_inputs(SHAPE, N_STEPS, seed=0)
    st = DenoiseStep(SHAPE, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=0)
    assert st.fused and st.concurrent and st.n_draw == 12
    _load(st, x)
    ref_attn, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                           x["prompt_len"], SHAPE.W)
    committed = np.zeros(SHAPE.C, dtype=np.uint8)
    records = []
    for t in range(N_STEPS):
        st.run(step_idx=t)
        torch.cuda.synchronize()
        ref = steps[t]
        got = {k: host(getattr(st, k)).copy() for k in KEYS}
        records.append(got)
        assert_abs(got["lse"], ref["lse"], what=f"step {t} lse")
        assert_abs(got["ent"], ref["entropy"], what=f"step {t} entropy")
        assert np.array_equal(got["commit"][0], ref["commit"]), f"step {t} commit set"
        assert np.array_equal(got["tokens"][0], ref["tokens"]), f"step {t} tokens"
        assert got["n_commit"][0] == ref["n_commit"] >= 1
        committed |= ref["commit"].astype(np.uint8)
        assert np.array_equal(got["committed"][0], committed), f"step {t} carried commit mask"
        assert_rel(got["e_sc"], ref["e"], what=f"step {t} expected embedding")
        want = reads[t]
        assert np.array_equal(got["noise_tok"], want["tokens"]), f"step {t} noise draws"
        assert np.array_equal(got["chosen"], want["chosen"]), f"step {t} chosen labels"
        assert np.array_equal(got["resampled"], want["resampled"]), f"step {t} gate"
        assert np.array_equal(got["n_reads"], want["n_reads"]), f"step {t} reads"
        for s, k in enumerate(x["n_labels"]):
            assert_abs(got["q_avg"][s, :k], want["q_avg"][s, :k], what=f"step {t} slot {s}")
        h_next = oracle.canvas_update(x["h"], got["e_sc"], x["e"], got["tok_state"][0],
                                      got["committed"][0])
        assert np.array_equal(got["h"], h_next), f"step {t} next canvas input"
    st.check()
    assert_rel(host(st.attn_out), ref_attn, what="attention")
    assert_abs(host(st.attn_lse), ref_lse, what="attention lse")
    # committed positions never re-enter: the final state is the union of the steps
    _, final_committed, final_tokens = oracle.denoise_loop(
        x["h"], x["w"], x["e"], x["inv_t"], x["cand"][0].astype(bool), SHAPE.gamma, N_STEPS)
    assert np.array_equal(records[-1]["committed"][0].astype(bool), final_committed)
    assert np.array_equal(records[-1]["tok_state"][0], final_tokens)
    assert sum(r["n_commit"][0] for r in records) == int(final_committed.sum())

    # the same eight steps as CUDA graphs (captured before any replay), bit for bit
    _load(st, x)
    for t in range(N_STEPS):
        st.capture(t)
    _load(st, x)
    for t in range(N_STEPS):
        st.replay(t)
        torch.cuda.synchronize()
        for k in KEYS:
            assert np.array_equal(host(getattr(st, k)), records[t][k]), (t, k)
    st.check()
