"""GPU parity at the long-context and batch-sweep shapes, at full size.

* Long-context read: one request with a 110,707-token prompt (tau-home.com,
  "cache reuse": the length of the long-context example), a 256-token canvas
  with three slots (2 / 26 / 5 labels, four reads), vocabulary 262144,
  d_model 2816, 8 / 2 heads of 512, W = 128, run as ReadStep, the read the
  benchmark times (the attention on a side stream beside the slot read).  The
  attention is compared with the oracle on every row of every head (about 870
  key tiles per row block, long split ranges, the lazy rescale over them), the
  slot read bit for bit on its decisions (one slot forced to resample, one
  forced to a dominant label, one left as drawn; re-drawn until the margins
  hold).
* Batch sweep, batch 64 at prompt 8192: DenoiseStep over 64 full canvases
  (16384 rows: the fused heads pass over 64 row groups, the self-conditioning
  GEMM in its split-K configuration, the slot reads of 192 slots in their own
  W pass, every request's commit), compared on sampled rows, requests and
  slots.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from structured_slot_reads_gb300.read import ReadStep
from structured_slot_reads_gb300.step import DenoiseStep
from tests import margins
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def full_weights():
    shape = configs.LONG_CONTEXT
    w, e = inputs.weights(shape.V, shape.D, 4242)
    return dict(w=w, e=e, w64=w.astype(np.float64), e64=e.astype(np.float64), wd=dev_bf16(w),
                ed=dev_bf16(e))


def test_long_context_read(full_weights):
    shape = configs.LONG_CONTEXT
    assert shape.P == 110707 and shape.C == 256 and shape.d_head == 512
    fw = full_weights
    seed = 11
    st = ReadStep(shape, fw["wd"], fw["ed"], seed=seed)
    assert st.concurrent
    row, req, lab, n = (host(t) for t in (st.slot_row, st.slot_req, st.label_ids, st.n_labels))
    h = inputs.hidden(st.M, shape.D, seed)
    inv_t = inputs.inv_temperature(st.M, seed)
    h, want = margins.prepare_slot_inputs(h, fw["w64"], fw["e"], inv_t, row, req, lab, n, seed,
                                          0, shape.R, shape.gate, ["high", "low", None])
    att = inputs.attention_inputs(shape, seed)
    st.h.copy_(dev_bf16(h))
    st.inv_t.copy_(dev(inv_t))
    for k in ("q", "kc", "vc", "kenc", "venc"):
        getattr(st, k).copy_(dev_bf16(att[k]))
    st.prompt_len.copy_(dev(att["prompt_len"]))
    dg.dg_clear_status()
    st.run(step_idx=0)
    torch.cuda.synchronize()
    st.check()
    got = {k: host(v) for k, v in st.out.items()}
    assert np.array_equal(got["tokens"], want["tokens"])
    assert np.array_equal(got["chosen"], want["chosen"])
    assert np.array_equal(got["resampled"], want["resampled"])
    assert np.array_equal(got["n_reads"], want["n_reads"])
    assert got["resampled"][0] == 1 and got["resampled"][1] == 0
    for s, k in enumerate(n):
        assert_abs(got["q_avg"][s, :k], want["q_avg"][s, :k], what=f"slot {s} distribution")
        assert_abs(got["lp"][s, :, :k], want["lp"][s, :, :k], what=f"slot {s} logprobs")
    assert_abs(got["h_slot"], want["h_slot"], what="slot entropy")
    # the attention over the whole 110,707-token prompt, every row and head
    ref, ref_lse = oracle.attn_decode(att["q"], att["kc"], att["vc"], att["kenc"], att["venc"],
                                      att["prompt_len"], shape.W)
    assert_rel(host(st.attn_out), ref, what="long-context attention")
    assert_abs(host(st.attn_lse), ref_lse, what="long-context attention lse")


def test_batch64_full_step(full_weights):
    shape = configs.scaled(configs.FULL_CANVAS, name="sweep_step_b64", B=64, P=8192)
    fw = full_weights
    seed = 13
    M = shape.B * shape.C
    dev_ = "cuda"
    st = DenoiseStep(shape, fw["wd"], fw["ed"], seed=seed)
    assert st.concurrent and st.n_draw == 0 and st.S == 192       # slots in their own pass
    row, req, lab, n = inputs.slot_table(shape, seed)
    h = inputs.hidden(M, shape.D, seed)
    inv_t = inputs.inv_temperature(M, seed)
    # the slots of three sampled requests carry margins (one forced to resample,
    # one to a dominant label, the rest as drawn)
    reqs = [0, 37, 63]
    sel = np.array([s for s in range(len(row)) if req[s] in reqs])
    modes = ["high", "low", None] * len(reqs)
    h, want = margins.prepare_slot_inputs(h, fw["w64"], fw["e"], inv_t, row, req, lab, n, seed, 0,
                                          shape.R, shape.gate, modes, sel=sel)
    st.h0.copy_(dev_bf16(h))
    st.inv_t.copy_(dev(inv_t))
    # the attention inputs are drawn on the device (2 GB of prompt KV); the sampled
    # requests are copied back for the oracle
    for i, k in enumerate(("q", "kc", "vc", "kenc", "venc")):
        getattr(st, k).copy_(inputs.device_normal_bf16(getattr(st, k).shape, 1.0, 100 + i, dev_))
    st.cand.fill_(1)
    st.set_slots(row, req, lab, n)
    st.reset_state()
    dg.dg_clear_status()
    st.run(step_idx=0)
    torch.cuda.synchronize()
    st.check()

    # heads pass on sampled rows: group boundaries, the last row, random rows
    rng = np.random.default_rng(seed)
    rows = np.unique(np.concatenate([[0, 127, 128, 255, 256, 8191, 8192, M - 1],
                                     rng.choice(M, 8, replace=False)]))
    lse, ent, maxz, arg = oracle.lmhead_stats(h[rows], fw["w64"], inv_t[rows])
    assert_abs(host(st.lse)[rows], lse, what="lse")
    assert_abs(host(st.ent)[rows], ent, what="entropy")
    assert_abs(host(st.maxz)[rows], maxz, what="max logit")
    # self-conditioning (split-K P.E over 16384 rows) on the same rows
    e_ref = oracle.selfcond_embed(h[rows], fw["w64"], fw["e64"], inv_t[rows])
    e_sc = host(st.e_sc)
    assert_rel(e_sc[rows], e_ref, what="expected embedding")

    # every request's commit: the oracle's rule on the GPU's entropies (float64
    # prefix sums), skipped only where a prefix sum lies within 1e-3 of gamma
    ent_all = host(st.ent).astype(np.float64).reshape(shape.B, shape.C)
    arg_all = host(st.argmax).reshape(shape.B, shape.C)
    cand = np.ones((shape.B, shape.C), np.uint8)
    gamma = np.full(shape.B, shape.gamma)
    cm, tk, nc = oracle.commit(ent_all, arg_all, cand, gamma)
    compared = 0
    for b in range(shape.B):
        cs = np.cumsum(np.sort(ent_all[b]))
        if np.min(np.abs(cs - shape.gamma)) <= 1e-3:
            continue
        assert np.array_equal(host(st.commit)[b], cm[b]), f"request {b} commit set"
        assert np.array_equal(host(st.tokens)[b], tk[b]), f"request {b} tokens"
        assert host(st.n_commit)[b] == nc[b] >= 1
        compared += 1
    assert compared >= 60
    # the committed rows' tokens are the full-vocabulary argmax (where it is clear)
    cr = np.nonzero(host(st.commit).reshape(-1))[0][:24]
    z = (h[cr].astype(np.float64) @ fw["w64"].T) * inv_t[cr][:, None]
    clear = top2_gap(z) > margins.ARGMAX_MARGIN
    assert clear.sum() >= 20
    assert np.array_equal(host(st.tokens).reshape(-1)[cr][clear], np.argmax(z, axis=1)[clear])
    # the next canvas input of the sampled rows, from the GPU's own expected embedding
    committed = host(st.committed).reshape(-1)
    tok_state = host(st.tok_state).reshape(-1)
    h_next = oracle.canvas_update(h[rows], e_sc[rows], fw["e"], tok_state[rows], committed[rows])
    assert np.array_equal(host(st.h)[rows], h_next)

    # slot reads of the sampled requests, decisions bit for bit
    got = {k: host(getattr(st, k)) for k in ("chosen", "resampled", "n_reads", "q_avg",
                                            "noise_tok")}
    assert np.array_equal(got["noise_tok"][sel], want["tokens"])
    assert np.array_equal(got["chosen"][sel], want["chosen"])
    assert np.array_equal(got["resampled"][sel], want["resampled"])
    assert np.array_equal(got["n_reads"][sel], want["n_reads"])
    for j, s in enumerate(sel):
        k = n[s]
        assert_abs(got["q_avg"][s, :k], want["q_avg"][j, :k], what=f"slot {s} distribution")

    # attention of two whole requests (every row and head over 8192 prompt keys)
    out = host(st.attn_out)
    lse_a = host(st.attn_lse)
    for b in (0, 63):
        x = {k: host(getattr(st, k)[b:b + 1]) for k in ("q", "kc", "vc", "kenc", "venc")}
        ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                          [shape.P], shape.W)
        assert_rel(out[b:b + 1], ref, what=f"attention, request {b}")
        assert_abs(lse_a[b:b + 1], ref_lse, what=f"attention lse, request {b}")
