"""The read-only step against an NVFP4 checkpoint (ReadStep(fp4=True); tau-home.com,
"Running NVFP4 locally with a Jev-compatible System One endpoint"), on the GPU.

The slot read is dg_slot_noise, the block-scaled pass over the draw rows (rows
and weights NVFP4, one gathered label row per draw) and dg_slot_finish: 12 draw
rows (one request: the skinny pass) or 24 (two requests: the GEMM form).  Against
the oracle on the same operands: the noise rows exactly as dg_slot_noise forms
them, quantised to NVFP4 with their own tensor scale, the weights quantised the
same way, then the plain label logits, log-normalisers and slot read of the
dequantised operands.  Tokens bit-exact; label logprobs and slot distributions
2e-3 absolute; the gate, the number of reads and the choice exact, on inputs
re-drawn until every slot's entropy is 1e-3 away from the gate and its top two
probabilities are 1e-3 apart.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from structured_slot_reads_gb300.read import ReadStep
from tests.gpu_util import assert_abs, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L = dg.MAX_LABELS


def _dequantized(x):
    c, s, g = oracle.quantize_nvfp4(x)
    return oracle.dequantize_nvfp4(c, s, g)


def _want(x, row, req, lab, n, shape, step, wq):
    R, V = shape.R, shape.V
    rows, toks = oracle.slot_noise_rows(x["h"], x["e"], row, req, 0, step, R, V)
    inv_d = np.repeat(x["inv_t"][row], R)
    rq = _dequantized(rows)
    z = oracle.label_logits(rq, wq, inv_d, np.repeat(lab, R, axis=0), np.repeat(n, R))
    lse, _, _, _ = oracle.lmhead_stats(rq, wq, inv_d)
    want = oracle.slot_read(z.reshape(len(row), R, L), lse.reshape(len(row), R), n, R, shape.gate)
    want["tokens"] = toks
    return want


def _margins_ok(want, n, gate):
    for s, k in enumerate(n):
        if k == 0:
            continue
        if abs(want["h_draw"][s, 0] - gate) <= 1e-3:
            return False
        q = np.sort(want["q_avg"][s, :k])[::-1]
        if k > 1 and q[0] - q[1] <= 1e-3:
            return False
    return True


@pytest.mark.parametrize("B", [1, 2])
def test_read_step_nvfp4_matches_oracle(B):
    shape = configs.scaled(configs.SINGLE_READ, B=B, C=128, P=600, D=256, V=4096,
                           slots=[(61, 2), (100, 26), (120, 5)])
    step = 2
    for seed in range(4, 30):
        x = inputs.step_inputs(shape, seed=seed)
        st = ReadStep(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=0, concurrent=False,
                      fp4=True)
        row, req, lab, n = (host(t) for t in (st.slot_row, st.slot_req, st.label_ids,
                                              st.n_labels))
        oc, osc = oracle.from_mma_layout(host(st.codes), host(st.sf), shape.V)
        wq = oracle.dequantize_nvfp4(oc, osc, host(st.g)[0])
        want = _want(x, row, req, lab, n, shape, step, wq)
        if _margins_ok(want, n, shape.gate):
            break
    else:
        pytest.fail("no seed gave every slot its margins")
    # the weights' quantisation itself is the oracle's
    c_o, s_o, g_o = oracle.quantize_nvfp4(x["w"])
    assert host(st.g)[0] == g_o and np.array_equal(oc, c_o) and np.array_equal(osc, s_o)
    st.h.copy_(dev_bf16(x["h"]))
    st.inv_t.copy_(dev(x["inv_t"]))
    for k in ("q", "kc", "vc", "kenc", "venc"):
        getattr(st, k).copy_(dev_bf16(x[k]))
    st.prompt_len.copy_(dev(x["prompt_len"]))
    keys = ("q_avg", "h_slot", "chosen", "lp", "resampled", "n_reads", "tokens")
    dg.dg_clear_status()
    st.run(step_idx=step)
    torch.cuda.synchronize()
    st.check()
    got = {k: host(st.out[k]).copy() for k in keys}
    assert np.array_equal(got["tokens"], want["tokens"])
    compared = 0
    for s, k in enumerate(n):
        assert_abs(got["lp"][s, :, :k], want["lp"][s, :, :k], what=f"label logprobs slot {s}")
        assert_abs(got["q_avg"][s, :k], want["q_avg"][s, :k], what=f"slot distribution {s}")
        compared += 1
    assert compared == len(n)
    assert np.array_equal(got["chosen"], want["chosen"])
    assert np.array_equal(got["resampled"], want["resampled"])
    assert np.array_equal(got["n_reads"], want["n_reads"])
    # the side-stream schedule gives the same slot read bit for bit
    serial = got
    st.concurrent = True
    st.run(step_idx=step)
    torch.cuda.synchronize()
    for k in keys:
        assert np.array_equal(host(st.out[k]), serial[k]), k
