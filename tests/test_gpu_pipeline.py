"""HostPipeline: end-to-end steps with host transfers overlapped with compute.

Three consecutive steps of the tiny read shape, each with its own host inputs
(different hidden rows, queries and temperatures), run once serially (upload,
step, download, one after the other) and once through the pipeline (eager
and graph replay): every decision read back must be identical, including the
commit state carried from step to step.
"""
import numpy as np
import pytest

from structured_slot_reads_gb300 import configs, inputs
from structured_slot_reads_gb300.step import DenoiseStep, HostPipeline
from tests.gpu_util import dev, dev_bf16

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _host_inputs(st, shape, seed):
    x = inputs.step_inputs(shape, seed)
    ins, outs = st.host_buffers()
    bf = torch.bfloat16
    ins["h0"].copy_(torch.from_numpy(x["h"]).to(bf))
    ins["inv_t"].copy_(torch.from_numpy(x["inv_t"]))
    for k in ("q", "kc", "vc", "kenc", "venc"):
        ins[k].copy_(torch.from_numpy(x[k]).to(bf))
    ins["cand"].copy_(torch.from_numpy(x["cand"]))
    return ins, outs


def _setup(shape):
    x = inputs.step_inputs(shape, 0)
    st = DenoiseStep(shape, dev_bf16(x["w"]), dev_bf16(x["e"]), seed=3)
    st.prompt_len.copy_(dev(x["prompt_len"]))
    st.set_slots(x["slot_row"], x["slot_req"], x["label_ids"], x["n_labels"])
    return st


@pytest.mark.parametrize("use_graphs", [False, True])
def test_pipeline_matches_serial_steps(use_graphs):
    shape = configs.TINY
    st = _setup(shape)
    bufs = [_host_inputs(st, shape, 10 + i) for i in range(3)]
    # serial reference
    st.reset_state()
    want = []
    for i, (ins, _) in enumerate(bufs):
        outs = st.host_buffers()[1]
        st.upload(ins)
        st.run(step_idx=i)
        st.download(outs)
        torch.cuda.synchronize()
        want.append({k: v.clone() for k, v in outs.items()})
    # pipelined
    pipe = HostPipeline(st, use_graphs=use_graphs)
    if use_graphs:
        pipe.prepare(range(3))              # capture does not execute
        torch.cuda.synchronize()
    st.reset_state()
    total = 0
    for i, (ins, outs) in enumerate(bufs):
        h2d, d2h = pipe.submit(i, ins, outs)
        total += h2d
    assert pipe.sync() == 0     # the device status word read after the steps is clean
    # one arena copy per step: every input tensor plus the alignment gaps
    assert total == 3 * bufs[0][0].arena.numel()
    assert bufs[0][0].arena.numel() >= sum(t.numel() * t.element_size() for t in bufs[0][0].values())
    for i, (_, outs) in enumerate(bufs):
        for k, v in want[i].items():
            assert torch.equal(outs[k], v), (i, k)
    # the steps did commit something, so the carried state was exercised
    assert int(want[-1]["n_commit"].sum()) > 0
