"""The lm-head pass for callers that cannot allocate device memory.

dg_lmhead_logsoftmax_entropy_noalloc takes no workspace: its scratch is a fixed
array inside the library, for callers whose allocator is closed to them.  It
must give what dg_lmhead_logsoftmax_entropy gives (with a caller-allocated
workspace) on the same inputs, on consecutive calls that reuse the array, and
reject row counts beyond the array's capacity.  This file is collected last so
a stop-at-first-failure run has already run every other test; it also passes on
its own in a fresh process.
"""
import numpy as np
import pytest

from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import TOL_LOGPROB, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _outs(M):
    f = [torch.empty(M, dtype=torch.float32, device="cuda") for _ in range(3)]
    return f + [torch.empty(M, dtype=torch.int32, device="cuda")]


def _with_workspace(d, h, M, w, it):
    lse, ent, mz, arg = _outs(M)
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, M), dtype=torch.uint8,
                     device="cuda")
    assert dg.dg_lmhead_logsoftmax_entropy(d, h, M, w, it, None, None, None, 0, lse, ent, mz, arg,
                                           None, ws) == dg.DG_OK
    return lse, ent, mz, arg


def _without_workspace(d, h, M, w, it):
    lse, ent, mz, arg = _outs(M)
    rc = dg.dg_lmhead_logsoftmax_entropy_noalloc(d, h, M, w, it, lse, ent, mz, arg)
    assert rc == dg.DG_OK, dg.strerror(rc)
    return lse, ent, mz, arg


def test_noalloc_matches_workspace_path_on_two_calls_in_a_row():
    V, D = 8192, 512
    d = dg.make_dims(d_model=D, V=V)
    w, _ = inputs.weights(V, D, 21)
    wd = dev_bf16(w)
    # two consecutive calls with different shapes and inputs share the scratch array
    for call, M in enumerate((300, 12)):
        h = dev_bf16(inputs.hidden(M, D, 40 + call))
        it = dev(inputs.inv_temperature(M, 50 + call))
        ref = _with_workspace(d, h, M, wd, it)
        got = _without_workspace(d, h, M, wd, it)
        torch.cuda.synchronize()
        for a, b in zip(got[:3], ref[:3]):
            assert np.max(np.abs(host(a) - host(b))) <= TOL_LOGPROB
        assert np.array_equal(host(got[3]), host(ref[3]))
    assert dg.dg_get_status() == 0


def test_noalloc_rejects_rows_beyond_the_fixed_scratch():
    d = dg.make_dims(d_model=128, V=1024)
    M = dg.DG_NOALLOC_MAX_ROWS + 1
    x = torch.zeros((M, 128), dtype=torch.bfloat16, device="cuda")
    lse, ent, mz, arg = _outs(M)
    rc = dg.dg_lmhead_logsoftmax_entropy_noalloc(d, x, M, x, lse, lse, ent, mz, arg)
    assert rc == dg.DG_ERR_SHAPE
