"""The device status path of a bounded wait that runs out, without any GPU fault:
a barrier that nothing arrives on is waited for 20 ms, the kernel records
DG_DEV_TIMEOUT and returns, and the context keeps working afterwards."""
import numpy as np
import pytest

from structured_slot_reads_gb300 import dg
from tests.gpu_util import dev, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def test_wait_that_runs_out_sets_timeout_and_leaves_the_context_usable():
    waited = torch.zeros(1, dtype=torch.int32, device="cuda")
    dg.dg_clear_status()
    assert dg.dg_check_wait_timeout(20_000_000, waited) == dg.DG_OK
    torch.cuda.synchronize()
    assert dg.dg_get_status() & dg.DG_DEV_TIMEOUT
    us = int(host(waited)[0])
    assert 20_000 <= us < 1_000_000
    dg.dg_clear_status()
    assert dg.dg_get_status() == 0
    # the same context runs a library kernel normally afterwards
    chosen = dev(np.array([2, 0], np.int32))
    lab2 = torch.empty((1, 26), dtype=torch.int32, device="cuda")
    n2 = torch.empty(1, dtype=torch.int32, device="cuda")
    rc = dg.dg_ask_if_select(chosen, 2, dev(np.array([0], np.int32)), dev(np.array([2], np.int32)),
                             dev(np.array([0], np.int32)), dev(np.full((1, 26), 5, np.int32)),
                             dev(np.array([3], np.int32)), 1, 1, lab2, n2)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    assert int(host(n2)[0]) == 3 and dg.dg_get_status() == 0
