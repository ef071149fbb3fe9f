"""GPU parity of one attention launch over a batch mixing decoder-mode and
encoder-mode requests (dg_attn_mixed) against the oracle, contiguous and paged."""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("mode,rows,plen", [
    ([0, 1, 0, 1], [64, 300, 40, 129], [200, 0, 77, 0]),    # two of each, ragged
    ([1, 0], [256, 256], [0, 1000]),                        # prefill beside a full canvas
])
def test_mixed_batch_matches_oracle(paged, mode, rows, plen):
    B, C, hq, hkv, W = len(mode), max(rows), 8, 2, 32
    P = max(max(plen), 1)
    shp = configs.StepShape("t", B=B, C=C, P=P, Hq=hq, Hkv=hkv, d_head=512, W=W, D=8, V=8)
    x = inputs.attention_inputs(shp, 13, prompt_len=np.maximum(np.array(plen, np.int32), 0))
    dims = dg.make_dims(B=B, C=C, P_max=P, Hq=hq, Hkv=hkv, d_head=512, W=W)
    out = torch.zeros((B, C, hq, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, hq, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(dg.dg_workspace_bytes(dims, dg.DG_WS_ATTN, 0), 256), dtype=torch.uint8,
                     device="cuda")
    if paged:
        pk, pv, table = inputs.paged_layout(x["kenc"], x["venc"], np.array(plen), 16, 13)
        ke, ve, tb, ppr, npg, ps = dev_bf16(pk), dev_bf16(pv), dev(table), table.shape[1], \
            pk.shape[0], 16
    else:
        ke, ve, tb, ppr, npg, ps = dev_bf16(x["kenc"]), dev_bf16(x["venc"]), None, 0, 0, 0
    dg.dg_clear_status()
    rc = dg.dg_attn_mixed(dims, dev(np.array(mode, np.int32)), dev(np.array(rows, np.int32)),
                          dev_bf16(x["q"]), dev_bf16(x["kc"]), dev_bf16(x["vc"]), ke, ve, tb, ppr,
                          npg, ps, dev(np.array(plen, np.int32)), out, lse, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    assert dg.dg_get_status() == 0
    ref, ref_lse = oracle.attn_mixed(mode, rows, x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                     np.array(plen), W)
    got, got_lse = host(out), host(lse)
    for b, n in enumerate(rows):
        assert_rel(got[b, :n], ref[b, :n], what=f"request {b} (mode {mode[b]})")
        assert_abs(got_lse[b][:, :n], ref_lse[b][:, :n], what=f"request {b} lse")
        assert np.all(got[b, n:] == 0), "rows past rows_len are not written"
