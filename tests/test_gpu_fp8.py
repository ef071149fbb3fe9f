"""GPU parity of the 8-bit lm-head pass: the e4m3 row quantiser (bit-exact) and the
statistics of the quantised operands against the oracle's float64 statistics of
the dequantised operands."""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from tests.gpu_util import assert_abs, dev, dev_bf16, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _quantize(x):
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    assert dg.dg_quantize_rows_e4m3(dev_bf16(x), rows, cols, q, sc) == dg.DG_OK
    torch.cuda.synchronize()
    return q, sc


def _fp8_stats(q_h, s_h, q_w, s_w, inv_t, D, V):
    M = q_h.shape[0]
    d = dg.make_dims(d_model=D, V=V)
    f = lambda: torch.empty(M, dtype=torch.float32, device="cuda")  # noqa: E731
    lse, ent, mz = f(), f(), f()
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, M), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_lmhead_logsoftmax_entropy_fp8(d, q_h, s_h, M, q_w, s_w, dev(inv_t), lse, ent, mz,
                                             am, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return host(lse), host(ent), host(mz), host(am)


def test_quantize_rows_bit_exact():
    x = inputs.normal_bf16((64, 2816), 1.0, 7, 1)
    x[5] = 0.0
    x[9] *= np.float32(1e-4)
    x[11, ::7] *= np.float32(300.0)   # wide dynamic range: many values land on subnormals
    x = inputs.to_bf16(x)
    q, sc = _quantize(x)
    wq, wsc = oracle.quantize_rows_e4m3(x)
    assert np.array_equal(host(sc), wsc)
    assert np.array_equal(host(q), wq)


@pytest.mark.parametrize("M", [12, 64, 200])
def test_fp8_lmhead_matches_oracle(M):
    V, D = 4096, 256
    h = inputs.hidden(M, D, 3)
    w, _ = inputs.weights(V, D, 3)
    inv_t = inputs.inv_temperature(M, 3)
    q_h, s_h = _quantize(h)
    q_w, s_w = _quantize(w)
    lse, ent, mz, am = _fp8_stats(q_h, s_h, q_w, s_w, inv_t, D, V)
    hd = oracle.dequantize_rows(host(q_h), host(s_h))
    wd = oracle.dequantize_rows(host(q_w), host(s_w))
    o_lse, o_ent, o_mz, o_am = oracle.lmhead_stats(hd, wd, inv_t)
    assert_abs(lse, o_lse, what="fp8 lse")
    assert_abs(ent, o_ent, what="fp8 entropy")
    assert_abs(mz, o_mz, what="fp8 max logit")
    gap = top2_gap((hd @ wd.T) * inv_t[:, None])
    ok = gap > 1e-3
    assert ok.sum() >= M // 2
    assert np.array_equal(am[ok], o_am[ok])


def test_fp8_lmhead_full_vocabulary_sampled_rows():
    """Full 262144 x 2816 W; 256 canvas rows; 16 rows compared with the oracle."""
    shape = configs.FULL_CANVAS
    w, _ = inputs.weights(shape.V, shape.D, 11)
    M = 256
    h = inputs.hidden(M, shape.D, 11)
    inv_t = inputs.inv_temperature(M, 11)
    q_w, s_w = _quantize(w)
    q_h, s_h = _quantize(h)
    lse, ent, mz, am = _fp8_stats(q_h, s_h, q_w, s_w, inv_t, shape.D, shape.V)
    rows = np.random.default_rng(0).choice(M, 16, replace=False)
    hd = oracle.dequantize_rows(host(q_h)[rows], host(s_h)[rows])
    wd = oracle.dequantize_rows(host(q_w), host(s_w))
    o_lse, o_ent, o_mz, _ = oracle.lmhead_stats(hd, wd, inv_t[rows])
    assert_abs(lse[rows], o_lse, what="fp8 lse (full vocabulary)")
    assert_abs(ent[rows], o_ent, what="fp8 entropy (full vocabulary)")
    assert_abs(mz[rows], o_mz, what="fp8 max logit (full vocabulary)")
