"""GPU parity of the 8-bit lm-head pass: the e4m3 row quantiser (bit-exact) and the
statistics of the quantised operands against the oracle's float64 statistics of
the dequantised operands."""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import configs, dg, inputs
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host, top2_gap

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
    rc = dg.dg_lmhead_logsoftmax_entropy_fp8(d, q_h, s_h, M, q_w, s_w, dev(inv_t), None, None,
                                             None, 0, lse, ent, mz, am, None, ws)
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


@pytest.mark.parametrize("cols", [16392, 40960])
def test_quantize_long_rows_bit_exact(cols):
    """Rows of at least 16384 values take the chunked path (many blocks per row)."""
    x = inputs.normal_bf16((6, cols), 1.0, 8, cols)
    x[2] = 0.0
    x[4] *= np.float32(1e-5)
    x[5, ::11] += np.float32(12.0)     # a few values 2^17 above the rest: subnormals
    x = inputs.to_bf16(np.exp(x).astype(np.float32) * (np.arange(6)[:, None] != 2))
    assert np.all(np.isfinite(x))
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


# ---- the self-conditioning P . E on 8-bit operands -------------------------
def _quantize_cols(x):
    rows, cols = x.shape
    qt = torch.empty((cols, rows), dtype=torch.uint8, device="cuda")
    sc = torch.empty(cols, dtype=torch.float32, device="cuda")
    assert dg.dg_quantize_cols_e4m3(dev_bf16(x), rows, cols, qt, sc) == dg.DG_OK
    torch.cuda.synchronize()
    return qt, sc


def _probs(M, V, seed):
    """Positive, skewed bf16 rows standing in for the unnormalised probabilities."""
    z = inputs.normal_bf16((M, V), 1.0, seed, 9)
    return inputs.to_bf16(np.exp(1.5 * z).astype(np.float32))


def _pe8(p8, p_scale, row_scale, e8t, e_scale, M, V, D):
    d = dg.make_dims(d_model=D, V=V)
    out = torch.empty((M, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_PROBS_EMBED8, M), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_selfcond_from_probs8(d, p8, p_scale, row_scale, M, e8t, e_scale, out, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return host(out)


@pytest.mark.parametrize("rows,cols", [(4096, 256), (1000, 200), (300, 70)])
def test_quantize_cols_bit_exact(rows, cols):
    x = inputs.normal_bf16((rows, cols), 0.05, 11, rows)
    x[:, 3] = 0.0
    x[::13, 5] *= np.float32(200.0)
    x = inputs.to_bf16(x)
    qt, sc = _quantize_cols(x)
    wq, wsc = oracle.quantize_cols_e4m3(x)
    assert np.array_equal(host(sc), wsc)
    assert np.array_equal(host(qt), wq)


@pytest.mark.parametrize("M,V,D", [(256, 8192, 256), (100, 4096, 200), (300, 4096, 128)])
def test_selfcond_from_probs8_matches_oracle(M, V, D):
    """Probabilities quantised per row on the GPU (bit-exact, checked) and E per
    column; the GEMM of the quantised operands against the float64 definition."""
    p = _probs(M, V, M)
    e = inputs.normal_bf16((V, D), D ** -0.5, 5, D)
    row_scale = (1.0 / inputs.inv_temperature(M, 4)).astype(np.float32)   # any positive factor
    p8, p_s = _quantize(p)
    e8t, e_s = _quantize_cols(e)
    wp8, wps = oracle.quantize_rows_e4m3(p)
    we8t, wes = oracle.quantize_cols_e4m3(e)
    assert np.array_equal(host(p8), wp8) and np.array_equal(host(e8t), we8t)
    got = _pe8(p8, p_s, dev(row_scale), e8t, e_s, M, V, D)
    want = oracle.selfcond_fp8(wp8, wps, row_scale, we8t, wes)
    assert_rel(got, want, tol=1e-4, what="8-bit P.E")
    got1 = _pe8(p8, p_s, None, e8t, e_s, M, V, D)          # row_scale NULL means 1
    assert_rel(got1, oracle.selfcond_fp8(wp8, wps, None, we8t, wes), tol=1e-4, what="no row scale")


def test_selfcond_from_probs8_full_vocabulary_sampled():
    """Full 256 x 262144 x 2816 shapes: sampled columns of the quantised E and
    sampled outputs against the oracle."""
    M, V, D = 256, configs.FULL_CANVAS.V, configs.FULL_CANVAS.D
    _, e = inputs.weights(V, D, 2025)
    p = _probs(M, V, 7)
    p8, p_s = _quantize(p)
    e8t, e_s = _quantize_cols(e)
    cols = np.array([0, 1, 255, 256, 1407, 2047, 2048, 2815])
    we8t, wes = oracle.quantize_cols_e4m3(e[:, cols])
    g8 = host(e8t[torch.from_numpy(cols).cuda()])
    assert np.array_equal(g8, we8t) and np.array_equal(host(e_s)[cols], wes)
    rows = np.array([0, 127, 128, 255])
    wp8, wps = oracle.quantize_rows_e4m3(p[rows])
    assert np.array_equal(host(p8)[rows], wp8)
    got = _pe8(p8, p_s, None, e8t, e_s, M, V, D)
    want = oracle.selfcond_fp8(wp8, wps, None, we8t, wes)
    assert_rel(got[np.ix_(rows, cols)], want, tol=1e-4, what="8-bit P.E, full vocabulary")
