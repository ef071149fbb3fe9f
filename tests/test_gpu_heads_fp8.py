"""GPU parity of the fused pass on e4m3 operands (dg_denoise_heads_fp8; tau-home.com,
"Running NVFP4 locally with a Jev-compatible System One endpoint"; 24-ai.news,
"Measured performance": the FP8 checkpoint).

Canvas rows, draw rows and W are quantised by dg_quantize_rows_e4m3 (checked
bit-exact against the oracle in test_gpu_fp8.py); the pass is compared with the
oracle's float64 statistics of the dequantised operands: lse, entropy and max
logit 2e-3 absolute, argmax where the top two logits are 1e-3 apart, the draw
rows' normalisers 2e-3, their gathered label logits 2e-3, and the normalised
probabilities 1e-2 relative against the softmax of the dequantised logits.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import assert_abs, dev, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L = dg.MAX_LABELS


def _quantize(x):
    rows, cols = x.shape
    q = torch.empty((rows, cols), dtype=torch.uint8, device="cuda")
    sc = torch.empty(rows, dtype=torch.float32, device="cuda")
    xd = torch.from_numpy(np.ascontiguousarray(x)).to("cuda").to(torch.bfloat16)
    assert dg.dg_quantize_rows_e4m3(xd, rows, cols, q, sc) == dg.DG_OK
    torch.cuda.synchronize()
    return q, sc


def _run(q_h, s_h, q_d, s_d, q_w, s_w, inv_t, inv_d, V, D, gather=None):
    M = q_h.shape[0]
    nd = 0 if q_d is None else q_d.shape[0]
    d = dg.make_dims(d_model=D, V=V)
    f32 = torch.float32
    lse, ent, mz = (torch.empty(M, dtype=f32, device="cuda") for _ in range(3))
    am = torch.empty(M, dtype=torch.int32, device="cuda")
    lse_d = torch.empty(max(nd, 1), dtype=f32, device="cuda")
    scale = torch.empty(M, dtype=f32, device="cuda")
    ld = dg.dg_probs_ld(V)
    probs = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_HEADS, M), dtype=torch.uint8,
                     device="cuda")
    ids = n = lz = None
    R = 0
    if gather is not None:
        ids_h, n_h, R = gather
        ids, n = dev(ids_h), dev(n_h)
        lz = torch.full((nd, L), 12345.0, dtype=f32, device="cuda")
    rc = dg.dg_denoise_heads_fp8(d, q_h, s_h, M, q_d, s_d, nd, q_w, s_w, dev(inv_t),
                                 dev(inv_d) if nd else None, lse, ent, mz, am,
                                 lse_d if nd else None, ids, n, R, lz, scale, probs, ld, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    out = dict(lse=host(lse), ent=host(ent), mz=host(mz), am=host(am), lse_d=host(lse_d)[:nd],
               p=host(probs)[:, :V].astype(np.float64) * host(scale)[:, None])
    if lz is not None:
        out["lz"] = host(lz)
    return out


@pytest.mark.parametrize("M,nd,V,D", [(256, 12, 4096, 256), (100, 5, 3000, 192),
                                      (1, 16, 1024, 128), (300, 0, 2500, 320),
                                      (64, 0, 4096, 256), (384, 16, 2504, 144)])
def test_fp8_heads_matches_oracle(M, nd, V, D):
    h = inputs.hidden(M, D, 21 + M)
    w, _ = inputs.weights(V, D, 22 + V)
    inv_t = inputs.inv_temperature(M, 23)
    draws = inputs.hidden(nd, D, 24) if nd else None
    inv_d = inputs.inv_temperature(nd, 25) if nd else None
    q_h, s_h = _quantize(h)
    q_w, s_w = _quantize(w)
    q_d, s_d = _quantize(draws) if nd else (None, None)
    got = _run(q_h, s_h, q_d, s_d, q_w, s_w, inv_t, inv_d, V, D)
    hd = oracle.dequantize_rows(host(q_h), host(s_h))
    wd = oracle.dequantize_rows(host(q_w), host(s_w))
    o_lse, o_ent, o_mz, o_am = oracle.lmhead_stats(hd, wd, inv_t)
    assert_abs(got["lse"], o_lse, what="fp8 heads lse")
    assert_abs(got["ent"], o_ent, what="fp8 heads entropy")
    assert_abs(got["mz"], o_mz, what="fp8 heads max logit")
    z = (hd @ wd.T) * inv_t[:, None]
    clear = top2_gap(z) > 1e-3
    assert clear.sum() >= (M + 1) // 2
    assert np.array_equal(got["am"][clear], o_am[clear])
    ref_p = np.exp(z - o_lse[:, None])
    np.testing.assert_allclose(got["p"].sum(axis=1), 1.0, atol=5e-3)
    assert np.max(np.abs(got["p"] - ref_p) / (ref_p + 1e-30)) < 1e-2
    if nd:
        dd = oracle.dequantize_rows(host(q_d), host(s_d))
        d_lse, _, _, _ = oracle.lmhead_stats(dd, wd, inv_d)
        assert_abs(got["lse_d"], d_lse, what="fp8 draw-row lse")


def test_fp8_heads_label_gather():
    """Three slots of four draws: each draw's label logits z/T gathered from the
    accumulators, against the oracle's label logits of the dequantised operands."""
    M, V, D, R = 64, 4096, 256, 4
    S = 3
    nd = S * R
    h = inputs.hidden(M, D, 31)
    w, _ = inputs.weights(V, D, 32)
    inv_t = inputs.inv_temperature(M, 33)
    draws = inputs.hidden(nd, D, 34)
    inv_d = inputs.inv_temperature(nd, 35)
    rng = np.random.default_rng(36)
    ids = np.stack([rng.choice(V, L, replace=False) for _ in range(S)]).astype(np.int32)
    ids[0] = np.arange(L)                 # the first tile's rows
    ids[1] = np.arange(V - L, V)          # the last (ragged) tile's rows
    n = np.array([L, 7, 1], np.int32)
    q_h, s_h = _quantize(h)
    q_w, s_w = _quantize(w)
    q_d, s_d = _quantize(draws)
    got = _run(q_h, s_h, q_d, s_d, q_w, s_w, inv_t, inv_d, V, D, gather=(ids, n, R))
    wd = oracle.dequantize_rows(host(q_w), host(s_w))
    dd = oracle.dequantize_rows(host(q_d), host(s_d))
    want = oracle.label_logits(dd, wd, inv_d, np.repeat(ids, R, axis=0), np.repeat(n, R))
    for j in range(nd):
        k = n[j // R]
        assert_abs(got["lz"][j, :k], want[j, :k], what=f"fp8 label logits draw {j}")
        assert np.all(got["lz"][j, k:] == 12345.0)


def test_fp8_heads_full_vocabulary_sampled_rows():
    """262144 x 2816 W, 256 canvas rows and 12 draw rows: sampled canvas rows and
    every draw row's normaliser against the oracle over the whole vocabulary."""
    M, nd, V, D = 256, 12, 262144, 2816
    w, _ = inputs.weights(V, D, 41)
    h = inputs.hidden(M, D, 42)
    inv_t = inputs.inv_temperature(M, 43)
    draws = inputs.hidden(nd, D, 44)
    inv_d = inputs.inv_temperature(nd, 45)
    q_w, s_w = _quantize(w)
    del w
    q_h, s_h = _quantize(h)
    q_d, s_d = _quantize(draws)
    got = _run(q_h, s_h, q_d, s_d, q_w, s_w, inv_t, inv_d, V, D)
    rows = np.array([0, 7, 127, 128, 200, 255])
    wd = oracle.dequantize_rows(host(q_w), host(s_w))
    hd = oracle.dequantize_rows(host(q_h)[rows], host(s_h)[rows])
    o_lse, o_ent, o_mz, _ = oracle.lmhead_stats(hd, wd, inv_t[rows])
    assert_abs(got["lse"][rows], o_lse, what="fp8 heads lse (full vocabulary)")
    assert_abs(got["ent"][rows], o_ent, what="fp8 heads entropy (full vocabulary)")
    assert_abs(got["mz"][rows], o_mz, what="fp8 heads max logit (full vocabulary)")
    dd = oracle.dequantize_rows(host(q_d), host(s_d))
    d_lse, _, _, _ = oracle.lmhead_stats(dd, wd, inv_d)
    assert_abs(got["lse_d"], d_lse, what="fp8 draw-row lse (full vocabulary)")
