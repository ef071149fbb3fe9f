"""GPU parity of the block-scaled NVFP4 lm-head pass (weights and rows both NVFP4 on
tcgen05's kind::mxf4nvf4; tau-home.com, "DiffusionGemma like Jev", "Running NVFP4
locally with a Jev-compatible System One endpoint": the quantised checkpoint).

The quantiser in the pass's layout is bit-exact against the oracle's quantisation
(codes and scale atoms, oracle.to_mma_layout); the statistics are compared with
the oracle's plain statistics of the dequantised rows and weights (each quantised
by the oracle with its own tensor scale), 2e-3 absolute, argmax where the top two
logits are 1e-3 apart; the label gather with the oracle's label logits.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import assert_abs, dev, dev_bf16, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

L = 26


def _quantize(wd, V, D):
    codes = torch.empty(dg.dg_nvfp4_mma_codes_bytes(V, D), dtype=torch.uint8, device="cuda")
    sf = torch.empty(((V + 127) // 128, D // 64, 512), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    assert dg.dg_quantize_nvfp4_mma(wd, V, D, codes, sf, g) == dg.DG_OK
    return codes, sf, g


def _stats(h, codes, sf, g, inv_t, V, D, gather=None):
    M = h.shape[0]
    d = dg.make_dims(d_model=D, V=V)
    f32 = torch.float32
    out = [torch.empty(M, dtype=f32, device="cuda") for _ in range(3)]
    arg = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD_NVFP4_MMA, M), dtype=torch.uint8,
                     device="cuda")
    if gather is None:
        slots = (None, None, None, 0, out[0], out[1], out[2], arg, None, ws)
        lp = None
    else:
        slot_row, ids, n = gather
        lp = torch.full((len(slot_row), L), 12345.0, dtype=f32, device="cuda")
        slots = (dev(slot_row), dev(ids), dev(n), len(slot_row), out[0], out[1], out[2], arg,
                 lp, ws)
    rc = dg.dg_lmhead_logsoftmax_entropy_nvfp4_mma(d, dev_bf16(h), M, codes, sf, g, dev(inv_t),
                                                   *slots)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    res = [host(x) for x in out] + [host(arg)]
    return res + ([host(lp)] if lp is not None else [])


def _dequantized(x):
    """The oracle's NVFP4 quantisation of x (its own tensor scale), dequantised."""
    c, s, g = oracle.quantize_nvfp4(x)
    return oracle.dequantize_nvfp4(c, s, g)


@pytest.mark.parametrize("V,D", [(1000, 256), (4096, 128), (300, 2816), (130, 192), (257, 320)])
def test_quantizer_mma_layout_bit_exact(V, D):
    w = inputs.normal_bf16((V, D), 1.0 / np.sqrt(D), 5 + V, 1)
    w[3, 64:80] = 0.0                         # a zero block
    w[7, :16] *= 40.0                          # a block far above the rest
    w = inputs.to_bf16(w)
    codes, sf, g = _quantize(dev_bf16(w), V, D)
    torch.cuda.synchronize()
    oc, osc, og = oracle.quantize_nvfp4(w)
    packed, atoms = oracle.to_mma_layout(oc, osc)
    assert host(g)[0] == og
    assert np.array_equal(host(codes), packed.reshape(-1))
    assert np.array_equal(host(sf), atoms)


@pytest.mark.parametrize("M,V,D", [(12, 4096, 256), (1, 1024, 64), (16, 3000, 192),
                                   (5, 2500, 2816), (16, 2048, 3072), (7, 1100, 320),
                                   # the GEMM form: one and two 128-row tiles per group,
                                   # ragged rows, vocabularies and K blocks
                                   (17, 2048, 128), (100, 3000, 192), (256, 8192, 512),
                                   (300, 2500, 320), (40, 1000, 3136)])
def test_nvfp4_mma_lmhead_stats(M, V, D):
    h = inputs.hidden(M, D, 11 + M)
    w, _ = inputs.weights(V, D, 12 + V)
    inv_t = inputs.inv_temperature(M, 13)
    codes, sf, g = _quantize(dev_bf16(w), V, D)
    lse, ent, maxz, arg = _stats(h, codes, sf, g, inv_t, V, D)
    oc, osc = oracle.from_mma_layout(host(codes), host(sf), V)
    wq = oracle.dequantize_nvfp4(oc, osc, host(g)[0])
    hq = _dequantized(h)
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(hq, wq, inv_t)
    assert_abs(lse, o_lse, what="lse")
    assert_abs(ent, o_ent, what="entropy")
    assert_abs(maxz, o_maxz, what="max logit")
    z = (hq @ wq.T) * inv_t[:, None]
    clear = top2_gap(z) > 1e-3
    assert clear.sum() >= (M + 1) // 2
    assert np.array_equal(arg[clear], o_arg[clear])


def test_nvfp4_mma_label_gather():
    M, V, D = 12, 4096, 256
    h = inputs.hidden(M, D, 51)
    w, _ = inputs.weights(V, D, 52)
    inv_t = inputs.inv_temperature(M, 53)
    codes, sf, g = _quantize(dev_bf16(w), V, D)
    slot_row = np.array([0, 4, 11], np.int32)
    rng = np.random.default_rng(54)
    ids = np.stack([rng.choice(V, L, replace=False) for _ in slot_row]).astype(np.int32)
    ids[0] = np.arange(L)
    ids[1] = np.arange(V - L, V)
    n = np.array([L, 5, 1], np.int32)
    lse, _, _, _, lp = _stats(h, codes, sf, g, inv_t, V, D, gather=(slot_row, ids, n))
    oc, osc = oracle.from_mma_layout(host(codes), host(sf), V)
    wq = oracle.dequantize_nvfp4(oc, osc, host(g)[0])
    hq = _dequantized(h)
    z = oracle.label_logits(hq[slot_row], wq, inv_t[slot_row], ids, n)
    o_lse, _, _, _ = oracle.lmhead_stats(hq[slot_row], wq, inv_t[slot_row])
    want = z - o_lse[:, None]
    for s in range(len(slot_row)):
        assert_abs(lp[s, :n[s]], want[s, :n[s]], what=f"label lp slot {s}")
        assert np.all(lp[s, n[s]:] == 12345.0)


@pytest.mark.parametrize("M", [12, 256])
def test_nvfp4_mma_full_vocabulary(M):
    """262144 x 2816 weights and 12 slot-draw rows (the skinny pass) or 256 canvas
    rows (the GEMM form): the quantiser on two 128-row tiles and the statistics of
    every row (12) or of sampled rows (256) over the whole vocabulary."""
    V, D = 262144, 2816
    w, _ = inputs.weights(V, D, 77)
    codes, sf, g = _quantize(dev_bf16(w), V, D)
    h = inputs.hidden(M, D, 78)
    inv_t = inputs.inv_temperature(M, 79)
    lse, ent, maxz, arg = _stats(h, codes, sf, g, inv_t, V, D)
    gh = host(g)[0]
    assert gh == oracle.tensor_scale(np.abs(w).max())
    sl = slice(1024, 1280)
    oc, osc, _ = oracle.quantize_nvfp4(w[sl], g=gh)
    packed, atoms = oracle.to_mma_layout(oc, osc)
    blocks = codes.view(V // 128, -1)    # one row of blocks per 128-row tile
    assert np.array_equal(host(blocks[8:10]), packed.reshape(2, -1))
    assert np.array_equal(host(sf[8:10]), atoms)
    oc_all, osc_all = oracle.from_mma_layout(host(codes), host(sf), V)
    wq = oracle.dequantize_nvfp4(oc_all, osc_all, gh)
    rows = np.arange(M) if M <= 16 else np.array([0, 5, 127, 128, 200, 255])
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(_dequantized(h)[rows], wq, inv_t[rows])
    assert_abs(lse[rows], o_lse, what="lse")
    assert_abs(ent[rows], o_ent, what="entropy")
    assert_abs(maxz[rows], o_maxz, what="max logit")


def test_nvfp4_mma_refusals():
    d = dg.make_dims(d_model=256, V=1024)
    buf = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    f = torch.empty(64, dtype=torch.float32, device="cuda")
    i = torch.empty(64, dtype=torch.int32, device="cuda")
    h = torch.zeros((17, 256), dtype=torch.bfloat16, device="cuda")
    # d_model past 3072 with the rows resident (16 or fewer), and not a multiple of 64
    for dm in (3136, 96):
        dd = dg.make_dims(d_model=dm, V=1024)
        rc = dg.dg_lmhead_logsoftmax_entropy_nvfp4_mma(dd, h, 4, buf, buf, f, f, None, None,
                                                       None, 0, f, f, f, i, None, buf)
        assert rc == dg.DG_ERR_SHAPE
    assert dg.dg_quantize_nvfp4_mma(h, 4, 96, buf, buf, f) == dg.DG_ERR_SHAPE
    # a workspace one byte short
    need = dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD_NVFP4_MMA, 4)
    rc = dg.dg_lmhead_logsoftmax_entropy_nvfp4_mma(d, h, 4, buf, buf, f, f, None, None, None, 0,
                                                   f, f, f, i, None, buf[:need - 1])
    assert rc == dg.DG_ERR_WORKSPACE
