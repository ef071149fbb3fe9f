"""GPU parity of the 4-bit lm-head pass: the NVFP4 quantiser (bit-exact against the
oracle's quantisation, in the K-block-major layout) and the statistics pass
against NVFP4 weights (against the oracle's plain statistics of the dequantised
weights, 2e-3 absolute; argmax where the top two logits are 1e-3 apart)."""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import assert_abs, dev, dev_bf16, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _quantize(wd, V, D):
    codes = torch.empty((D // 64, V, 32), dtype=torch.uint8, device="cuda")
    scales = torch.empty((D // 64, V, 4), dtype=torch.uint8, device="cuda")
    g = torch.empty(1, dtype=torch.float32, device="cuda")
    assert dg.dg_quantize_nvfp4(wd, V, D, codes, scales, g) == dg.DG_OK
    return codes, scales, g


def _stats(h, codes, scales, g, inv_t, V, D):
    M = h.shape[0]
    d = dg.make_dims(d_model=D, V=V)
    f32 = torch.float32
    out = [torch.empty(M, dtype=f32, device="cuda") for _ in range(3)]
    arg = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, M), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_lmhead_logsoftmax_entropy_nvfp4(d, dev_bf16(h), M, codes, scales, g, dev(inv_t),
                                               None, None, None, 0, out[0], out[1], out[2], arg,
                                               None, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return [host(x) for x in out] + [host(arg)]


@pytest.mark.parametrize("V,D", [(1000, 256), (4096, 128), (300, 2816)])
def test_quantizer_bit_exact(V, D):
    w = inputs.normal_bf16((V, D), 1.0 / np.sqrt(D), 5 + V, 1)
    w[3, 64:80] = 0.0                         # a zero block
    w[7, :16] *= 40.0                          # a block far above the rest
    w = inputs.to_bf16(w)                      # the operand both sides read
    codes, scales, g = _quantize(dev_bf16(w), V, D)
    torch.cuda.synchronize()
    oc, osc, og = oracle.quantize_nvfp4(w)
    ckb, skb = oracle.to_kblock_layout(oc, osc)
    assert host(g)[0] == og
    assert np.array_equal(host(codes), ckb)
    assert np.array_equal(host(scales), skb)


@pytest.mark.parametrize("M,V,D", [(12, 4096, 256), (256, 8192, 512), (300, 3000, 192),
                                   (1, 1024, 64), (16, 3000, 192), (17, 2048, 128)])
def test_nvfp4_lmhead_stats(M, V, D):
    h = inputs.hidden(M, D, 11 + M)
    w, _ = inputs.weights(V, D, 12 + V)
    inv_t = inputs.inv_temperature(M, 13)
    codes, scales, g = _quantize(dev_bf16(w), V, D)
    lse, ent, maxz, arg = _stats(h, codes, scales, g, inv_t, V, D)
    oc, osc = oracle.from_kblock_layout(host(codes), host(scales))
    wq = oracle.dequantize_nvfp4(oc, osc, host(g)[0])
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(h, wq, inv_t)
    assert_abs(lse, o_lse, what="lse")
    assert_abs(ent, o_ent, what="entropy")
    assert_abs(maxz, o_maxz, what="max logit")
    z = (h.astype(np.float64) @ wq.T) * inv_t[:, None]
    clear = top2_gap(z) > 1e-3
    assert clear.sum() >= M // 2
    assert np.array_equal(arg[clear], o_arg[clear])


@pytest.mark.parametrize("M", [256, 12])
def test_nvfp4_lmhead_full_vocabulary_sampled_rows(M):
    """262144 x 2816 weights: the quantiser on a slice of rows (with the whole
    tensor's scale) and the statistics of sampled rows: 256 canvas rows (the
    GEMM form) and 12 slot-draw rows (the skinny form, rows resident)."""
    V, D = 262144, 2816
    w, _ = inputs.weights(V, D, 77)
    wd = dev_bf16(w)
    codes, scales, g = _quantize(wd, V, D)
    h = inputs.hidden(M, D, 78)
    inv_t = inputs.inv_temperature(M, 79)
    lse, ent, maxz, arg = _stats(h, codes, scales, g, inv_t, V, D)
    gh = host(g)[0]
    assert gh == oracle.tensor_scale(np.abs(w).max())
    # quantiser bit-exact on rows [1000, 1256) of every K block
    sl = slice(1000, 1256)
    oc, osc, _ = oracle.quantize_nvfp4(w[sl], g=gh)
    ckb, skb = oracle.to_kblock_layout(oc, osc)
    assert np.array_equal(host(codes[:, sl]), ckb)
    assert np.array_equal(host(scales[:, sl]), skb)
    oc_all, osc_all = oracle.from_kblock_layout(host(codes), host(scales))
    wq = oracle.dequantize_nvfp4(oc_all, osc_all, gh)
    rows = np.array([0, 5, 127, 128, 200, 255]) if M == 256 else np.arange(M)
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(h[rows], wq, inv_t[rows])
    assert_abs(lse[rows], o_lse, what="lse")
    assert_abs(ent[rows], o_ent, what="entropy")
    assert_abs(maxz[rows], o_maxz, what="max logit")


@pytest.mark.parametrize("M", [12, 40])
def test_nvfp4_lmhead_tiny_block_scales(M):
    """One block far above the rest makes the tensor scale large, so every other
    block's e4m3 scale is small and its widened products are tiny (below f16's
    normal range in the skinny form, which works in f16 times 2^-14).  Rows of
    magnitude ~400 make the logits depend on those products alone (the large
    block meets zero row entries): flushing them would move lse by several nats."""
    V, D = 1024, 256
    w = inputs.normal_bf16((V, D), 1e-3, 91, 1)
    w[0, :16] = 1000.0
    w = inputs.to_bf16(w)
    h = inputs.normal_bf16((M, D), 400.0, 92, 1)
    h[:, :16] = 0.0
    h = inputs.to_bf16(h)
    inv_t = np.ones(M, np.float32)
    codes, scales, g = _quantize(dev_bf16(w), V, D)
    lse, ent, maxz, arg = _stats(h, codes, scales, g, inv_t, V, D)
    oc, osc = oracle.from_kblock_layout(host(codes), host(scales))
    wq = oracle.dequantize_nvfp4(oc, osc, host(g)[0])
    # every other block: e2m1 x scale below 1, i.e. below 2^-14 once times 2^-14
    assert (np.abs(wq[1:]) / host(g)[0]).max() < 1.0
    o_lse, o_ent, o_maxz, _ = oracle.lmhead_stats(h, wq, inv_t)
    assert np.all(o_lse - np.log(V) > 1.0)                         # logits far from flat
    assert_abs(lse, o_lse, what="lse (tiny block scales)")
    assert_abs(ent, o_ent, what="entropy (tiny block scales)")
    assert_abs(maxz, o_maxz, what="max logit (tiny block scales)")
