"""GPU parity of the encoder-mode prefill (dg_prefill_attn) against the oracle.

Causal attention of each request's prompt over itself on the tensor-core
kernel, the paged KV it writes (bit-exact copies), the decoder-mode read of
those pages, and sampled rows of an 8192-token prompt.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _prefill(x, lens, hq, hkv, page_size=0, seed=0):
    B, P = x["q"].shape[:2]
    d = x["q"].shape[3]
    dims = dg.make_dims(B=B, P_max=P, Hq=hq, Hkv=hkv, d_head=d)
    out = torch.zeros((B, P, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros((B, hq, P), dtype=torch.float32, device="cuda")
    ws = torch.empty(max(dg.dg_workspace_bytes(dims, dg.DG_WS_PREFILL, 0), 256),
                     dtype=torch.uint8, device="cuda")
    pool_k = pool_v = table = None
    ppr = n_pages = 0
    if page_size:
        table_np, n_pages = inputs.page_table(lens, page_size, seed)
        ppr = table_np.shape[1]
        table = dev(table_np)
        pool_k = torch.zeros((n_pages, page_size, hkv, d), dtype=torch.bfloat16, device="cuda")
        pool_v = torch.zeros_like(pool_k)
    dg.dg_clear_status()
    rc = dg.dg_prefill_attn(dims, dev_bf16(x["q"]), dev_bf16(x["k"]), dev_bf16(x["v"]),
                            dev(np.asarray(lens, np.int32)), out, lse, table, ppr, n_pages,
                            page_size, pool_k, pool_v, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    assert dg.dg_get_status() == 0
    res = dict(out=host(out), lse=host(lse))
    if page_size:
        res.update(pool_k=host(pool_k), pool_v=host(pool_v), table=table_np, n_pages=n_pages)
    return res


def _check(got, want_out, want_lse, lens, rows=None):
    for b, n in enumerate(lens):
        idx = np.arange(n) if rows is None else np.array([r for r in rows if r < n])
        if idx.size == 0:
            continue
        assert_rel(got["out"][b, idx], want_out[b, idx], what=f"prefill output, request {b}")
        assert_abs(got["lse"][b][:, idx], want_lse[b][:, idx], what=f"prefill lse, request {b}")
        if rows is None:
            assert np.all(got["out"][b, n:] == 0), "rows past the prompt are not written"


@pytest.mark.parametrize("hq,hkv,lens,P", [
    (8, 2, [300, 77], 300),       # GQA 4:1, two requests, a ragged one
    (8, 1, [200], 200),           # GQA 8:1 (16 positions per query block)
    (2, 2, [129, 0, 31], 160),    # one head per KV head; an empty prompt
])
def test_prefill_reduced(hq, hkv, lens, P):
    x = inputs.prefill_inputs(len(lens), P, hq, hkv, 512, seed=5)
    got = _prefill(x, lens, hq, hkv)
    want_out, want_lse = oracle.prefill_attn(x["q"], x["k"], x["v"], lens)
    _check(got, want_out, want_lse, lens)


def test_prefill_writes_the_pages_decode_reads():
    B, P, hq, hkv, C, W, ps = 3, 260, 8, 2, 64, 16, 16
    lens = [260, 100, 17]
    x = inputs.prefill_inputs(B, P, hq, hkv, 512, seed=8)
    got = _prefill(x, lens, hq, hkv, page_size=ps, seed=8)
    want_out, want_lse = oracle.prefill_attn(x["q"], x["k"], x["v"], lens)
    _check(got, want_out, want_lse, lens)
    pk, pv = oracle.paged_write(x["k"], x["v"], lens, got["table"], ps, got["n_pages"])
    assert np.array_equal(got["pool_k"], pk) and np.array_equal(got["pool_v"], pv)
    # the decoder-mode read of the written pages equals the read of contiguous prompt KV
    from structured_slot_reads_gb300 import configs
    shp = configs.StepShape("t", B=B, C=C, P=P, Hq=hq, Hkv=hkv, d_head=512, W=W, D=8, V=8)
    a = inputs.attention_inputs(shp, 9, prompt_len=np.array(lens, np.int32))
    dims = dg.make_dims(B=B, C=C, P_max=P, Hq=hq, Hkv=hkv, d_head=512, W=W)
    out = torch.empty((B, C, hq, 512), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, hq, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(dims, dg.DG_WS_ATTN, 0), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_attn_decode(dims, dev_bf16(a["q"]), dev_bf16(a["kc"]), dev_bf16(a["vc"]),
                           dev_bf16(got["pool_k"]), dev_bf16(got["pool_v"]), dev(got["table"]),
                           got["table"].shape[1], got["n_pages"], ps,
                           dev(np.array(lens, np.int32)), out, lse, ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attn_decode(a["q"], a["kc"], a["vc"], x["k"], x["v"],
                                      np.array(lens), W)
    assert_rel(host(out), ref, what="decode over the prefill's pages")
    assert_abs(host(lse), ref_lse, what="decode lse over the prefill's pages")


def test_prefill_8192_sampled_rows():
    lens = [8192]
    x = inputs.prefill_inputs(1, 8192, 8, 2, 512, seed=11)
    got = _prefill(x, lens, 8, 2)
    rows = [0, 1, 31, 32, 127, 128, 4095, 4096, 8190, 8191]
    want_out, want_lse = oracle.prefill_attn(x["q"], x["k"], x["v"], lens, rows=rows)
    _check(got, want_out, want_lse, lens, rows=rows)
