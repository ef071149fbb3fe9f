"""GPU parity of each library call against the float64 oracle (through the C ABI).

Sizes are chosen so the oracle finishes in seconds while the kernels still see
several tiles and ragged tails: vocabularies that are not multiples of the
256-wide vocabulary tile, d_model not a multiple of the 64-wide K block, more
rows than one 128-row M tile, several 16-token pages per request.
"""
import numpy as np
import pytest

import oracle
from structured_slot_reads_gb300 import dg, inputs
from tests.gpu_util import assert_abs, assert_rel, dev, dev_bf16, host, top2_gap

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def _lm_inputs(M, V, D, seed):
    h = inputs.hidden(M, D, seed)
    w, e = inputs.weights(V, D, seed)
    inv_t = inputs.inv_temperature(M, seed)
    return h, w, e, inv_t


def _run_lmhead(h, w, inv_t):
    M, D = h.shape
    V = w.shape[0]
    d = dg.make_dims(d_model=D, V=V)
    out = [torch.empty(M, dtype=torch.float32, device="cuda") for _ in range(3)]
    arg = torch.empty(M, dtype=torch.int32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_LMHEAD, M), dtype=torch.uint8, device="cuda")
    hd, wd, it = dev_bf16(h), dev_bf16(w), dev(inv_t)
    rc = dg.dg_lmhead_logsoftmax_entropy(d, hd, M, wd, it, None, None, None, 0, out[0], out[1],
                                         out[2], arg, None, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return [host(x) for x in out] + [host(arg)]


def test_philox_matches_oracle_bit_exact():
    rng = np.random.default_rng(0)
    n = 4096
    ctr = rng.integers(0, 2**32, size=(n, 4), dtype=np.uint64).astype(np.uint32)
    ctr[:3] = [[0, 0, 0, 0], [0xffffffff] * 4, [0x243f6a88, 0x85a308d3, 0x13198a2e, 0x03707344]]
    for seed in (0, 0xFFFFFFFFFFFFFFFF, 0x299f31d0a4093822, 123456789):
        c = dev(ctr.view(np.int32))
        out = torch.empty_like(c)
        assert dg.dg_philox_fill(seed, c, n, out) == dg.DG_OK
        torch.cuda.synchronize()
        got = host(out).view(np.uint32)
        want = oracle.philox4x32_10(ctr, oracle.seed_key(seed))
        assert np.array_equal(got, want)


@pytest.mark.parametrize("M,V,D", [(1, 1024, 128), (12, 4096, 256), (200, 3000, 200),
                                   (256, 8192, 512), (300, 2048, 128),
                                   # up to 16 rows: the skinny form (rows resident, vocabulary
                                   # on the accumulator lanes), ragged vocabulary and K tail
                                   (16, 3000, 200), (5, 2500, 2816), (17, 1024, 128)])
def test_lmhead_stats(M, V, D):
    h, w, _, inv_t = _lm_inputs(M, V, D, seed=M + V)
    lse, ent, maxz, arg = _run_lmhead(h, w, inv_t)
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(h, w, inv_t)
    assert_abs(lse, o_lse, what="lse")
    assert_abs(ent, o_ent, what="entropy")
    assert_abs(maxz, o_maxz, what="max logit")
    z = (h.astype(np.float64) @ w.astype(np.float64).T) * inv_t[:, None]
    gap = top2_gap(z)
    clear = gap > 1e-3
    assert np.array_equal(arg[clear], o_arg[clear])
    # rows without a clear winner: the GPU's choice must attain the maximum
    rows = np.nonzero(~clear)[0]
    assert np.all(z[rows, arg[rows]] >= o_maxz[rows] - 1e-3)


def test_lmhead_uniform_rows_give_ln_v():
    M, V, D = 5, 4096, 128
    h = np.zeros((M, D), np.float32)
    w, _ = inputs.weights(V, D, 3)
    lse, ent, maxz, arg = _run_lmhead(h, w, np.ones(M, np.float32))
    assert_abs(ent, np.full(M, np.log(V)), what="uniform entropy")
    assert_abs(lse, np.full(M, np.log(V)), what="uniform lse")
    assert np.all(arg == 0)


@pytest.mark.parametrize("M,V,D", [(12, 4096, 256), (256, 4096, 512), (100, 3000, 200)])
def test_selfcond_embed(M, V, D):
    h, w, e, inv_t = _lm_inputs(M, V, D, seed=7 + M)
    lse, _, _, _ = _run_lmhead(h, w, inv_t)
    d = dg.make_dims(d_model=D, V=V)
    out = torch.empty((M, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_SELFCOND, M), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_selfcond_embed(d, dev_bf16(h), M, dev_bf16(w), dev_bf16(e), dev(inv_t), dev(lse),
                              out, ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    assert_rel(host(out), oracle.selfcond_embed(h, w, e, inv_t), what="expected embedding")


def _attn_case(B, C, plen, hq, hkv, d, W, seed, paged=False, page_size=16, sm_share=0):
    from structured_slot_reads_gb300 import configs
    shp = configs.StepShape("t", B=B, C=C, P=max(plen), Hq=hq, Hkv=hkv, d_head=d, W=W, D=8, V=8)
    x = inputs.attention_inputs(shp, seed, prompt_len=np.array(plen, np.int32))
    dims = dg.make_dims(B=B, C=C, P_max=max(plen), Hq=hq, Hkv=hkv, d_head=d, W=W,
                        sm_share=sm_share)
    out = torch.empty((B, C, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, hq, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(dims, dg.DG_WS_ATTN, 0), dtype=torch.uint8,
                     device="cuda")
    if paged:
        pk, pv, table = inputs.paged_layout(x["kenc"], x["venc"], x["prompt_len"], page_size, seed)
        rc = dg.dg_attn_decode(dims, dev_bf16(x["q"]), dev_bf16(x["kc"]), dev_bf16(x["vc"]),
                               dev_bf16(pk), dev_bf16(pv), dev(table), table.shape[1],
                               pk.shape[0], page_size, dev(x["prompt_len"]), out, lse, ws)
    else:
        rc = dg.dg_attn_decode(dims, dev_bf16(x["q"]), dev_bf16(x["kc"]), dev_bf16(x["vc"]),
                               dev_bf16(x["kenc"]), dev_bf16(x["venc"]), None, 0, 0, 0,
                               dev(x["prompt_len"]), out, lse, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                      x["prompt_len"], W)
    assert_rel(host(out), ref, what="attention output")
    assert_abs(host(lse), ref_lse, what="attention lse")


@pytest.mark.parametrize("case", [
    dict(B=1, C=32, plen=[64], hq=2, hkv=1, d=64, W=8),            # tiny read shape
    dict(B=2, C=40, plen=[100, 0], hq=4, hkv=4, d=64, W=3),        # MHA, empty prompt
    dict(B=1, C=96, plen=[70], hq=8, hkv=2, d=512, W=16),          # d=512, GQA 4:1
    dict(B=2, C=64, plen=[130, 17], hq=8, hkv=2, d=512, W=200),    # window wider than canvas
    # tensor-core kernel (d = 512): split-KV with the combine, one split, GQA 8:1 and 1:1,
    # a ragged last query block, rows with no visible key in a split, empty splits
    dict(B=1, C=256, plen=[3000], hq=8, hkv=2, d=512, W=128),
    dict(B=5, C=128, plen=[200, 0, 77, 300, 129], hq=8, hkv=2, d=512, W=128),
    dict(B=1, C=40, plen=[260], hq=8, hkv=1, d=512, W=5),
    dict(B=1, C=200, plen=[140], hq=2, hkv=2, d=512, W=30),
    dict(B=1, C=256, plen=[0], hq=8, hkv=2, d=512, W=100),
    dict(B=2, C=64, plen=[1000, 0], hq=8, hkv=2, d=512, W=20),
])
def test_attention_contiguous(case):
    _attn_case(**case, seed=11)


@pytest.mark.parametrize("sm_share", [1, 19, 40, 100000])
def test_attention_sm_share(sm_share):
    """Planning for a share of the SMs changes the key splits (1 SM: one split, no
    combine; more than the device has: all SMs), never the result beyond rounding:
    the full-canvas attention shape and a paged ragged batch match the oracle."""
    _attn_case(B=1, C=256, plen=[4096], hq=8, hkv=2, d=512, W=128, seed=3, sm_share=sm_share)
    _attn_case(B=3, C=64, plen=[700, 129, 0], hq=8, hkv=2, d=512, W=16, seed=4, paged=True,
               sm_share=sm_share)


def test_attention_rescales_when_late_keys_dominate():
    """Prompt keys from position 256 on are scaled by 8 (exact in bf16), so the
    scores of later key tiles exceed the first tiles' maximum by far more than
    the lazy-rescale headroom and the output accumulator must be rescaled.  Three
    requests of 256 rows fill the GPU without splitting the key range, so one CTA
    sees every key tile."""
    B, C, P, hq, hkv, d, W = 3, 256, 600, 8, 2, 512, 16
    from structured_slot_reads_gb300 import configs
    shp = configs.StepShape("t", B=B, C=C, P=P, Hq=hq, Hkv=hkv, d_head=d, W=W, D=8, V=8)
    x = inputs.attention_inputs(shp, 21)
    x["kenc"][:, 256:] *= 8.0
    dims = dg.make_dims(B=B, C=C, P_max=P, Hq=hq, Hkv=hkv, d_head=d, W=W)
    out = torch.empty((B, C, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, hq, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(dims, dg.DG_WS_ATTN, 0), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_attn_decode(dims, dev_bf16(x["q"]), dev_bf16(x["kc"]), dev_bf16(x["vc"]),
                           dev_bf16(x["kenc"]), dev_bf16(x["venc"]), None, 0, 0, 0,
                           dev(x["prompt_len"]), out, lse, ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                                      x["prompt_len"], W)
    assert_rel(host(out), ref, what="attention output")
    assert_abs(host(lse), ref_lse, what="attention lse")


@pytest.mark.parametrize("case", [
    dict(B=3, C=48, plen=[37, 16, 90], hq=8, hkv=2, d=512, W=8),
    dict(B=2, C=32, plen=[5, 64], hq=2, hkv=1, d=64, W=4),
    dict(B=4, C=64, plen=[700, 513, 129, 1000], hq=8, hkv=2, d=512, W=128),
])
def test_attention_paged(case):
    _attn_case(**case, seed=5, paged=True)


@pytest.mark.parametrize("page_size", [8, 32, 64, 128])
def test_attention_paged_page_sizes(page_size):
    """Pages of 8, 32 and 64 keys take the CTA-pair tensor-core kernel (its half-tiles
    of 64 keys span whole pages); 128 takes the single-CTA tensor-core kernel.  All
    match the oracle.  (A page size the tensor-core kernel cannot take, e.g. 24, is
    refused before launch: tests/test_abi_host.py.)"""
    _attn_case(B=2, C=64, plen=[300, 77], hq=8, hkv=2, d=512, W=16, seed=9, paged=True,
               page_size=page_size)


@pytest.mark.parametrize("page_size", [16, 128])
def test_attention_bad_page_entries_are_masked(page_size):
    """A page-table entry outside the pool (negative or >= n_pages) reads as masked
    keys and sets DG_DEV_BAD_PAGE: the output equals the oracle's attention over
    the prompt with that page's keys left out (the prompt keys carry no position,
    so dropping them is the same as masking them).  Covers the CTA-pair kernel
    (16), the single-CTA kernel (128) and the warp-level kernel (24)."""
    from structured_slot_reads_gb300 import configs
    B, C, plen, hq, hkv, d, W = 2, 64, [700, 300], 8, 2, 512, 16
    shp = configs.StepShape("t", B=B, C=C, P=max(plen), Hq=hq, Hkv=hkv, d_head=d, W=W, D=8, V=8)
    x = inputs.attention_inputs(shp, 13, prompt_len=np.array(plen, np.int32))
    pk, pv, table = inputs.paged_layout(x["kenc"], x["venc"], x["prompt_len"], page_size, 13)
    n_pages = pk.shape[0]
    bad = {0: 3, 1: 1}                      # request -> its page index made invalid
    table = table.copy()
    table[0, bad[0]] = -1
    table[1, bad[1]] = n_pages
    dims = dg.make_dims(B=B, C=C, P_max=max(plen), Hq=hq, Hkv=hkv, d_head=d, W=W)
    out = torch.empty((B, C, hq, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, hq, C), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(dims, dg.DG_WS_ATTN, 0), dtype=torch.uint8,
                     device="cuda")
    dg.dg_clear_status()
    rc = dg.dg_attn_decode(dims, dev_bf16(x["q"]), dev_bf16(x["kc"]), dev_bf16(x["vc"]),
                           dev_bf16(pk), dev_bf16(pv), dev(table), table.shape[1], n_pages,
                           page_size, dev(x["prompt_len"]), out, lse, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    assert dg.dg_get_status() & dg.DG_DEV_BAD_PAGE
    dg.dg_clear_status()
    # the oracle's prompt: each request's keys without its invalid page
    kenc = np.zeros_like(x["kenc"])
    venc = np.zeros_like(x["venc"])
    plen2 = np.zeros(B, np.int32)
    for b in range(B):
        keep = np.ones(plen[b], bool)
        keep[bad[b] * page_size:(bad[b] + 1) * page_size] = False
        n = int(keep.sum())
        kenc[b, :n] = x["kenc"][b, :plen[b]][keep]
        venc[b, :n] = x["venc"][b, :plen[b]][keep]
        plen2[b] = n
    ref, ref_lse = oracle.attn_decode(x["q"], x["kc"], x["vc"], kenc, venc, plen2, W)
    assert_rel(host(out), ref, what="attention output")
    assert_abs(host(lse), ref_lse, what="attention lse")


def test_slot_noise_rows_bit_exact():
    M, V, D = 64, 1024, 128
    h, w, e, inv_t = _lm_inputs(M, V, D, seed=3)
    slot_row = np.array([17, 40, 63], np.int32)
    slot_req = np.array([0, 1, 1], np.int32)
    S, R, seed, step = 3, 4, 0xDEADBEEF12345, 5
    d = dg.make_dims(d_model=D, V=V)
    rows = torch.empty((S * R, D), dtype=torch.bfloat16, device="cuda")
    it = torch.empty(S * R, dtype=torch.float32, device="cuda")
    tok = torch.empty((S, R), dtype=torch.int32, device="cuda")
    rc = dg.dg_slot_noise(d, dev_bf16(h), M, dev_bf16(e), dev(inv_t), dev(slot_row), dev(slot_req),
                          S, R, seed, step, rows, it, tok)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    o_rows, o_tok = oracle.slot_noise_rows(h, e, slot_row, slot_req, seed, step, R, V)
    assert np.array_equal(host(tok), o_tok)
    assert np.array_equal(host(rows), o_rows)
    assert np.array_equal(host(it), np.repeat(inv_t[slot_row], R))


def _commit_case(B, C, gamma, seed, frac_open=1.0, state=False):
    rng = np.random.default_rng(seed)
    # entropies with distinct values spaced > 4e-3 apart so the order and cut are unique
    ent = np.stack([rng.permutation(C) * 0.01 + rng.uniform(0, 1e-3, C) for _ in range(B)])
    ent = (ent + 0.5).astype(np.float32)
    arg = rng.integers(0, 262144, (B, C)).astype(np.int32)
    cand = (rng.random((B, C)) < frac_open).astype(np.uint8)
    gam = np.full(B, gamma, np.float32)
    # keep the cut away from gamma
    for b in range(B):
        order = np.lexsort((np.arange(C), ent[b]))
        order = order[cand[b][order] == 1]
        cs = np.cumsum(ent[b][order].astype(np.float64))
        if np.any(np.abs(cs - gam[b]) < 4e-3):
            gam[b] += 2e-2
    committed = (rng.random((B, C)) < 0.2).astype(np.uint8) if state else np.zeros((B, C), np.uint8)
    tok_state = np.where(committed == 1, 7, -1).astype(np.int32)
    d = dg.make_dims(B=B, C=C)
    cm = torch.empty((B, C), dtype=torch.uint8, device="cuda")
    tk = torch.empty((B, C), dtype=torch.int32, device="cuda")
    nc = torch.empty(B, dtype=torch.int32, device="cuda")
    cs_d, ts_d = dev(committed), dev(tok_state)
    rc = dg.dg_commit(d, dev(ent), dev(arg), dev(cand), dev(gam), cs_d if state else None,
                      ts_d if state else None, cm, tk, nc)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    open_ = cand & (1 - committed)
    o_cm, o_tk, o_n = oracle.commit(ent, arg, open_, gam)
    assert np.array_equal(host(cm), o_cm)
    assert np.array_equal(host(tk), o_tk)
    assert np.array_equal(host(nc), o_n)
    if state:
        assert np.array_equal(host(cs_d), committed | o_cm.astype(np.uint8))
        assert np.array_equal(host(ts_d), np.where(o_cm == 1, arg, tok_state))


@pytest.mark.parametrize("B,C,gamma,frac,state", [(1, 256, 25.6, 1.0, False), (4, 32, 3.2, 1.0, False),
                                                  (8, 256, 25.6, 0.5, True), (2, 1000, 40.0, 0.3, True),
                                                  (3, 64, 0.1, 1.0, False), (2, 16, 1e9, 0.0, False)])
def test_commit(B, C, gamma, frac, state):
    _commit_case(B, C, gamma, seed=B * C, frac_open=frac, state=state)


@pytest.mark.parametrize("shift", [0, 1])
def test_canvas_update_bit_exact(shift):
    """16-byte aligned buffers (one thread per 8 values) and buffers 4 or 8 bytes
    past a 16-byte boundary (the row-per-CTA form): the same bits as the oracle."""
    M, V, D = 40, 512, 136
    h0 = inputs.hidden(M, D, 1)
    emb, _ = inputs.weights(V, D, 1)
    e_sc = (np.random.default_rng(2).standard_normal((M, D)) * 0.05).astype(np.float32)
    committed = (np.arange(M) % 3 == 0).astype(np.uint8)
    tokens = np.where(committed == 1, np.arange(M) * 7 % V, -1).astype(np.int32)
    d = dg.make_dims(d_model=D, V=V)

    def shifted(x, k):
        # a view k elements into a larger buffer: 2 bf16 or 2 floats past 16-byte alignment
        buf = torch.empty(x.numel() + 8, dtype=x.dtype, device="cuda")
        v = buf[k:k + x.numel()].view(x.shape)
        v.copy_(x)
        return v

    k = 2 * shift
    h0_d, es_d = shifted(dev_bf16(h0), k), shifted(dev(e_sc), k)
    out = shifted(torch.zeros((M, D), dtype=torch.bfloat16, device="cuda"), k)
    rc = dg.dg_canvas_update(d, h0_d, es_d, dev_bf16(emb), dev(tokens), dev(committed), M, out)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    want = oracle.canvas_update(h0, e_sc, emb, tokens, committed)
    assert np.array_equal(host(out), want)


def test_status_word_clean_after_valid_calls():
    dg.dg_clear_status()
    test_slot_noise_rows_bit_exact()
    assert dg.dg_get_status() == 0


def _tiled(wd, V, D):
    d = dg.make_dims(d_model=D, V=V)
    out = torch.empty(dg.dg_heads_weights_bytes(d) // 2, dtype=torch.bfloat16, device="cuda")
    assert dg.dg_heads_weights_tile(d, wd, out) == dg.DG_OK
    return out


def _run_heads(h, draws, w, inv_t, inv_t_draw, with_probs=True, tiled=False):
    M, D = h.shape
    V = w.shape[0]
    nd = 0 if draws is None else draws.shape[0]
    d = dg.make_dims(d_model=D, V=V)
    f32 = torch.float32
    lse, ent, maxz = (torch.empty(M, dtype=f32, device="cuda") for _ in range(3))
    arg = torch.empty(M, dtype=torch.int32, device="cuda")
    lse_d = torch.empty(max(nd, 1), dtype=f32, device="cuda")
    scale = torch.empty(M, dtype=f32, device="cuda")
    ld = dg.dg_probs_ld(V)
    probs = torch.empty((M, ld), dtype=torch.bfloat16, device="cuda") if with_probs else None
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_HEADS, M), dtype=torch.uint8, device="cuda")
    wd = w if isinstance(w, torch.Tensor) else dev_bf16(w)
    wt = _tiled(wd, V, D) if tiled else None
    rc = dg.dg_denoise_heads(d, dev_bf16(h), M, dev_bf16(draws) if nd else None, nd, wd,
                             dev(inv_t), dev(inv_t_draw) if nd else None, lse, ent, maxz, arg,
                             lse_d if nd else None, None, None, 0, None, scale, probs, ld, ws,
                             w_tiled=wt)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    return dict(lse=host(lse), ent=host(ent), maxz=host(maxz), arg=host(arg),
                lse_draw=host(lse_d)[:nd], scale=scale, probs=probs, ld=ld, dims=d)


@pytest.mark.parametrize("M,nd,V,D", [(256, 12, 8192, 512), (100, 5, 3000, 200),
                                      (300, 12, 2048, 128), (64, 0, 4096, 256), (1, 16, 1024, 128),
                                      (200, 0, 5000, 256),
                                      # several 256-row groups, ragged vocabularies
                                      (520, 0, 4000, 128), (384, 16, 2504, 192),
                                      # batched canvases: the warp-per-row reference
                                      (1100, 8, 2048, 128),
                                      # 16 row groups x 19 CTAs: two waves of balanced ranges
                                      (4096, 0, 4096, 128)])
def test_denoise_heads_fused_pass(M, nd, V, D):
    h, w, e, inv_t = _lm_inputs(M, V, D, seed=31 + M)
    draws = inputs.hidden(nd, D, 99) if nd else None
    inv_d = inputs.inv_temperature(nd, 98) if nd else None
    got = _run_heads(h, draws, w, inv_t, inv_d)
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(h, w, inv_t)
    assert_abs(got["lse"], o_lse, what="lse")
    assert_abs(got["ent"], o_ent, what="entropy")
    assert_abs(got["maxz"], o_maxz, what="max logit")
    z = (h.astype(np.float64) @ w.astype(np.float64).T) * inv_t[:, None]
    clear = top2_gap(z) > 1e-3
    assert np.array_equal(got["arg"][clear], o_arg[clear])
    if nd:
        d_lse, _, _, _ = oracle.lmhead_stats(draws, w, inv_d)
        assert_abs(got["lse_draw"], d_lse, what="draw-row lse")
    # the probabilities, normalised, are the softmax
    p = host(got["probs"])[:, :V].astype(np.float64) * host(got["scale"])[:, None]
    ref_p = np.exp(z - o_lse[:, None])
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=5e-3)
    assert np.max(np.abs(p - ref_p) / (ref_p + 1e-30)) < 1e-2
    # and feed the expected embedding
    ed = dev_bf16(e)
    out = torch.empty((M, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(got["dims"], dg.DG_WS_PROBS_EMBED, M),
                     dtype=torch.uint8, device="cuda")
    rc = dg.dg_selfcond_from_probs(got["dims"], got["probs"], got["ld"], got["scale"], M, ed,
                                   out, ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    assert_rel(host(out), oracle.selfcond_embed(h, w, e, inv_t), what="expected embedding")


@pytest.mark.parametrize("V,D", [(1000, 128), (224, 64), (4096, 2816), (2504, 192)])
def test_heads_weights_tiled_layout(V, D):
    """dg_heads_weights_tile against the layout written out with numpy: 224-row
    tiles of 64-column blocks, block (t, kb) contiguous, zero rows past V."""
    w = inputs.normal_bf16((V, D), 1.0, 7 + V, 1)
    got = host(_tiled(dev_bf16(w), V, D))
    tiles = -(-V // 224)
    pad = np.zeros((tiles * 224, D), np.float32)
    pad[:V] = w
    want = pad.reshape(tiles, 224, D // 64, 64).transpose(0, 2, 1, 3).reshape(-1)
    assert got.shape == want.shape and np.array_equal(got, want)


@pytest.mark.parametrize("M,nd,V,D", [(256, 12, 8192, 512), (100, 5, 3000, 192),
                                      (384, 16, 2504, 192), (1, 16, 1024, 128),
                                      (1100, 8, 2048, 128), (64, 0, 4096, 256),
                                      (256, 12, 262144, 2816)])
def test_denoise_heads_tiled_weights_bit_identical(M, nd, V, D):
    """The pass on W's tiled copy reads the same values in the same order: every
    output bit-identical to the pass on the row-major W (without draw rows the
    copy is not used), including the 262144 x 2816 lm-head of the full canvas."""
    h, w, _, inv_t = _lm_inputs(M, V, D, seed=5 + M)
    wd = dev_bf16(w)
    del w
    draws = inputs.hidden(nd, D, 99) if nd else None
    inv_d = inputs.inv_temperature(nd, 98) if nd else None
    a = _run_heads(h, draws, wd, inv_t, inv_d)
    b = _run_heads(h, draws, wd, inv_t, inv_d, tiled=True)
    for k in ("lse", "ent", "maxz", "arg", "lse_draw"):
        assert np.array_equal(a[k], b[k]), k
    assert torch.equal(a["scale"], b["scale"])
    assert torch.equal(a["probs"][:, :V], b["probs"][:, :V])


@pytest.mark.parametrize("M,V,D", [(2048, 2048, 2816), (4096, 1024, 2816), (256, 4096, 2816)])
def test_selfcond_from_probs_split_k(M, V, D):
    """out = prob_scale * (P~ E) against the float64 definition, in the split-K
    configurations the GEMM picks: 2048 and 4096 rows make 88 and 176 output tiles,
    split by whole-tile rounds into waves; 256 rows make 11 tiles on 7/8 of the SMs."""
    rng = np.random.default_rng(M + V)
    ld = dg.dg_probs_ld(V)
    p = np.zeros((M, ld), np.float32)
    p[:, :V] = np.exp(rng.normal(0.0, 2.0, (M, V))).astype(np.float32)
    p = inputs.to_bf16(p)
    scale = (1.0 / p[:, :V].astype(np.float64).sum(axis=1)).astype(np.float32)
    _, e = inputs.weights(V, D, 17)
    d = dg.make_dims(d_model=D, V=V)
    out = torch.empty((M, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_PROBS_EMBED, M), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_selfcond_from_probs(d, dev_bf16(p), ld, dev(scale), M, dev_bf16(e), out, ws)
    assert rc == dg.DG_OK, dg.strerror(rc)
    torch.cuda.synchronize()
    want = (p[:, :V].astype(np.float64) @ e.astype(np.float64)) * scale[:, None].astype(np.float64)
    assert_rel(host(out), want, what="expected embedding")


@pytest.mark.parametrize("nd", [0, 4])
def test_denoise_heads_exact_for_far_logits(nd):
    """Rows with logits far above their reference (which is read off the first 8
    vocabulary entries): the CTA that meets one raises its reference by whole powers
    of two and rescales what it already wrote, the finalize brings the other CTAs'
    probabilities to it, so the statistics and the self-conditioning probabilities
    stay exact; no status bit is set.  Row 3 has one logit 200 nats up (CTA-local
    raise, several hundred log2 units); row 5 has two, 60 and 120 nats up, in two
    CTA ranges (two raises of different size); row 6 one in the first tile."""
    M, V, D = 8, 65536, 128
    h, w, e, inv_t = _lm_inputs(M, V, D, seed=5)

    def plant(row, vid, nats):
        wl = w[vid].astype(np.float64)
        x = h[row].astype(np.float64) + (nats / float(inv_t[row])) * wl / np.dot(wl, wl)
        h[row] = inputs.to_bf16(x.astype(np.float32))

    plant(3, 40000, 200.0)
    plant(5, 3000, 60.0)
    plant(5, 61000, 120.0)
    plant(6, 100, 150.0)
    draws = inputs.hidden(nd, D, 77) if nd else None
    inv_d = inputs.inv_temperature(nd, 78) if nd else None
    dg.dg_clear_status()
    got = _run_heads(h, draws, w, inv_t, inv_d)
    assert dg.dg_get_status() == 0
    o_lse, o_ent, o_maxz, o_arg = oracle.lmhead_stats(h, w, inv_t)
    assert_abs(got["lse"], o_lse, what="lse")
    assert_abs(got["ent"], o_ent, what="entropy")
    assert_abs(got["maxz"], o_maxz, what="max logit")
    assert got["arg"][3] == 40000 and got["arg"][5] == 61000 and got["arg"][6] == 100
    z = (h.astype(np.float64) @ w.astype(np.float64).T) * inv_t[:, None]
    clear = top2_gap(z) > 1e-3
    assert np.array_equal(got["arg"][clear], o_arg[clear])
    # the probabilities: P.E from them is the expected embedding of every row
    d = got["dims"]
    out = torch.empty((M, D), dtype=torch.float32, device="cuda")
    ws = torch.empty(dg.dg_workspace_bytes(d, dg.DG_WS_PROBS_EMBED, M), dtype=torch.uint8,
                     device="cuda")
    rc = dg.dg_selfcond_from_probs(d, got["probs"], got["ld"], got["scale"], M, dev_bf16(e), out,
                                   ws)
    assert rc == dg.DG_OK
    torch.cuda.synchronize()
    assert_rel(host(out), oracle.selfcond_embed(h, w, e, inv_t), what="expected embedding")
    if nd:
        d_lse, _, _, _ = oracle.lmhead_stats(draws, w, inv_d)
        assert_abs(got["lse_draw"], d_lse, what="draw-row lse")
