"""Pins for the oracle's decoder-mode windowed attention."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attn_decode, paged_to_contiguous


def _inputs(B=2, C=12, P=(5, 9), hq=4, hkv=2, d=8, seed=0):
    rng = np.random.default_rng(seed)
    pmax = max(P)
    return dict(
        q=rng.standard_normal((B, C, hq, d)),
        kc=rng.standard_normal((B, C, hkv, d)),
        vc=rng.standard_normal((B, C, hkv, d)),
        kenc=rng.standard_normal((B, pmax, hkv, d)),
        venc=rng.standard_normal((B, pmax, hkv, d)),
        prompt_len=np.array(P),
    )


def _sdpa(x, window):
    """Library reference: torch SDPA in float64 with an explicit boolean mask."""
    q = torch.tensor(x["q"])
    B, C, hq, d = q.shape
    hkv = x["kc"].shape[2]
    outs, lses = [], []
    for b in range(B):
        P = int(x["prompt_len"][b])
        k = torch.cat([torch.tensor(x["kenc"][b, :P]), torch.tensor(x["kc"][b])], 0)
        v = torch.cat([torch.tensor(x["venc"][b, :P]), torch.tensor(x["vc"][b])], 0)
        k = k.repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)  # [hq, P+C, d]
        v = v.repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)
        qb = q[b].permute(1, 0, 2)  # [hq, C, d]
        i = torch.arange(C)[:, None]
        j = torch.arange(C)[None, :]
        mask = torch.cat([torch.ones(C, P, dtype=torch.bool), (i - j).abs() <= window], 1)
        o = F.scaled_dot_product_attention(qb, k, v, attn_mask=mask)
        s = (qb @ k.transpose(1, 2)) / np.sqrt(d)
        lse = torch.logsumexp(s.masked_fill(~mask, float("-inf")), dim=-1)
        outs.append(o.permute(1, 0, 2).numpy())
        lses.append(lse.numpy())
    return np.stack(outs), np.stack(lses)


@pytest.mark.parametrize("window", [0, 1, 3, 11, 40])
def test_matches_torch_sdpa_with_mask(window):
    x = _inputs(seed=window)
    out, lse = attn_decode(**x, window=window)
    ref, ref_lse = _sdpa(x, window)
    np.testing.assert_allclose(out, ref, atol=1e-12)
    np.testing.assert_allclose(lse, ref_lse, atol=1e-12)


def test_wide_window_is_full_bidirectional():
    x = _inputs(seed=9)
    C = x["q"].shape[1]
    a, la = attn_decode(**x, window=C - 1)
    b, lb = attn_decode(**x, window=10 * C)
    np.testing.assert_array_equal(a, b)
    np.testing.assert_array_equal(la, lb)


def test_no_prompt_zero_window_returns_own_value():
    x = _inputs(P=(0, 0), seed=3)
    out, _ = attn_decode(**x, window=0)
    hq, hkv = x["q"].shape[2], x["kc"].shape[2]
    for h in range(hq):
        np.testing.assert_allclose(out[:, :, h], x["vc"][:, :, h // (hq // hkv)], atol=1e-15)


def test_gqa_group_mapping():
    x = _inputs(seed=4)
    # making KV head 1 identical to KV head 0 must make all query heads of both groups
    # agree with a single-KV-head run
    x1 = {k: (v.copy() if hasattr(v, "copy") else v) for k, v in x.items()}
    for key in ("kc", "vc", "kenc", "venc"):
        x1[key][:, :, 1] = x1[key][:, :, 0]
    out, _ = attn_decode(**x1, window=2)
    x2 = dict(x1)
    for key in ("kc", "vc", "kenc", "venc"):
        x2[key] = x1[key][:, :, :1]
    out2, _ = attn_decode(**x2, window=2)
    np.testing.assert_allclose(out, out2, atol=1e-14)


def test_paged_equals_contiguous():
    rng = np.random.default_rng(11)
    B, hkv, d, ps = 3, 2, 8, 4
    plen = np.array([5, 12, 1])
    need = [(p + ps - 1) // ps for p in plen]
    total = sum(need) + 2
    perm = rng.permutation(total)
    pool_k = rng.standard_normal((total, ps, hkv, d))
    pool_v = rng.standard_normal((total, ps, hkv, d))
    table = np.full((B, max(need)), -1)
    n = 0
    for b in range(B):
        for p in range(need[b]):
            table[b, p] = perm[n]
            n += 1
    kenc, venc = paged_to_contiguous(pool_k, pool_v, table, plen, ps)
    for b in range(B):
        for j in range(plen[b]):
            np.testing.assert_array_equal(kenc[b, j], pool_k[table[b, j // ps], j % ps])
            np.testing.assert_array_equal(venc[b, j], pool_v[table[b, j // ps], j % ps])


# ---- encoder-mode prefill -----------------------------------------------------
def _prefill_inputs(B=2, P=11, lens=(11, 6), hq=4, hkv=2, d=8, seed=3):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((B, P, hq, d)), rng.standard_normal((B, P, hkv, d)),
            rng.standard_normal((B, P, hkv, d)), np.array(lens))


def test_prefill_matches_torch_causal_sdpa():
    """Library reference: torch SDPA in float64 with is_causal=True, per request prefix."""
    from oracle import prefill_attn
    q, k, v, lens = _prefill_inputs()
    out, lse = prefill_attn(q, k, v, lens)
    hq, hkv, d = q.shape[2], k.shape[2], q.shape[3]
    for b, n in enumerate(lens):
        qb = torch.tensor(q[b, :n]).permute(1, 0, 2)
        kb = torch.tensor(k[b, :n]).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)
        vb = torch.tensor(v[b, :n]).repeat_interleave(hq // hkv, dim=1).permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(qb, kb, vb, is_causal=True).permute(1, 0, 2)
        assert np.allclose(out[b, :n], ref.numpy(), atol=1e-12)
        s = (qb @ kb.transpose(1, 2)) / np.sqrt(d)
        s = s.masked_fill(torch.triu(torch.ones(n, n, dtype=torch.bool), 1), float("-inf"))
        assert np.allclose(lse[b, :, :n], torch.logsumexp(s, -1).numpy(), atol=1e-12)
        assert np.all(out[b, n:] == 0)


def test_prefill_first_row_is_its_own_value_and_rows_subset_agrees():
    from oracle import prefill_attn
    q, k, v, lens = _prefill_inputs()
    out, _ = prefill_attn(q, k, v, lens)
    for h in range(q.shape[2]):
        assert np.allclose(out[:, 0, h], v[:, 0, h // 2], atol=1e-12)  # only key 0 is visible
    part, part_lse = prefill_attn(q, k, v, lens, rows=[0, 5, 10])
    full, full_lse = prefill_attn(q, k, v, lens)
    for r in (0, 5, 10):
        assert np.allclose(part[:, r][r < lens], full[:, r][r < lens], atol=1e-12)


def test_prefill_gqa_head_mapping():
    """Making KV head 1 differ changes exactly the query heads 2 and 3 (group of 2)."""
    from oracle import prefill_attn
    q, k, v, lens = _prefill_inputs()
    out0, _ = prefill_attn(q, k, v, lens)
    v2 = v.copy()
    v2[:, :, 1] += 1.0
    out1, _ = prefill_attn(q, k, v2, lens)
    assert np.allclose(out0[:, :, :2], out1[:, :, :2])
    assert np.allclose(out1[:, :, 2:][:, :6], out0[:, :, 2:][:, :6] + 1.0)


def test_paged_write_inverts_paged_to_contiguous():
    from oracle import paged_write
    q, k, v, lens = _prefill_inputs()
    ps, B = 4, k.shape[0]
    pages = (k.shape[1] + ps - 1) // ps
    perm = np.random.default_rng(0).permutation(B * pages + 3)
    table = perm[:B * pages].reshape(B, pages)
    pk, pv = paged_write(k, v, lens, table, ps, B * pages + 3)
    ke, ve = paged_to_contiguous(pk, pv, table, lens, ps)
    for b, n in enumerate(lens):
        assert np.array_equal(ke[b, :n], k[b, :n]) and np.array_equal(ve[b, :n], v[b, :n])
    assert np.count_nonzero(pk.reshape(pk.shape[0], -1).any(axis=1)) == sum(
        (n + ps - 1) // ps for n in lens)


def test_mixed_batch_reduces_to_its_modes():
    """All-decoder batches equal attn_decode; all-encoder batches equal prefill_attn."""
    from oracle import attn_mixed, prefill_attn
    x = _inputs(B=2, C=12, P=(5, 9))
    n = np.array([12, 12])
    out, lse = attn_mixed(np.zeros(2, int), n, x["q"], x["kc"], x["vc"], x["kenc"], x["venc"],
                          x["prompt_len"], 3)
    ref, ref_lse = attn_decode(x["q"], x["kc"], x["vc"], x["kenc"], x["venc"], x["prompt_len"], 3)
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, ref_lse, atol=1e-12)
    out, lse = attn_mixed(np.ones(2, int), np.array([12, 7]), x["q"], x["kc"], x["vc"], None,
                          None, x["prompt_len"], 3)
    ref, ref_lse = prefill_attn(x["q"], x["kc"], x["vc"], np.array([12, 7]))
    assert np.allclose(out, ref, atol=1e-12) and np.allclose(lse, ref_lse, atol=1e-12)
