"""Seeded synthetic inputs for the structured-read denoise step.

This module only draws random numbers and converts them to the storage
formats the library reads (bf16 held in float32 / uint16 bits, fp32, int32).
It holds none of the method's arithmetic, so both the CUDA path's tests and
the CPU oracle can be fed from it.

Recipe (one independent NumPy PCG64 stream per tensor, keyed by
(seed, stream id, ...)):
  hidden rows, Q, K, V, encoder K/V  ~ N(0, 1), rounded to bf16
  lm-head W and embedding table E   ~ N(0, 1/d_model) (std 1/sqrt(d_model)), bf16
  temperature T ~ U(0.5, 2) per row, stored as fp32 1/T
  label ids: uniform without replacement from the vocabulary
  template token ids: uniform, fixed per seed
  paged layout: each request's 16-token pages scattered over a shared pool
The device variants (``device_*``) draw the same distributions with torch on
the GPU for large benchmark tensors; they are not bit-identical to the NumPy
draws and are never used where the oracle must see the same values.
"""
import numpy as np

from .configs import StepShape

S_H, S_W, S_E, S_INVT, S_Q, S_KC, S_VC, S_KENC, S_VENC = 1, 2, 3, 4, 5, 6, 7, 8, 9
S_LABELS, S_TEMPLATE, S_PROMPT, S_PAGES, S_SLOTS, S_GROUPS = 10, 11, 12, 13, 14, 15
S_PQ, S_PK, S_PV = 16, 17, 18

MAX_LABELS = 26


def _rng(*key):
    return np.random.default_rng([int(k) & 0xFFFFFFFF for k in key])


def to_bf16(x):
    """float32 -> nearest bf16 (ties to even), returned as float32 values."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    r = ((u >> 16) & 1) + np.uint32(0x7FFF)
    out = ((u + r) & np.uint32(0xFFFF0000)).view(np.float32)
    return out


def bf16_bits(x):
    """bf16-valued float32 array -> uint16 bit patterns (upper halves)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def normal_bf16(shape, std, *key):
    z = _rng(*key).standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        z *= np.float32(std)
    return to_bf16(z)


def hidden(M, D, seed, attempt=0):
    return normal_bf16((M, D), 1.0, seed, S_H, attempt)


def redraw_rows(h, rows, seed, attempt):
    """Replace the given rows of ``h`` by fresh draws for ``attempt`` (>0)."""
    h = h.copy()
    for i in rows:
        h[i] = normal_bf16((h.shape[1],), 1.0, seed, S_H, attempt, 1000003 + int(i))
    return h


def weights(V, D, seed):
    """lm-head W and embedding table E, both [V, D] ~ N(0, 1/D) in bf16."""
    std = 1.0 / np.sqrt(D)
    return normal_bf16((V, D), std, seed, S_W), normal_bf16((V, D), std, seed, S_E)


def inv_temperature(M, seed):
    t = _rng(seed, S_INVT).uniform(0.5, 2.0, size=M)
    return (1.0 / t).astype(np.float32)


def prompt_lengths(shape: StepShape, seed, lo=512):
    if shape.B == 1 or not shape.paged:
        return np.full(shape.B, shape.P, dtype=np.int32)
    lo = min(lo, max(1, shape.P // 2))
    return _rng(seed, S_PROMPT).integers(lo, shape.P + 1, size=shape.B).astype(np.int32)


def attention_inputs(shape: StepShape, seed, prompt_len=None):
    """Q [B,C,Hq,d], canvas K/V [B,C,Hkv,d], encoder K/V [B,Pmax,Hkv,d] ~ N(0,1) bf16."""
    B, C, hq, hkv, d = shape.B, shape.C, shape.Hq, shape.Hkv, shape.d_head
    if prompt_len is None:
        prompt_len = prompt_lengths(shape, seed)
    pmax = int(max(prompt_len)) if B else 0
    return dict(
        q=normal_bf16((B, C, hq, d), 1.0, seed, S_Q),
        kc=normal_bf16((B, C, hkv, d), 1.0, seed, S_KC),
        vc=normal_bf16((B, C, hkv, d), 1.0, seed, S_VC),
        kenc=normal_bf16((B, pmax, hkv, d), 1.0, seed, S_KENC),
        venc=normal_bf16((B, pmax, hkv, d), 1.0, seed, S_VENC),
        prompt_len=np.asarray(prompt_len, dtype=np.int32),
    )


def prefill_inputs(B, P, Hq, Hkv, d, seed):
    """Prompt-side Q [B, P, Hq, d] and K, V [B, P, Hkv, d] of an encoder prefill, N(0,1) bf16."""
    return dict(q=normal_bf16((B, P, Hq, d), 1.0, seed, S_PQ),
                k=normal_bf16((B, P, Hkv, d), 1.0, seed, S_PK),
                v=normal_bf16((B, P, Hkv, d), 1.0, seed, S_PV))


def paged_layout(kenc, venc, prompt_len, page_size, seed, spare_pages=7):
    """Scatter each request's prompt KV into pages of a shared pool.

    Returns pool_k, pool_v [n_pages, page_size, Hkv, d] and page_table
    [B, max_pages] int32 (-1 past a request's last page).  Pages are assigned
    from a random permutation of the pool so neighbours are not adjacent.
    """
    B = kenc.shape[0]
    hkv, d = kenc.shape[2], kenc.shape[3]
    table, total = page_table(prompt_len, page_size, seed, spare_pages)
    pool_k = np.zeros((total, page_size, hkv, d), dtype=np.float32)
    pool_v = np.zeros_like(pool_k)
    for b in range(B):
        for pg in range((int(prompt_len[b]) + page_size - 1) // page_size):
            page = int(table[b, pg])
            lo = pg * page_size
            hi = min(lo + page_size, int(prompt_len[b]))
            pool_k[page, : hi - lo] = kenc[b, lo:hi]
            pool_v[page, : hi - lo] = venc[b, lo:hi]
    return pool_k, pool_v, table


def page_table(prompt_len, page_size, seed, spare_pages=7):
    """Page table [B, max_pages] int32 (-1 past a request's last page) and the pool size.

    Pages come from a random permutation of the pool, handed out request by
    request, so a request's pages are scattered through the pool.
    """
    B = len(prompt_len)
    need = [(int(p) + page_size - 1) // page_size for p in prompt_len]
    total = sum(need) + spare_pages
    perm = _rng(seed, S_PAGES).permutation(total)
    table = np.full((B, max(max(need) if need else 0, 1)), -1, dtype=np.int32)
    nxt = 0
    for b in range(B):
        table[b, :need[b]] = perm[nxt:nxt + need[b]]
        nxt += need[b]
    return table, total


def label_set(n, V, *key):
    return _rng(*key).choice(V, size=n, replace=False).astype(np.int32)


def slot_table(shape: StepShape, seed, L=MAX_LABELS):
    """Slot rows, request ids and label ids for the slots of ``shape`` (same for every request).

    Returns slot_row [S] (flattened canvas row b*C + pos), slot_req [S],
    label_ids [S, L] (-1 padded; L = 26 unless a wide table is asked for), n_labels [S].
    """
    rows, reqs, labs, ns = [], [], [], []
    for b in range(shape.B):
        for j, (pos, k) in enumerate(shape.slots):
            rows.append(b * shape.C + pos)
            reqs.append(b)
            lab = np.full(L, -1, dtype=np.int32)
            lab[:k] = label_set(k, shape.V, seed, S_LABELS, b, j)
            labs.append(lab)
            ns.append(k)
    if not rows:
        return (np.zeros(0, np.int32), np.zeros(0, np.int32),
                np.zeros((0, L), np.int32), np.zeros(0, np.int32))
    return (np.array(rows, np.int32), np.array(reqs, np.int32),
            np.stack(labs), np.array(ns, np.int32))


def candidates(shape: StepShape, slot_row=None):
    """Commit candidates [B, C] (1 = open).  All positions when the canvas is
    fully open, else only the slot positions (the rest holds template ids)."""
    cand = np.zeros((shape.B, shape.C), dtype=np.uint8)
    if shape.all_open:
        cand[:] = 1
    elif slot_row is not None:
        for r in slot_row:
            cand[int(r) // shape.C, int(r) % shape.C] = 1
    return cand


def template_tokens(shape: StepShape, seed):
    return _rng(seed, S_TEMPLATE).integers(0, shape.V, size=(shape.B, shape.C)).astype(np.int32)


def two_stage_tables(shape: StepShape, seed, n_groups=9, group_size=9, last_group=5):
    """Config of the two-stage ask_if read (77 synthetic intents -> 9 groups).

    Per request: a stage-1 group slot with ``n_groups`` labels, 0-3 other
    stage-1 slots with 2-26 labels, and one stage-2 item slot whose label set
    is the item list of the chosen group (its question carries ask_if = group).
    Returns a list of dicts, one per request.
    """
    rng = _rng(seed, S_GROUPS)
    out = []
    C = shape.C
    for b in range(shape.B):
        n_other = int(rng.integers(0, 4))
        positions = rng.choice(np.arange(8, C - 8), size=2 + n_other, replace=False)
        group_labels = label_set(n_groups, shape.V, seed, S_GROUPS, b, 0)
        others = []
        for j in range(n_other):
            k = int(rng.integers(2, MAX_LABELS + 1))
            others.append((int(positions[2 + j]), label_set(k, shape.V, seed, S_GROUPS, b, 10 + j)))
        items = []
        for g in range(n_groups):
            k = last_group if g == n_groups - 1 else group_size
            items.append(label_set(k, shape.V, seed, S_GROUPS, b, 100 + g))
        out.append(dict(group_pos=int(positions[0]), group_labels=group_labels,
                        others=others, item_pos=int(positions[1]), item_labels=items))
    return out


def step_inputs(shape: StepShape, seed, with_attention=True):
    """Every input of one denoise step for ``shape`` as NumPy arrays."""
    M = shape.B * shape.C
    W, E = weights(shape.V, shape.D, seed)
    slot_row, slot_req, label_ids, n_labels = slot_table(shape, seed)
    d = dict(h=hidden(M, shape.D, seed), w=W, e=E, inv_t=inv_temperature(M, seed),
             slot_row=slot_row, slot_req=slot_req, label_ids=label_ids, n_labels=n_labels,
             cand=candidates(shape, slot_row), template=template_tokens(shape, seed),
             gamma=np.full(shape.B, shape.gamma, dtype=np.float32))
    if with_attention:
        d.update(attention_inputs(shape, seed))
    return d


# ---------------------------------------------------------------------------
# device-side draws for large benchmark tensors (torch, no oracle involvement)
# ---------------------------------------------------------------------------
def device_normal_bf16(shape, std, seed, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.empty(tuple(shape), dtype=torch.float32, device=device)
    t.normal_(0.0, float(std), generator=g)
    return t.to(torch.bfloat16)


def device_uniform(shape, lo, hi, seed, device):
    import torch
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    t = torch.empty(tuple(shape), dtype=torch.float32, device=device)
    t.uniform_(lo, hi, generator=g)
    return t
